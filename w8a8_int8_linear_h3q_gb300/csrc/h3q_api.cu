// h3q_api.cu -- the C ABI declared in include/h3q.h: argument validation,
// device check, and the launch sequence of each entry point.  No entry point
// allocates device memory; every launch goes on the caller's stream.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "h3q_abi_checks.cuh"
#include "h3q_internal.cuh"

namespace h3q {

namespace {
constexpr int64_t kMaxK = 133143;            // K * 127^2 < 2^31
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 65536;
constexpr int64_t kMaxN = int64_t(65535) * 128;
}  // namespace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

h3q_status check_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 16) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (K % 16 != 0 || K > kMaxK) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (M > kMaxRows || N > kMaxN) return H3Q_ERR_UNSUPPORTED_SHAPE;
  return H3Q_OK;
}

// The current device must be an sm_103 part (the kernels are built for sm_103a only).
h3q_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_NO_DEVICE;
  }
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_NO_DEVICE;
  }
  return (major == 10 && minor == 3) ? H3Q_OK : H3Q_ERR_NO_DEVICE;
}

// With H3Q_VERBOSE set in the environment, CUDA errors are also printed.
h3q_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return H3Q_OK;
  if (std::getenv("H3Q_VERBOSE")) std::fprintf(stderr, "h3q: %s\n", cudaGetErrorString(e));
  return H3Q_ERR_CUDA;
}

}  // namespace h3q

namespace {

using h3q::aligned16;
using h3q::check_device;
using h3q::check_shape;
using h3q::from_cuda;

// Word `index` of the status block of a workspace last used with (M, K).
h3q_status read_status_word(const void* workspace, int64_t M, int64_t K, int index,
                            int64_t* value, cudaStream_t stream) {
  if (!workspace || !value) return H3Q_ERR_INVALID_ARG;
  if (M < 1 || K < 1) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(workspace)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  const uint8_t* wsp = static_cast<const uint8_t*>(workspace);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, wsp + h3q::workspace_layout(M, 1, K).status + 4 * index,
                      sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  *value = int64_t(word);
  return H3Q_OK;
}

// The launch sequence of a (grouped) Linear call; the per-Linear pointers are
// already checked.
h3q_status run_linear(const uint16_t* x, int8_t* xq, float* xs, const h3q::LinearGroup& grp,
                      int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (!xs || !workspace) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(M, N, K)) return st;
  const h3q::WorkspaceLayout lay = h3q::workspace_layout(M, N, K, grp.G);
  if (workspace_bytes < lay.total) return H3Q_ERR_INVALID_ARG;
  const void* ptrs[] = {x, xq, xs, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;

  uint8_t* wsp = static_cast<uint8_t*>(workspace);
  uint16_t* act = reinterpret_cast<uint16_t*>(wsp + lay.act);
  uint32_t* amax = reinterpret_cast<uint32_t*>(wsp + lay.amax);
  uint32_t* status = reinterpret_cast<uint32_t*>(wsp + lay.status);
  uint32_t* nwpart = reinterpret_cast<uint32_t*>(wsp + lay.nwpart);
  uint2* list = reinterpret_cast<uint2*>(wsp + lay.list);
  const bool code_acts = x || xq;
  // Zero the status block, and the activation norm maxima when the
  // activations are coded anew (they sit just before the status block).
  const size_t zero_from = code_acts ? lay.amax : lay.status;
  if (cudaMemsetAsync(wsp + zero_from, 0, lay.nwpart - zero_from, stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  // A2, or the FP16 coding of pre-quantised activations, or (x == xq == NULL)
  // the activations a previous call left coded in this workspace.
  const int64_t ldh = h3q::gemm_tc_coded_ld(K);
  if (x) {
    if (h3q_status st =
            from_cuda(h3q::launch_quantize_act(x, M, K, xq, xs, act, ldh, amax, stream, status)))
      return st;
  } else if (xq) {
    if (h3q_status st = from_cuda(h3q::launch_int8_to_f16(xq, M, K, ldh, act, amax, stream)))
      return st;
  }
  // Weight-row norms, where the activations alone do not settle exactness.
  if (h3q_status st =
          from_cuda(h3q::launch_weight_norms(grp, N, K, amax, M, nwpart, stream)))
    return st;
  // A3 + A4: the tiles kept on one accumulator (exact over the whole K, or
  // through checked checkpoints), of every Linear in one launch; then the
  // rest of every Linear in K chunks, in one more launch (which exits at
  // once when there are none).
  if (h3q_status st = from_cuda(h3q::launch_gemm_wide(act, xs, grp, M, N, K, amax, nwpart,
                                                      status, list, stream)))
    return st;
  const size_t cap = h3q::fallback_list_capacity(M, N);
  if (h3q_status st = from_cuda(h3q::launch_gemm_tc(act, xs, grp, M, N, K, status, list,
                                                    status + 2, cap, stream)))
    return st;
  return H3Q_OK;
}

}  // namespace

extern "C" {

const char* h3q_status_string(int status) {
  switch (status) {
    case H3Q_OK: return "ok";
    case H3Q_ERR_INVALID_ARG: return "invalid argument";
    case H3Q_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case H3Q_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case H3Q_ERR_NONFINITE: return "non-finite weight";
    case H3Q_ERR_CUDA: return "CUDA error";
    case H3Q_ERR_TIMEOUT: return "device-side wait timed out";
    case H3Q_ERR_NO_DEVICE: return "no sm_103 CUDA device is current";
    default: return "unknown status";
  }
}

int h3q_version(void) { return 100; }

h3q_status h3q_quantize_weights(const void* w, int w_dtype, int64_t N, int64_t K,
                                int8_t* q_out, float* scale_out, cudaStream_t stream) {
  if (!w || !q_out || !scale_out) return H3Q_ERR_INVALID_ARG;
  if (w_dtype != H3Q_DTYPE_F32 && w_dtype != H3Q_DTYPE_BF16) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(1, N, K)) return st;
  if (!aligned16(w) || !aligned16(q_out) || !aligned16(scale_out)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  if (h3q_status st = from_cuda(h3q::launch_quantize_weights(w, w_dtype, N, K, q_out,
                                                             scale_out, stream)))
    return st;
  // Offline call: read the scales back and reject any non-finite (NaN-marked) row.
  std::vector<float> host(static_cast<size_t>(N));
  if (cudaMemcpyAsync(host.data(), scale_out, size_t(N) * sizeof(float), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  for (float s : host)
    if (!(s > 0.f && s <= 3.4028234663852886e38f)) return H3Q_ERR_NONFINITE;
  return H3Q_OK;
}

h3q_status h3q_quantize_act(const uint16_t* x, int64_t M, int64_t K, int8_t* q_out,
                            float* scale_out, cudaStream_t stream) {
  if (!x || !q_out || !scale_out) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(M, 1, K)) return st;
  if (!aligned16(x) || !aligned16(q_out) || !aligned16(scale_out)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  return from_cuda(
      h3q::launch_quantize_act(x, M, K, q_out, scale_out, nullptr, K, nullptr, stream));
}

size_t h3q_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  return h3q::workspace_layout(M, N, K).total;
}

h3q_status h3q_linear_w8a8(const uint16_t* x, int8_t* xq, float* xs, const int8_t* wq,
                           const float* ws, const uint16_t* bias, int64_t M, int64_t N,
                           int64_t K, uint16_t* y, int32_t* acc_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!wq || !ws) return H3Q_ERR_INVALID_ARG;
  if (!y && !acc_out) return H3Q_ERR_INVALID_ARG;  // nothing to write
  const void* ptrs[] = {wq, ws, bias, y, acc_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
  h3q::LinearGroup grp = {};
  grp.G = 1;
  grp.wq[0] = wq;
  grp.ws[0] = ws;
  grp.bias[0] = bias;
  grp.y[0] = y;
  grp.acc[0] = acc_out;
  return run_linear(x, xq, xs, grp, M, N, K, workspace, workspace_bytes, stream);
}

size_t h3q_linear_grouped_workspace_bytes(int G, int64_t M, int64_t N, int64_t K) {
  if (G < 1 || G > h3q::kMaxGroup || M < 1 || N < 1 || K < 1) return 0;
  return h3q::workspace_layout(M, N, K, G).total;
}

h3q_status h3q_linear_w8a8_grouped(const uint16_t* x, int8_t* xq, float* xs, int G,
                                   const int8_t* const* wq, const float* const* ws,
                                   const uint16_t* const* bias, int64_t M, int64_t N, int64_t K,
                                   uint16_t* const* y, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  if (G < 1 || G > h3q::kMaxGroup) return H3Q_ERR_INVALID_ARG;
  if (!wq || !ws || !y) return H3Q_ERR_INVALID_ARG;
  h3q::LinearGroup grp = {};
  grp.G = G;
  for (int g = 0; g < G; ++g) {
    if (!wq[g] || !ws[g] || !y[g]) return H3Q_ERR_INVALID_ARG;
    const void* ptrs[] = {wq[g], ws[g], bias ? bias[g] : nullptr, y[g]};
    for (const void* p : ptrs)
      if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
    grp.wq[g] = wq[g];
    grp.ws[g] = ws[g];
    grp.bias[g] = bias ? bias[g] : nullptr;
    grp.y[g] = y[g];
    grp.acc[g] = nullptr;
  }
  return run_linear(x, xq, xs, grp, M, N, K, workspace, workspace_bytes, stream);
}

h3q_status h3q_workspace_status(const void* workspace, int64_t M, int64_t K,
                                cudaStream_t stream) {
  if (!workspace) return H3Q_ERR_INVALID_ARG;
  if (M < 1 || K < 1) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(workspace)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  const uint8_t* wsp = static_cast<const uint8_t*>(workspace);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, wsp + h3q::workspace_layout(M, 1, K).status, sizeof(word),
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  return word ? H3Q_ERR_TIMEOUT : H3Q_OK;
}

h3q_status h3q_linear_chunked_tiles(const void* workspace, int64_t M, int64_t K,
                                    int64_t* tiles, cudaStream_t stream) {
  return read_status_word(workspace, M, K, 1, tiles, stream);
}

h3q_status h3q_linear_checkpointed_tiles(const void* workspace, int64_t M, int64_t K,
                                         int64_t* tiles, cudaStream_t stream) {
  return read_status_word(workspace, M, K, 6, tiles, stream);
}

h3q_status h3q_quantize_weights_affine(const void* w, int w_dtype, int bits, int64_t N,
                                       int64_t K, uint8_t* q_out, float* ab_out,
                                       cudaStream_t stream) {
  if (!w || !q_out || !ab_out) return H3Q_ERR_INVALID_ARG;
  if (w_dtype != H3Q_DTYPE_F32 && w_dtype != H3Q_DTYPE_BF16) return H3Q_ERR_INVALID_ARG;
  if (bits != 8 && bits != 4) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(1, N, K)) return st;
  if (K % 64) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w) || !aligned16(q_out) || !aligned16(ab_out)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  if (h3q_status st = from_cuda(h3q::launch_quantize_weights_affine(w, w_dtype, bits, N, K,
                                                                    q_out, ab_out, stream)))
    return st;
  // Offline call: read the steps back and reject any NaN-marked (non-finite) group.
  std::vector<float> host(static_cast<size_t>(N) * size_t(K / 64) * 2);
  if (cudaMemcpyAsync(host.data(), ab_out, host.size() * sizeof(float), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  for (size_t i = 0; i < host.size(); i += 2)
    if (!(host[i] > 0.f && host[i] <= 3.4028234663852886e38f)) return H3Q_ERR_NONFINITE;
  return H3Q_OK;
}

h3q_status h3q_linear_affine_w8(const uint16_t* x, const uint8_t* q, const float* ab,
                                const uint16_t* bias, int64_t M, int64_t N, int64_t K,
                                uint16_t* y, uint32_t* status, cudaStream_t stream) {
  if (!x || !q || !ab || !y || !status) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(M, N, K)) return st;
  if (K % 64) return H3Q_ERR_UNSUPPORTED_SHAPE;
  const void* ptrs[] = {x, q, ab, bias, y, status};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), stream) != cudaSuccess) return H3Q_ERR_CUDA;
  h3q::LinearGroup grp = {};
  grp.G = 1;
  grp.wq[0] = reinterpret_cast<const int8_t*>(q);
  grp.bias[0] = bias;
  grp.y[0] = y;
  const float* abs_[1] = {ab};
  return from_cuda(h3q::launch_gemm_affine(x, grp, abs_, M, N, K, status, stream));
}

h3q_status h3q_linear_w8a8_mma_sync(const int8_t* xq, const float* xs, const int8_t* wq,
                                    const float* ws, const uint16_t* bias, int64_t M, int64_t N,
                                    int64_t K, uint16_t* y, int32_t* acc_out,
                                    cudaStream_t stream) {
  if (!xq || !xs || !wq || !ws) return H3Q_ERR_INVALID_ARG;
  if (!y && !acc_out) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = check_shape(M, N, K)) return st;
  const void* ptrs[] = {xq, xs, wq, ws, bias, y, acc_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;
  return from_cuda(h3q::launch_gemm_mma_s8(xq, xs, wq, ws, bias, M, N, K, y, acc_out, stream));
}

}  // extern "C"
