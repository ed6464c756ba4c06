// h3q_api.cu -- the C ABI declared in include/h3q.h: argument validation,
// device check, and the launch sequence of each entry point.  No entry point
// allocates device memory; every launch goes on the caller's stream.
#include <cstdio>
#include <vector>

#include "h3q_internal.cuh"

namespace {

constexpr int64_t kMaxK = 133143;            // K * 127^2 < 2^31
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxN = int64_t(65535) * 128;

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

h3q_status from_cuda(cudaError_t e) { return e == cudaSuccess ? H3Q_OK : H3Q_ERR_CUDA; }

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
  return from_cuda(h3q::launch_quantize_act(x, M, K, q_out, scale_out, nullptr, stream));
}

size_t h3q_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)N;
  if (M < 1 || K < 1) return 0;
  const size_t b = size_t(M) * size_t(K) * 2u;      // FP16-coded activations
  return (b + 255u) & ~size_t(255);
}

h3q_status h3q_linear_w8a8(const uint16_t* x, int8_t* xq, float* xs, const int8_t* wq,
                           const float* ws, const uint16_t* bias, int64_t M, int64_t N,
                           int64_t K, uint16_t* y, int32_t* acc_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!xs || !wq || !ws) return H3Q_ERR_INVALID_ARG;
  if (!x && !xq) return H3Q_ERR_INVALID_ARG;       // no activations at all
  if (!y && !acc_out) return H3Q_ERR_INVALID_ARG;  // nothing to write
  if (h3q_status st = check_shape(M, N, K)) return st;
  const size_t need = h3q_linear_workspace_bytes(M, N, K);
  if (x && !xq && (!workspace || workspace_bytes < need)) return H3Q_ERR_INVALID_ARG;
  const void* ptrs[] = {x, xq, xs, wq, ws, bias, y, acc_out, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = check_device()) return st;

  // A2 (unless pre-quantised).  The INT8 activations go to xq, or to the
  // workspace when the caller does not want them.
  int8_t* qa = xq ? xq : static_cast<int8_t*>(workspace);
  if (x) {
    if (h3q_status st = from_cuda(h3q::launch_quantize_act(x, M, K, qa, xs, nullptr, stream)))
      return st;
  }
  // A3 + A4.
  return from_cuda(h3q::launch_gemm_mma_s8(qa, xs, wq, ws, bias, M, N, K, y, acc_out, stream));
}

}  // extern "C"
