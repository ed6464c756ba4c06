// h3q_noalloc.cu -- h3q_linear_w8a8 for callers that cannot allocate device
// memory.
//
// Some callers run where a device allocation is not allowed or not safe at
// call time: an inference engine's plugin enqueue that is handed only its
// input and output buffers, or a serving loop that must not block on (or fail
// in) the allocator once it is warmed up.  For them this entry point takes the
// scratch that h3q_linear_w8a8 needs from a fixed array compiled into the
// library instead of a caller-provided workspace.
//
// The array lives in device memory of every GPU that loads the library, for as
// long as the process runs.  Host code must not hand its symbol to a kernel:
// on the host the name stands for a host-side placeholder, not a device
// address.  Its device address is looked up once per device with
// cudaGetSymbolAddress and kept.
#include <mutex>

#include "h3q_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 256;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on first use).
h3q_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return H3Q_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return H3Q_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return H3Q_OK;
}

}  // namespace

extern "C" {

h3q_status h3q_linear_w8a8_noalloc(const uint16_t* x, int8_t* xq, float* xs, const int8_t* wq,
                                   const float* ws, const uint16_t* bias, int64_t M, int64_t N,
                                   int64_t K, uint16_t* y, int32_t* acc_out,
                                   cudaStream_t stream) {
  if (!x && !xq) return H3Q_ERR_INVALID_ARG;   // no reuse of earlier contents here
  if (!xs || !wq || !ws) return H3Q_ERR_INVALID_ARG;
  if (!y && !acc_out) return H3Q_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 16) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (h3q_linear_workspace_bytes(M, N, K) > kScratchBytes) return H3Q_ERR_UNSUPPORTED_SHAPE;
  void* scratch = nullptr;
  if (h3q_status st = scratch_for_current_device(&scratch)) return st;
  return h3q_linear_w8a8(x, xq, xs, wq, ws, bias, M, N, K, y, acc_out, scratch, kScratchBytes,
                         stream);
}

}  // extern "C"
