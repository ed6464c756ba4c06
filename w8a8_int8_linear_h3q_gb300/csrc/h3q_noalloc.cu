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
// address.  Its device address is looked up with cudaGetSymbolAddress, with
// the device current, once per CUDA context, and kept: a device reset makes a
// new primary context, in which the module and the array are loaded anew, so
// the next call looks the address up again.
#include <cuda.h>

#include <mutex>
#include <vector>

#include "h3q_abi_checks.cuh"
#include "h3q_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// A driver entry point, looked up through the runtime (no -lcuda).
void* driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    p = nullptr;
  return p;
}

// The process-unique ID of the current context, or 0 if there is none.
// (Unlike the context handle, an ID is never reused after a context is
// destroyed, so a reset device cannot match a stale entry.)
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
  static const CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get || !get_id || get(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

struct CachedAddress {
  unsigned long long ctx_id;
  void* ptr;
};

std::mutex g_mu;
std::vector<CachedAddress> g_cache;

// Device address of g_scratch in the current context: looked up on the first
// call in that context (cudaGetSymbolAddress also makes the device's primary
// context current if no context is), then taken from the cache.  The caller
// has checked the device.
h3q_status scratch_for_current_device(void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = current_context_id();
  if (id)
    for (const CachedAddress& c : g_cache)
      if (c.ctx_id == id) {
        *out = c.ptr;
        return H3Q_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return H3Q_ERR_CUDA;
  }
  if (!id) id = current_context_id();
  if (!id) return H3Q_ERR_CUDA;
  g_cache.push_back({id, p});
  *out = p;
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
  if (h3q_status st = h3q::check_device()) return st;
  void* scratch = nullptr;
  if (h3q_status st = scratch_for_current_device(&scratch)) return st;
  return h3q_linear_w8a8(x, xq, xs, wq, ws, bias, M, N, K, y, acc_out, scratch, kScratchBytes,
                         stream);
}

h3q_status h3q_linear_w8a8_noalloc_status(int64_t M, int64_t K, cudaStream_t stream) {
  if (M < 1 || K < 16) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (h3q_linear_workspace_bytes(M, 1, K) > kScratchBytes) return H3Q_ERR_UNSUPPORTED_SHAPE;
  if (h3q_status st = h3q::check_device()) return st;
  void* scratch = nullptr;
  if (h3q_status st = scratch_for_current_device(&scratch)) return st;
  return h3q_workspace_status(scratch, M, K, stream);
}

}  // extern "C"
