// h3q_selftest.cu -- a check of the device-side failure path.
//
// Every wait in the library's kernels is bounded (the mbarrier helpers of
// h3q_tc_ptx.cuh): after the limit the kernel records a bit in the call's
// status word and returns, so a lost arrival becomes an error the host reads
// instead of a hung GPU.  This probe drives that path on purpose without any
// fault: one thread waits on an mbarrier that nothing arrives on, with the
// same helper the GEMM kernels use, until the helper gives up.
#include "h3q_internal.cuh"
#include "h3q_tc_ptx.cuh"

namespace h3q {
namespace {

constexpr uint32_t kProbeBit = 1u << 24;

__global__ void bounded_wait_probe_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // phase 0 never completes: the wait runs to its limit, then sets the bit
  if (threadIdx.x == 0) ptx::mbar_wait(&bar, 0, &abort_flag, status, kProbeBit);
}

}  // namespace
}  // namespace h3q

extern "C" h3q_status h3q_selftest_bounded_wait(uint32_t* status, cudaStream_t stream) {
  if (!status) return H3Q_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(status) % 4) return H3Q_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_NO_DEVICE;
  }
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), stream) != cudaSuccess) return H3Q_ERR_CUDA;
  h3q::bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(status);
  if (cudaGetLastError() != cudaSuccess) return H3Q_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, status, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return H3Q_ERR_CUDA;
  return word ? H3Q_ERR_TIMEOUT : H3Q_OK;
}
