// h3q_probe.cu -- throughput probe of the INT8 tensor instruction this part
// offers, the denominator of "% of dense INT8 peak".
//
// sm_103a has no INT8 form of tcgen05.mma; its one INT8 tensor instruction
// is the warp-level mma.sync m16n8k32 s8 x s8 -> s32.  This probe measures
// what that instruction sustains: every warp of a full grid (4 blocks of 8
// warps on every SM) runs 8 independent accumulator chains of it, so that
// issue and not dependency latency bounds the rate, and the launch is timed
// with CUDA events.  One m16n8k32 is 2 * 16 * 8 * 32 = 8192 integer
// operations (multiply and add counted separately).
#include "h3q_abi_checks.cuh"
#include "h3q_internal.cuh"

namespace h3q {
namespace {

constexpr int kProbeWarps = 8;       // warps per block
constexpr int kProbeBlocksPerSm = 4;
constexpr int kChains = 8;           // independent accumulators per warp
constexpr double kOpsPerMma = 2.0 * 16 * 8 * 32;

// The accumulators are folded into a value that is stored only if it equals
// an unlikely constant, so that the compiler keeps every MMA (results that
// are never used would be removed).
__device__ int g_probe_sink;

__global__ void __launch_bounds__(32 * kProbeWarps)
mma_s8_probe_kernel(int iters, uint32_t seed) {
  // operand fragments: any values, distinct per lane so that nothing is uniform
  const uint32_t a0 = seed ^ (threadIdx.x * 0x01010101u), a1 = a0 + 0x02020202u,
                 a2 = a0 ^ 0x40404040u, a3 = a1 ^ 0x20202020u;
  const uint32_t b0 = a0 * 3u, b1 = a1 * 5u;
  int d[kChains][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};\n"
          : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int sum = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) sum += d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3];
  if (sum == 0x7A5A5A5A) g_probe_sink = sum;
}

}  // namespace
}  // namespace h3q

extern "C" h3q_status h3q_probe_mma_s8_tops(double* tops, cudaStream_t stream) {
  if (!tops) return H3Q_ERR_INVALID_ARG;
  *tops = 0.0;
  if (h3q_status st = h3q::check_device()) return st;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_CUDA;
  }
  const dim3 grid(unsigned(h3q::kProbeBlocksPerSm * sms)), block(32 * h3q::kProbeWarps);
  const int iters = 16384;             // about 40 ms at 150 TOPS
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  h3q_status st = H3Q_OK;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    st = H3Q_ERR_CUDA;
  } else {
    h3q::mma_s8_probe_kernel<<<grid, block, 0, stream>>>(256, 1u);   // warm-up
    cudaEventRecord(e0, stream);
    h3q::mma_s8_probe_kernel<<<grid, block, 0, stream>>>(iters, 7u);
    cudaEventRecord(e1, stream);
    float ms = 0.f;
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || !(ms > 0.f)) {
      st = H3Q_ERR_CUDA;
    } else {
      const double ops = double(grid.x) * h3q::kProbeWarps * double(iters) * h3q::kChains *
                         h3q::kOpsPerMma;
      *tops = ops / (double(ms) * 1e-3) / 1e12;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaGetLastError();
  return st;
}
