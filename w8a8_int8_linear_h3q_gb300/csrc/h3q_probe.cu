// h3q_probe.cu -- throughput probes of the tensor instructions this library
// stands on.
//
// INT8: sm_103a has no INT8 form of tcgen05.mma; its one INT8 tensor
// instruction is the warp-level mma.sync m16n8k32 s8 x s8 -> s32, the
// denominator of "% of dense INT8 peak".  This probe measures what that
// instruction sustains: every warp of a full grid (4 blocks of 8 warps on
// every SM) runs 8 independent accumulator chains of it, so that issue and
// not dependency latency bounds the rate, and the launch is timed with CUDA
// events.  One m16n8k32 is 2 * 16 * 8 * 32 = 8192 integer operations
// (multiply and add counted separately).
//
// FP16: the instruction the hot GEMM issues for its exact INT8 products,
// tcgen05.mma.cta_group::2.kind::f16 with M = N = 256, K = 16 and an FP32
// accumulator in TMEM.  Every CTA pair of a full grid (one CTA per SM) keeps
// one k-block of operands resident -- B in shared memory with the 128-byte
// swizzle, A in TMEM as the hot kernel feeds it, or in shared memory -- and
// one thread of the even CTA issues MMAs over it back to back; nothing else
// runs, so the rate is the instruction's own ceiling on this part, the
// figure the hot kernel's tensor-pipe share is measured against.
#include <cuda_fp16.h>

#include "h3q_abi_checks.cuh"
#include "h3q_internal.cuh"
#include "h3q_tc_ptx.cuh"

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

namespace P = ptx;

constexpr int kPairProbeThreads = 128;        // 4 warps: one per TMEM lane quarter
constexpr uint32_t kPairProbeCols = 512;      // D in columns 0-255, A in 256-287
constexpr uint32_t kPairProbeA = 256;
constexpr double kFlopsPerPairMma = 2.0 * 256 * 256 * 16;

struct PairProbeSmem {
  uint16_t b[128 * 64];                       // this CTA's 128 rows of B, one 64-deep k-block
  uint16_t a[128 * 64];                       // this CTA's 128 rows of A (shared-memory form)
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};
// more than half an SM's shared memory, so that each SM holds one CTA (and
// the CTA the whole of TMEM)
constexpr size_t kPairProbeSmemBytes = 120 * 1024;
static_assert(sizeof(PairProbeSmem) + 1024 <= kPairProbeSmemBytes, "probe shared memory");

__device__ uint32_t g_pair_probe_err;

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread of the
// even CTA of a pair (each CTA holds 128 of the 256 rows of A).
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint16_t small_int_f16(int i, int mul, int add) {
  return __half_as_ushort(__int2half_rn((i * mul + add) % 255 - 127));
}

__global__ void __launch_bounds__(kPairProbeThreads, 1)
mma_f16_pair_probe_kernel(int iters, int a_in_smem) {
  extern __shared__ uint8_t smem_raw[];
  PairProbeSmem& sm = *reinterpret_cast<PairProbeSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = P::cluster_rank();
  // operands: small integers, exact in FP16, as the hot kernel's INT8 codes
  for (int i = threadIdx.x; i < 128 * 64; i += kPairProbeThreads) {
    sm.b[i] = small_int_f16(i, 37, 11 * int(rank));
    sm.a[i] = small_int_f16(i, 53, 5 * int(rank));
  }
  if (threadIdx.x == 0) {
    P::mbar_init(&sm.done, 1);
    sm.abort_flag = 0;
    P::fence_mbar_init();
  }
  // the tensor core reads shared memory through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) P::tmem_alloc_pair(&sm.tmem_base, kPairProbeCols);
  P::tc_fence_before();
  __syncthreads();
  P::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // A in TMEM: this warp's 32 lanes, one k-block (32 columns of FP16 pairs)
  uint32_t h[32];
#pragma unroll
  for (int j = 0; j < 32; ++j)
    h[j] = uint32_t(small_int_f16(lane, 7, 3 * j + warp)) |
           (uint32_t(small_int_f16(lane, 13, 5 * j + warp)) << 16);
  P::tmem_st32(tmem + (uint32_t(32 * warp) << 16) + kPairProbeA, h);
  P::tmem_wait_st();
  P::tc_fence_before();
  __syncthreads();
  P::cluster_sync();                              // both CTAs' operands are in place
  P::tc_fence_after();
  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t idesc = P::idesc_f16_f32(256, 256);
    const uint64_t bdesc = P::smem_desc_sw128(P::smem_u32(sm.b));
    const uint64_t adesc = P::smem_desc_sw128(P::smem_u32(sm.a));
    if (a_in_smem) {
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss_pair(tmem, adesc + uint64_t(kk * 2), bdesc + uint64_t(kk * 2), idesc,
                          (it | kk) ? 1u : 0u);
    } else {
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          P::mma_f16_ts_pair(tmem, tmem + kPairProbeA + uint32_t(kk * 8),
                             bdesc + uint64_t(kk * 2), idesc, (it | kk) ? 1u : 0u);
    }
    P::mma_commit_pair_mc(&sm.done, 1);
    if (!P::mbar_wait(&sm.done, 0, &sm.abort_flag, &g_pair_probe_err, 1u)) {
      // a timeout is recorded; still let the MMAs finish before TMEM is freed
      int no_abort = 0;
      volatile int* never = &no_abort;
      P::mbar_wait(&sm.done, 0, never, &g_pair_probe_err, 1u);
    }
  }
  P::tc_fence_before();
  __syncthreads();
  P::cluster_sync();                              // the MMAs are done with both CTAs' TMEM
  if (warp == 0) {
    P::tc_fence_after();
    P::tmem_dealloc_pair(tmem, kPairProbeCols);
  }
  P::cluster_sync();
}

}  // namespace
}  // namespace h3q

extern "C" h3q_status h3q_probe_mma_f16_pair_tflops(double* tflops, int a_in_smem,
                                                    cudaStream_t stream) {
  if (!tflops || (a_in_smem != 0 && a_in_smem != 1)) return H3Q_ERR_INVALID_ARG;
  *tflops = 0.0;
  if (h3q_status st = h3q::check_device()) return st;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaFuncSetAttribute(h3q::mma_f16_pair_probe_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(h3q::kPairProbeSmemBytes)) != cudaSuccess) {
    cudaGetLastError();
    return H3Q_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(h3q::kPairProbeThreads);
  cfg.dynamicSmemBytes = h3q::kPairProbeSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many pairs as can be resident at once (one wave), at most one per SM pair
  cfg.gridDim = dim3(unsigned(sms & ~1));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, h3q::mma_f16_pair_probe_kernel, &cfg) !=
          cudaSuccess ||
      clusters < 1) {
    cudaGetLastError();
    return H3Q_ERR_CUDA;
  }
  clusters = clusters < sms / 2 ? clusters : sms / 2;
  cfg.gridDim = dim3(unsigned(2 * clusters));
  const int iters = 16384;             // 65536 pair MMAs per pair: about 4 ms at 2 GHz
  const uint32_t zero = 0;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  h3q_status st = H3Q_OK;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(h3q::g_pair_probe_err, &zero, sizeof(zero), 0,
                              cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaLaunchKernelEx(&cfg, h3q::mma_f16_pair_probe_kernel, 256, a_in_smem) != cudaSuccess ||
      cudaEventRecord(e0, stream) != cudaSuccess ||
      cudaLaunchKernelEx(&cfg, h3q::mma_f16_pair_probe_kernel, iters, a_in_smem) !=
          cudaSuccess ||
      cudaEventRecord(e1, stream) != cudaSuccess) {
    st = H3Q_ERR_CUDA;
  } else {
    float ms = 0.f;
    uint32_t err = 0;
    if (cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || !(ms > 0.f) ||
        cudaMemcpyFromSymbol(&err, h3q::g_pair_probe_err, sizeof(err)) != cudaSuccess) {
      st = H3Q_ERR_CUDA;
    } else if (err) {
      st = H3Q_ERR_TIMEOUT;
    } else {
      *tflops = double(clusters) * double(iters) * 4.0 * h3q::kFlopsPerPairMma /
                (double(ms) * 1e-3) / 1e12;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaGetLastError();
  return st;
}

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
