// h3q_gemm_mma.cu -- A3 + A4 on the warp-level INT8 tensor path.
//
//   acc[m,n] = sum_k qa[m,k] * qw[n,k]           (mma.sync m16n8k32 s8 -> s32, exact)
//   y[m,n]   = BF16_RNE(acc * sa[m] * sw[n] + bias[n])       (h3q_epilogue.cuh)
//
// Sources: "feat(mps): support MiniMax-H3 INT8 inference on Apple M5"
// (LightX2V #1672), Validation (INT32 product of INT8 operands) and
// Summary by CodeRabbit (exact K tiles, no K padding); "MLX implementation
// and experiment report", What the default preserves (bias added before the
// one rounding of the output).
//
// Both operands are K-major INT8, so ldmatrix (no transpose) yields the
// m16n8k32 fragments of A (row-major) and B (column-major) directly.  Tiles are
// 128 x 128 x 64 with a 4-stage cp.async pipeline; rows past M or N and K
// chunks past K are zero-filled, so ragged tiles need no special case.  This
// is the legacy tensor path, kept as the exact baseline that the tcgen05
// kernel is measured against.
#include <cuda_bf16.h>

#include "h3q_epilogue.cuh"
#include "h3q_internal.cuh"

namespace h3q {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int kTileBytes = BM * BK;                 // one operand stage (BM == BN)
constexpr int kSmemBytes = STAGES * 2 * kTileBytes; // 64 KB

// Byte offset of 16-byte chunk `c` (0..3) of row `r` in a [rows x 64 B] tile,
// XOR-swizzled so that the 8 rows an ldmatrix phase reads hit 8 distinct
// 16-byte bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return uint32_t(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(THREADS)
gemm_mma_s8_kernel(const int8_t* __restrict__ A, const float* __restrict__ sa,
                   const int8_t* __restrict__ B, const float* __restrict__ sw,
                   const uint16_t* __restrict__ bias, int M, int N, int K,
                   uint16_t* __restrict__ Y, int32_t* __restrict__ ACC) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;            // 2 x 4 warps, warp tile 64 x 32
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int KT = (K + BK - 1) / BK;
  const uint32_t sbase = smem_u32(smem);

  auto load_stage = [&](int stage, int k0) {
    const uint32_t sA = sbase + stage * 2 * kTileBytes, sB = sA + kTileBytes;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * THREADS;               // 512 chunks of 16 B per operand
      const int r = idx >> 2, c = idx & 3, gk = k0 + c * 16;
      const bool kok = gk < K;
      const bool va = kok && (m0 + r) < M, vb = kok && (n0 + r) < N;
      cp_async16(sA + swz(r, c), va ? A + int64_t(m0 + r) * K + gk : A, va);
      cp_async16(sB + swz(r, c), vb ? B + int64_t(n0 + r) * K + gk : B, vb);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_stage(s, s * BK);
    asm volatile("cp.async.commit_group;\n" ::);
  }

  for (int kt = 0; kt < KT; ++kt) {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(STAGES - 2));
    __syncthreads();
    const int nxt = kt + STAGES - 1;
    if (nxt < KT) load_stage(nxt % STAGES, nxt * BK);
    asm volatile("cp.async.commit_group;\n" ::);

    const uint32_t sA = sbase + (kt % STAGES) * 2 * kTileBytes, sB = sA + kTileBytes;
#pragma unroll
    for (int kc = 0; kc < 4; kc += 2) {               // two k32 steps per 64-byte stage
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = wm * 64 + i * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4(sA + swz(r, kc + (lane >> 4)), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
        ldsm_x4(sB + swz(r, kc + ((lane >> 3) & 1)), bf[2 * j][0], bf[2 * j][1],
                bf[2 * j + 1][0], bf[2 * j + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::);

  // Epilogue: thread holds rows g, g+8 and columns 2t, 2t+1 of each m16n8 tile.
  const int g = lane >> 2, t = lane & 3;
  const bool n_even = (N & 1) == 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = n0 + wn * 32 + j * 8 + 2 * t;
    if (n >= N) continue;
    const bool two = n + 1 < N;
    const float sw0 = sw[n], sw1 = two ? sw[n + 1] : 0.f;
    const float b0 = bias ? bias_value(bias[n]) : 0.f;
    const float b1 = (bias && two) ? bias_value(bias[n + 1]) : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = m0 + wm * 64 + i * 16 + g + 8 * h;
        if (m >= M) continue;
        const int a0 = acc[i][j][2 * h], a1 = acc[i][j][2 * h + 1];
        const int64_t off = int64_t(m) * N + n;
        if (ACC) {
          if (two && n_even) {
            *reinterpret_cast<int2*>(ACC + off) = make_int2(a0, a1);
          } else {
            ACC[off] = a0;
            if (two) ACC[off + 1] = a1;
          }
        }
        if (Y) {
          const float s = sa[m];
          const __nv_bfloat162 v = __floats2bfloat162_rn(epilogue_value(a0, s, sw0, b0),
                                                         epilogue_value(a1, s, sw1, b1));
          if (two && n_even) {
            *reinterpret_cast<__nv_bfloat162*>(Y + off) = v;
          } else {
            Y[off] = __bfloat16_as_ushort(v.x);
            if (two) Y[off + 1] = __bfloat16_as_ushort(v.y);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_mma_s8(const int8_t* qa, const float* sa, const int8_t* qw,
                               const float* sw, const uint16_t* bias, int64_t M, int64_t N,
                               int64_t K, uint16_t* y, int32_t* acc, cudaStream_t s) {
  // Set on every call: the attribute belongs to the current device's context.
  cudaError_t e = cudaFuncSetAttribute(gemm_mma_s8_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(unsigned((M + BM - 1) / BM), unsigned((N + BN - 1) / BN));
  gemm_mma_s8_kernel<<<grid, THREADS, kSmemBytes, s>>>(qa, sa, qw, sw, bias, int(M), int(N),
                                                       int(K), y, acc);
  return cudaGetLastError();
}

}  // namespace h3q
