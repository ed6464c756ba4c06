// h3q_gemm_tc.cu -- A3 + A4 on the sm_103a 5th-generation tensor cores.
//
//   acc[m,n] = sum_k qa[m,k] * qw[n,k]          exact INT32
//   y[m,n]   = BF16_RNE(acc * sa[m] * sw[n] + bias[n])
//
// Sources: "feat(mps): support MiniMax-H3 INT8 inference on Apple M5"
// (LightX2V #1672) -- Validation (INT8 x INT8 with CPU INT32 references),
// opening description (native K = 5376, no K padding, no weight
// dequantisation), Summary by CodeRabbit (exact K tiles); "MLX implementation
// and experiment report", What the default preserves (bias before the one
// rounding).
//
// sm_103a has no INT8 tcgen05 MMA, so the product runs as exact integer
// arithmetic on the FP16 MMA (kind::f16, FP32 accumulate):
//   - every INT8 value is an FP16 value, every product |q_a q_w| <= 127^2 is
//     exact in FP32, and an FP32 sum of such integers is exact while every
//     partial sum stays within 2^24, which holds for any 1040 consecutive
//     K terms (2^24 / 127^2 = 1040.2);
//   - so K is cut into chunks of at most 1024, each chunk accumulates into a
//     fresh FP32 TMEM accumulator, and the epilogue warps fold every chunk
//     into INT32 running sums held in registers (cvt.rni of an
//     integer-valued FP32 is exact).  The result is the exact INT32 product.
// The weights stay INT8 in memory (no dequantisation).  TMA brings the INT8
// weights of a super-stage (two boxes of two k-blocks each) into 128-byte-
// swizzled shared memory; converter warps read their row from it, turn it
// into FP16 in registers and store it into TMEM, where the MMA reads it as its
// A operand.  The activations arrive already FP16-coded (written by the
// activation quantiser, rows padded with zeros to a multiple of 64) through
// TMA into 128-byte-swizzled shared memory: the B operand.  Copies are few
// and large: per super-stage one 3-D activation load per CTA (two whole
// k-block tiles, viewing a row as chunks of 64) and two weight loads.  The
// weights have their own producer and a deeper ring (three super-stages), so
// they are in shared memory before the converters need them; the activation
// slots are refilled as the MMAs release them.
//
// The MMA issue path is kept bare: on this part every instruction the
// issuing thread runs between two MMAs (a barrier wait, a commit) leaves the
// tensor pipe idle.  So the MMA thread synchronises once per super-stage of
// four k-blocks (16 MMAs): one wait on a barrier that the converter warps
// complete when both operands are in place (they also wait for the
// activation tiles), and one commit that frees the super-stage's activation
// and weight slots at once.
//
// Tile: 128 output channels (MMA M, TMEM lanes) x 128 tokens (MMA N).
// CTAs run in clusters of two that take adjacent channel blocks of the same
// token block (the fallback list names such channel-block pairs); each CTA
// loads all four activation tiles of a super-stage into its own shared
// memory, so the two CTAs share those tiles through L2 only, and a slot is
// refilled once this CTA's own MMAs have finished with it.  Persistent
// clusters walk the cluster tiles in groups of 16 token blocks so that the
// concurrently running tiles share weight and activation tiles in L2.
//
// Warp roles (480 threads):
//   warp 0      TMA producer of the activation tiles (2 super-stage slots)
//   warp 1      TMEM allocator and MMA issuer (the whole warp runs the loop,
//               one elected lane issues)
//   warp 2      TMA producer of the INT8 weight tiles (3 super-stage slots)
//   warps 3-6   converters: INT8 weights -> FP16 -> TMEM (2 super-stages)
//   warps 7-14  epilogue: chunk drains into INT32 running sums, then
//               dequant + bias + BF16 (and the optional raw INT32 output)
// TMEM: FP32 accumulators in columns 0-127 and 128-255, A super-stages in
// 256-383 and 384-511.
// Every wait is bounded in time; on a timeout the kernel records an error
// word, lets every role fall through, drains its in-flight copies and MMAs,
// frees TMEM and returns.
#include <cuda.h>

#include "h3q_epilogue.cuh"
#include "h3q_internal.cuh"
#include "h3q_tc_ptx.cuh"

namespace h3q {
namespace {

namespace P = ptx;

constexpr int BM = 128;                 // channels per tile
constexpr int BN = 128;                 // tokens per tile
constexpr int BK = 64;                  // K per k-block (128 bytes of FP16)
constexpr int SS = 4;                   // k-blocks per super-stage (16 MMAs)
constexpr int MAX_SS_PER_CHUNK = 4;     // 16 k-blocks = 1024 K: exact FP32 chunk
constexpr int SLOTS = 2;                // super-stage slots: activations (SMEM), FP16 weights (TMEM)
constexpr int W_SLOTS = 3;              // super-stage slots: INT8 weights (SMEM)
constexpr int GROUP_M = 16;             // token blocks per raster group
constexpr int CLUSTER = 2;              // CTAs on adjacent channel blocks of one token block
constexpr int NUM_CONV_WARPS = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int WPROD_WARP = 2;
constexpr int CONV_WARP0 = 3;
constexpr int EPI_WARP0 = CONV_WARP0 + NUM_CONV_WARPS;
constexpr int THREADS = 32 * (3 + NUM_CONV_WARPS + NUM_EPI_WARPS);
constexpr int B_STAGE_BYTES = BN * BK * 2;                 // 16 KB
constexpr int W_BOX_BYTES = BM * 2 * BK;                   // 16 KB: 128 rows x 2 k-blocks
constexpr uint32_t TM_D = 0;            // accumulators: cols 0-127 and 128-255
constexpr uint32_t TM_A = 256;          // A super-stages: 2 x (4 k-blocks x 32 cols)
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t IDESC = P::idesc_f16_f32(BM, BN);

// error word bits
constexpr uint32_t ERR_PRODUCER = 1u, ERR_MMA = 2u, ERR_CONVERT = 4u, ERR_EPILOGUE = 8u,
                   ERR_TEARDOWN = 16u;

struct __align__(1024) Smem {
  uint8_t b[SLOTS][SS][B_STAGE_BYTES];  // activation tiles of a super-stage slot
  uint8_t w[W_SLOTS][SS / 2][W_BOX_BYTES];  // INT8 weights: 128-byte rows, 128-byte swizzle
  uint64_t full_b[SLOTS];               // a slot's activation tiles have landed
  uint64_t full_w[W_SLOTS];             // a slot's INT8 weights have landed
  uint64_t empty_w[W_SLOTS];            // the converters have read them
  uint64_t full_a[SLOTS];               // A converted and B landed for a super-stage
  uint64_t empty_s[SLOTS];              // this CTA's MMAs are done with a slot
  uint64_t dfull[2];
  uint64_t dempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + slack for 1024-byte alignment

struct Shape {
  int G;              // Linears of the call (they share the activations)
  int list_cap;       // entries of one Linear's list
  int M, N, K;
  int KB;             // k-blocks
  int NSS;            // super-stages per tile
  int nchunks;        // exact-FP32 chunks per tile
  int sspc;           // super-stages per chunk (the last chunk may have fewer)
  int mt, nt;         // token blocks, channel blocks
  int ntc;            // channel-block groups of CLUSTER
  int tiles;          // cluster tiles: mt * ntc
};

// The weight maps and per-Linear operands of a call's G Linears.
struct Linears {
  CUtensorMap w[kMaxGroup];
  const float* sw[kMaxGroup];
  const uint16_t* bias[kMaxGroup];
  uint16_t* y[kMaxGroup];
  int32_t* acc[kMaxGroup];
};

// Cluster tile t -> Linear g, token block mb and the channel block nb of CTA
// `rank` (nb >= nt for the spare CTA of an odd channel-block count).  With
// lists, the tiles run through Linear 0's list, then Linear 1's, ... (cnt:
// the lists' lengths), and an entry names the tile: {token block,
// channel-block pair}.
__device__ __forceinline__ void tile_coords(const Shape& s, const uint2* list,
                                            const uint32_t (&cnt)[kMaxGroup], int t,
                                            uint32_t rank, int& g, int& mb, int& nb) {
  if (list) {
    g = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup - 1; ++i)
      if (g == i && t >= int(cnt[i])) {
        t -= int(cnt[i]);
        g = i + 1;
      }
    const uint2 e = list[int64_t(g) * s.list_cap + t];
    mb = int(e.x);
    nb = int(e.y) * CLUSTER + int(rank);
    return;
  }
  g = 0;
  const int per_group = GROUP_M * s.ntc;
  const int grp = t / per_group;                 // raster group of GROUP_M token blocks
  const int first_m = grp * GROUP_M;
  const int gm = min(GROUP_M, s.mt - first_m);
  const int r = t - grp * per_group;
  mb = first_m + r % gm;
  nb = (r / gm) * CLUSTER + int(rank);
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap act_map, const __grid_constant__ Linears lin,
               const float* __restrict__ sa, const Shape shp, uint32_t* __restrict__ err,
               const uint2* __restrict__ list, const uint32_t* __restrict__ list_len) {
  // With lists this grid may be scheduled before the kernel that writes them
  // has finished (programmatic dependent launch): wait for it first.  Every
  // CTA then reads the same tile counts, so all leave together (before any
  // cluster barrier) when there is nothing to do.
  if (list) ptx::grid_dependency_wait();
  uint32_t cnt[kMaxGroup] = {};
  int ntiles = shp.tiles;
  if (list) {
    ntiles = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup; ++i) {
      cnt[i] = i < shp.G ? list_len[i] : 0u;
      ntiles += int(cnt[i]);
    }
  }
  if (ntiles == 0) return;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_SLOTS; ++i) {
      P::mbar_init(&sm.full_w[i], 1);
      P::mbar_init(&sm.empty_w[i], NUM_CONV_WARPS * 32);
    }
    for (int i = 0; i < SLOTS; ++i) {
      P::mbar_init(&sm.full_b[i], 1);
      P::mbar_init(&sm.full_a[i], NUM_CONV_WARPS * 32);
      P::mbar_init(&sm.empty_s[i], 1);            // this CTA's commit
    }
    for (int i = 0; i < 2; ++i) {
      P::mbar_init(&sm.dfull[i], 1);
      P::mbar_init(&sm.dempty[i], NUM_EPI_WARPS * 32);
    }
    P::mbar_init(&sm.mma_done, 1);
    sm.abort_flag = 0;
    P::fence_mbar_init();
  }
  if (warp == 1) P::tmem_alloc(&sm.tmem_base, TM_COLS);
  P::tc_fence_before();
  __syncthreads();
  P::cluster_sync();                              // both CTAs of the cluster have started
  P::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t rank = P::cluster_rank();
  const int cid = int(P::cluster_id_x()), ncl = int(P::num_clusters_x());

  if (warp == 0) {
    // ---------------- TMA producer: activation tiles ----------------
    // warp-uniform: the waits by the whole warp, the copies by one elected lane
    const uint32_t leader = P::elect_one();
    if (leader) P::tma_prefetch_desc(&act_map);
    uint32_t gs = 0, gb = 0;             // super-stages seen, slots issued
    bool ok = true;
    for (int t = cid; ok && t < ntiles; t += ncl) {
      int g, mb, nb;
      tile_coords(shp, list, cnt, t, rank, g, mb, nb);
      for (int ss = 0; ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % SLOTS;
        // the slot is free once this CTA's MMAs finished its previous use
        if (!P::mbar_wait_warp(&sm.empty_s[slot], ((gs / SLOTS) & 1u) ^ 1u, abort_flag, err,
                               ERR_PRODUCER)) {
          ok = false;
          break;
        }
        // the super-stage's four activation tiles, two per copy (each box is
        // two whole k-block tiles); boxes past the last k-block arrive as zeros
        if (leader) {
          P::mbar_arrive_expect_tx(&sm.full_b[slot], SS * B_STAGE_BYTES);
#pragma unroll
          for (int h = 0; h < SS / 2; ++h)
            P::tma_load_3d(P::smem_u32(sm.b[slot][2 * h]), &act_map, &sm.full_b[slot], 0,
                           mb * BN, ss * SS + 2 * h);
        }
        __syncwarp();
        gb = gs + 1;
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (leader) {
      int no_abort = 0;
      volatile int* never = &no_abort;   // this drain does not follow the abort flag
      for (uint32_t i = gb > SLOTS ? gb - SLOTS : 0; i < gb; ++i)
        P::mbar_wait(&sm.full_b[i % SLOTS], (i / SLOTS) & 1u, never, err, ERR_TEARDOWN);
    }
    __syncwarp();
  } else if (warp == WPROD_WARP) {
    // ---------------- TMA producer: INT8 weight tiles ----------------
    const uint32_t leader = P::elect_one();
    if (leader)
      for (int i = 0; i < shp.G; ++i) P::tma_prefetch_desc(&lin.w[i]);
    uint32_t gs = 0, gw = 0;
    bool ok = true;
    for (int t = cid; ok && t < ntiles; t += ncl) {
      int g, mb, nb;
      tile_coords(shp, list, cnt, t, rank, g, mb, nb);
      const int wrow = min(nb, shp.nt - 1) * BM;
      for (int ss = 0; ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % W_SLOTS;
        if (!P::mbar_wait_warp(&sm.empty_w[slot], ((gs / W_SLOTS) & 1u) ^ 1u, abort_flag, err,
                               ERR_PRODUCER)) {
          ok = false;
          break;
        }
        if (leader) {
          P::mbar_arrive_expect_tx(&sm.full_w[slot], (SS / 2) * W_BOX_BYTES);
#pragma unroll
          for (int p = 0; p < SS / 2; ++p)
            P::tma_load_2d(P::smem_u32(sm.w[slot][p]), &lin.w[g], &sm.full_w[slot],
                           (ss * SS + 2 * p) * BK, wrow);
        }
        __syncwarp();
        gw = gs + 1;
      }
    }
    if (leader) {
      int no_abort = 0;
      volatile int* never = &no_abort;
      for (uint32_t i = gw > W_SLOTS ? gw - W_SLOTS : 0; i < gw; ++i)
        P::mbar_wait(&sm.full_w[i % W_SLOTS], (i / W_SLOTS) & 1u, never, err, ERR_TEARDOWN);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one wait and one commit per 16 MMAs ----------------
    // The whole warp runs the loop (warp-uniform waits, addresses and
    // descriptors) and one elected lane issues every MMA and commit: a loop run
    // by one lane alone loses issue slots to the busy warps of its SM
    // sub-partition, and the tensor pipe then waits for its MMAs.
    const uint32_t leader = P::elect_one();
    uint32_t gs = 0, gc = 0;            // super-stage and chunk counters
    bool ok = true;
    for (int t = cid; ok && t < ntiles; t += ncl) {
      for (int c = 0; ok && c < shp.nchunks; ++c, ++gc) {
        const int ss0 = c * shp.sspc, ss1 = min(shp.NSS, ss0 + shp.sspc);
        const uint32_t buf = gc & 1u;
        if (!P::mbar_wait_warp(&sm.dempty[buf], ((gc >> 1) & 1u) ^ 1u, abort_flag, err,
                               ERR_MMA)) {
          ok = false;
          break;
        }
        const uint32_t d_tmem = tmem + TM_D + buf * BN;
        for (int ss = ss0; ss < ss1; ++ss, ++gs) {
          const uint32_t slot = gs % SLOTS;
          if (!P::mbar_wait_warp(&sm.full_a[slot], (gs / SLOTS) & 1u, abort_flag, err, ERR_MMA)) {
            ok = false;
            break;
          }
          P::tc_fence_after();
          const uint32_t a_tmem = tmem + TM_A + slot * (SS * 32);
          const int nkb = min(SS, shp.KB - ss * SS);
          uint64_t bdesc[SS];
#pragma unroll
          for (int j = 0; j < SS; ++j) bdesc[j] = P::smem_desc_sw128(P::smem_u32(sm.b[slot][j]));
          if (leader) {
#pragma unroll
            for (int j = 0; j < SS; ++j) {
              if (j >= nkb) break;
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                P::mma_f16_ts(d_tmem, a_tmem + j * 32 + kk * 8, bdesc[j] + uint64_t(kk * 2),
                              IDESC, (ss > ss0 || j > 0 || kk > 0) ? 1u : 0u);
            }
            P::mma_commit(&sm.empty_s[slot]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) P::mma_commit(&sm.dfull[buf]);
        __syncwarp();
      }
    }
    // every MMA the leader issued has finished before TMEM is freed
    if (leader) {
      P::mma_commit(&sm.mma_done);
      int no_abort = 0;
      volatile int* never = &no_abort;
      P::mbar_wait(&sm.mma_done, 0, never, err, ERR_TEARDOWN);
    }
    __syncwarp();
  } else if (warp < EPI_WARP0) {
    // ---------------- converters: INT8 weights -> FP16 -> TMEM ----------------
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int r = 32 * q + lane;                  // channel row within the tile
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    // this row's 16-byte chunks in a 128-byte-swizzled INT8 box (two k-blocks)
    const uint32_t row_off = uint32_t(r) * 128u, xr = uint32_t(r & 7);
    uint32_t gs = 0;
    bool ok = true;
    for (int t = cid; ok && t < ntiles; t += ncl) {
      for (int ss = 0; ok && ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % SLOTS, ph = (gs / SLOTS) & 1u;
        const uint32_t wslot = gs % W_SLOTS;
        const int nkb = min(SS, shp.KB - ss * SS);
        if (!P::mbar_wait_warp(&sm.full_w[wslot], (gs / W_SLOTS) & 1u, abort_flag, err,
                               ERR_CONVERT)) {
          ok = false;
          break;
        }
        for (int j = 0; j < nkb; ++j) {
          const uint8_t* box = sm.w[wslot][j >> 1];
          const uint32_t cb = uint32_t(j & 1) * 4u;
          uint4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = *reinterpret_cast<const uint4*>(box + row_off + (((cb + uint32_t(i)) ^ xr) << 4));
          uint32_t h[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            P::s8x4_to_f16x4(v[i].x, h[8 * i + 0], h[8 * i + 1]);
            P::s8x4_to_f16x4(v[i].y, h[8 * i + 2], h[8 * i + 3]);
            P::s8x4_to_f16x4(v[i].z, h[8 * i + 4], h[8 * i + 5]);
            P::s8x4_to_f16x4(v[i].w, h[8 * i + 6], h[8 * i + 7]);
          }
          if (j == 0 &&
              !P::mbar_wait_warp(&sm.empty_s[slot], ph ^ 1u, abort_flag, err, ERR_CONVERT)) {
            ok = false;
            break;
          }
          P::tc_fence_after();
          P::tmem_st32(tmem + lane_base + TM_A + slot * (SS * 32) + uint32_t(j) * 32, h);
        }
        if (!ok) break;
        P::mbar_arrive(&sm.empty_w[wslot]);       // this slot's INT8 weights may be refilled
        // forward the readiness of the slot's activation tiles to the MMA thread
        if (!P::mbar_wait_warp(&sm.full_b[slot], ph, abort_flag, err, ERR_CONVERT)) {
          ok = false;
          break;
        }
        P::tmem_wait_st();
        P::tc_fence_before();
        P::mbar_arrive(&sm.full_a[slot]);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;     // token columns [64*half, +64)
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    uint32_t gc = 0;
    bool ok = true;
    for (int t = cid; ok && t < ntiles; t += ncl) {
      int g, mb, nb;
      tile_coords(shp, list, cnt, t, rank, g, mb, nb);
      const int n = nb * BM + 32 * q + lane;
      const bool n_ok = n < shp.N;
      int rs[64];                                 // exact INT32 running sums
#pragma unroll
      for (int j = 0; j < 64; ++j) rs[j] = 0;
      for (int c = 0; c < shp.nchunks; ++c, ++gc) {
        const uint32_t buf = gc & 1u;
        if (!P::mbar_wait_warp(&sm.dfull[buf], (gc >> 1) & 1u, abort_flag, err, ERR_EPILOGUE)) {
          ok = false;
          break;
        }
        P::tc_fence_after();
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t d[32];
          P::tmem_ld32(tmem + lane_base + TM_D + buf * BN + 64 * half + 32 * blk, d);
          P::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) rs[32 * blk + j] += __float2int_rn(__uint_as_float(d[j]));
        }
        P::tc_fence_before();
        P::mbar_arrive(&sm.dempty[buf]);
      }
      if (!ok) break;
      // final: dequantise the exact INT32 sums of this tile
      const uint16_t* bias = lin.bias[g];
      uint16_t* Y = lin.y[g];
      int32_t* ACC = lin.acc[g];
      const float swn = n_ok ? lin.sw[g][n] : 0.f;
      const float bn = (n_ok && bias) ? bias_value(bias[n]) : 0.f;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int m0 = mb * BN + 64 * half + 32 * blk;
        const float sa_l = (m0 + lane < shp.M) ? sa[m0 + lane] : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float saj = __shfl_sync(0xFFFFFFFFu, sa_l, j);
          const int m = m0 + j;
          if (n_ok && m < shp.M) {
            const int64_t off = int64_t(m) * shp.N + n;
            if (ACC) ACC[off] = rs[32 * blk + j];
            if (Y) Y[off] = float_to_bf16_bits(epilogue_value(rs[32 * blk + j], saj, swn, bn));
          }
        }
      }
    }
  }

  P::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    P::tc_fence_after();
    P::tmem_dealloc(tmem, TM_COLS);
  }
  P::cluster_sync();                              // both CTAs leave together
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

void* tensor_map_encoder() {
  static void* fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return p;
  }();
  return fn;
}

int64_t gemm_tc_coded_ld(int64_t K) { return (K + BK - 1) / BK * BK; }

size_t fallback_list_capacity(int64_t M, int64_t N) {
  const size_t mt = size_t((M + BN - 1) / BN);
  const size_t nt = size_t((N + BM - 1) / BM);
  return mt * ((nt + CLUSTER - 1) / CLUSTER);
}

WorkspaceLayout workspace_layout(int64_t M, int64_t N, int64_t K, int G) {
  auto up = [](size_t b) { return (b + 255u) & ~size_t(255); };
  const size_t mt2 = size_t((M + kNormTokens - 1) / kNormTokens);
  const size_t nt = size_t((N + BM - 1) / BM);
  WorkspaceLayout l;
  l.act = 0;
  l.amax = up(size_t(M) * size_t(gemm_tc_coded_ld(K)) * 2u);
  l.status = l.amax + up(mt2 * (1u + kNormSegs) * 4u);
  l.nwpart = l.status + 256u;
  l.list = l.nwpart + up(size_t(G) * nt * kNormParts * (1u + kNormSegs) * 4u);
  l.total = l.list + up(size_t(G) * fallback_list_capacity(M, N) * sizeof(uint2));
  return l;
}

cudaError_t launch_gemm_tc(const uint16_t* act_f16, const float* sa, const LinearGroup& grp,
                           int64_t M, int64_t N, int64_t K, uint32_t* err, const uint2* list,
                           const uint32_t* list_len, size_t list_cap, cudaStream_t s) {
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  // activations: a [M, ld] FP16 matrix viewed as (64-element chunk, row, chunk index),
  // so one box carries two whole k-block tiles, one after the other
  const int64_t ld = gemm_tc_coded_ld(K);
  CUtensorMap map;
  const cuuint64_t dims[3] = {cuuint64_t(BK), cuuint64_t(M), cuuint64_t(ld / BK)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2u, cuuint64_t(BK) * 2u};
  const cuuint32_t box[3] = {BK, BN, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(act_f16), dims,
          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // weights: [N, K] INT8 per Linear, boxes of 128 rows x 128 bytes (two k-blocks)
  Linears lin = {};
  const cuuint64_t wdims[2] = {cuuint64_t(K), cuuint64_t(N)};
  const cuuint64_t wstrides[1] = {cuuint64_t(K)};
  const cuuint32_t wbox[2] = {2 * BK, BM};
  for (int g = 0; g < kMaxGroup; ++g) {
    // unused entries repeat the first Linear's (never read)
    const int src = g < grp.G ? g : 0;
    if (enc(&lin.w[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(grp.wq[src]), wdims,
            wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    lin.sw[g] = grp.ws[src];
    lin.bias[g] = grp.bias[src];
    lin.y[g] = grp.y[src];
    lin.acc[g] = grp.acc[src];
  }

  Shape shp;
  shp.G = list ? grp.G : 1;
  shp.list_cap = int(list_cap);
  shp.M = int(M);
  shp.N = int(N);
  shp.K = int(K);
  shp.KB = int((K + BK - 1) / BK);
  shp.NSS = (shp.KB + SS - 1) / SS;
  shp.nchunks = (shp.NSS + MAX_SS_PER_CHUNK - 1) / MAX_SS_PER_CHUNK;
  shp.sspc = (shp.NSS + shp.nchunks - 1) / shp.nchunks;
  shp.mt = int((M + BN - 1) / BN);
  shp.nt = int((N + BM - 1) / BM);
  shp.ntc = (shp.nt + CLUSTER - 1) / CLUSTER;
  shp.tiles = shp.mt * shp.ntc;

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes));
  if (e != cudaSuccess) return e;
  // with lists, as many clusters as the largest possible list total asks
  const int64_t max_tiles = list ? int64_t(shp.G) * shp.tiles : shp.tiles;
  const int clusters = max_tiles < sms / CLUSTER ? int(max_tiles) : sms / CLUSTER;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(clusters * CLUSTER));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = list ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, map, lin, sa, shp, err, list, list_len);
}

}  // namespace h3q
