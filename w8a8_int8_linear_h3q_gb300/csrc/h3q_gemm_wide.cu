// h3q_gemm_wide.cu -- A3 + A4 on the sm_103a tensor cores for the tiles whose
// FP32 sums are exact over the whole K.
//
//   acc[m,n] = sum_k qa[m,k] * qw[n,k]          exact INT32
//   y[m,n]   = BF16_RNE(acc * sa[m] * sw[n] + bias[n])
//
// Sources: "feat(mps): support MiniMax-H3 INT8 inference on Apple M5"
// (LightX2V #1672) -- Validation (INT8 x INT8 with CPU INT32 references),
// opening description (native K = 5376, no weight dequantisation); "MLX
// implementation and experiment report", What the default preserves (bias
// before the one rounding).
//
// The arithmetic is the chunked kernel's (INT8 values carried exactly by the
// FP16 MMA, FP32 accumulation in TMEM); the exactness argument differs.  For
// a token row a and a channel row w, every partial sum the tensor core can
// form from the products a_k w_k, in any order and grouping, is at most
// sum_k |a_k w_k| <= |a|_2 |w|_2 in magnitude (Cauchy-Schwarz).  When
// |a|_2^2 |w|_2^2 <= 2^48, every partial sum is an integer of magnitude
// <= 2^24 and hence an FP32 value, so no addition rounds and one FP32
// accumulator carries the exact dot product over all of K.  The activation
// quantiser records, per block of 256 tokens, the largest sum of squares of a
// coded row.  A tile (256 channels x 256 tokens) is computed here when that
// maximum times the largest possible weight row (128^2 K) is at most 2^48 --
// which holds for activations whose codes are mostly small, as per-row absmax
// scaling of K = 5376 rows with outliers gives -- or, failing that, when it
// times the tile's largest weight-row sum of squares (from a pre-pass that
// runs only when some tile needs it) is.
//
// A tile that fails this test by a little (long K with Gaussian-like codes,
// where the tile's largest token and channel norms just cross the bound,
// although nearly every actual partial sum stays far below 2^24) can still
// keep one accumulator, with checkpoints.  K is cut into four norm segments;
// the quantiser and the pre-pass also record the largest sums of squares per
// segment.  Over a run of segments r the partial sums of the run move the
// accumulator by at most sqrt(A_r W_r) (Cauchy-Schwarz over the run, A_r and
// W_r the sums of the tile's per-segment maxima), so an accumulator that
// holds exactly S at the run's start stays exact through the run when
// max|S| + sqrt(A_r W_r) <= 2^24.  The scheduler plans the runs (greedily,
// each with sqrt(A_r W_r) <= 2^24 - 2^21); before each later run the MMA
// issuer stops, the epilogue warps read the accumulator (exact so far) and
// report max|S| over the tile, and the issuer checks the inequality with that
// value.  Should a check fail, the tile still runs to its end, but it is put
// on the fallback list, and the chunked kernel, which runs afterwards,
// overwrites its outputs.  The remaining tiles go to that list from the
// start.
//
// Against the chunked kernel this removes the per-chunk accumulator drains
// (one drain per tile) and lets each converted weight slice feed 256 tokens
// instead of 128, halving the converter warps' TMEM stores per MMA, which
// compete with the MMAs for TMEM.
//
// The two CTAs of a cluster work as a pair on one tile of 256 channels x 256
// tokens with the paired MMA (cta_group::2, M = 256): each CTA converts the
// weights of its own 128 channels into its own TMEM and holds the
// accumulator for them, and each CTA's shared memory holds only its half of
// the tile's tokens (128), which the pair MMA reads from both.  Half-size
// activation stages let the activation ring be four super-stages deep, and
// each CTA refills its own stages with no wait on the other.  One elected
// lane of the even CTA's MMA warp issues every MMA, while the whole warp runs
// the loop and waits on barriers that both CTAs' converter and epilogue
// threads arrive on; its commits arrive in both CTAs.
//
// Warp roles (736 threads per CTA):
//   warp 0      TMA producer of this CTA's activation half (4 super-stages)
//   warp 1      TMEM allocator; MMA issuer (the whole warp runs the loop,
//               one elected lane issues; even CTA only)
//   warp 2      tile scheduler (exactness test, fallback list) and TMA
//               producer of this CTA's INT8 weight tiles (4 super-stages)
//   warps 3-6   converters: INT8 weights -> FP16 -> TMEM (2 super-stages)
//   warps 7-22  epilogue: drain the accumulator to registers, release it,
//               then dequant + bias + BF16 (and the optional raw INT32)
// A super-stage is 2 k-blocks of 64 K: 8 pair MMAs of 256 x 256 x 16.
// TMEM (each CTA): the FP32 accumulator in columns 0-255, A super-stages in
// 256-319 and 320-383.  (Four A super-stages fit, but measured slower: the
// converters then run ahead into activation tiles that have not landed.)
// Every wait is bounded in time; on a timeout the kernel records an error
// bit, lets every role fall through, drains its in-flight copies and MMAs,
// frees TMEM and returns.
#include <cuda.h>

#include "h3q_epilogue.cuh"
#include "h3q_internal.cuh"
#include "h3q_tc_ptx.cuh"

namespace h3q {
namespace {

namespace P = ptx;

constexpr int BM = 128;                 // channels per CTA (TMEM lanes); the pair MMA has M = 256
constexpr int BN = kNormTokens;         // tokens per tile (MMA N)
constexpr int BNH = BN / 2;             // tokens held by each CTA of the pair
constexpr int BK = 64;                  // K per k-block (128 bytes of FP16)
constexpr int SS = 2;                   // k-blocks per super-stage (8 MMAs)
constexpr int B_SLOTS = 4;              // super-stage slots: activation halves (SMEM)
constexpr int A_SLOTS = 2;              // super-stage slots: FP16 weights (TMEM)
constexpr int W_SLOTS = 4;              // super-stage slots: INT8 weights (SMEM)
constexpr int SQ = 4;                   // tile-queue entries
constexpr int CLUSTER = 2;
constexpr uint16_t CLUSTER_MASK = (1u << CLUSTER) - 1;
constexpr int MMA_WARP = 1;
constexpr int SCHED_WARP = 2;
constexpr int CONV_WARP0 = 3;
constexpr int NUM_CONV_WARPS = 4;
constexpr int EPI_WARP0 = CONV_WARP0 + NUM_CONV_WARPS;
constexpr int NUM_EPI_WARPS = 16;
constexpr int THREADS = 32 * (EPI_WARP0 + NUM_EPI_WARPS);
// every warp but the scheduler takes each tile from the queue, with one
// arrival per warp: the activation producer, the MMA warp, the converters
// and the epilogue
constexpr int QUEUE_READERS = 2 + NUM_CONV_WARPS + NUM_EPI_WARPS;
constexpr int B_KBLOCK_BYTES = BNH * BK * 2;               // 16 KB
constexpr int W_BOX_BYTES = BM * SS * BK;                  // 16 KB: 128 rows x 2 k-blocks
constexpr uint32_t TM_D = 0;
constexpr uint32_t TM_A = BN;
constexpr uint32_t TM_COLS = 512;
static_assert(TM_A + A_SLOTS * SS * 32 <= TM_COLS, "TMEM columns");
// the converters find an A slot free through the super-stage barriers of the
// activation ring, so the A ring may not be deeper than that ring
static_assert(A_SLOTS <= B_SLOTS, "A ring deeper than the activation ring");
constexpr uint32_t IDESC = P::idesc_f16_f32(2 * BM, BN);
constexpr uint32_t IDESC_BF16 = P::idesc_bf16_f32(2 * BM, BN);
constexpr uint64_t kExactBound = uint64_t(1) << 48;        // |a|^2 |w|^2 limit
constexpr int NSEG = kNormSegs;
static_assert(SS * BK == kSegQuantum, "norm segments are whole super-stages");
constexpr uint32_t kAccExact = 1u << 24;   // FP32 holds every integer up to this
// a planned run's bound leaves this much room for the accumulator's value at
// the run's start
constexpr uint32_t kRunLimit = kAccExact - (1u << 21);
// ways through the kernel of a cluster tile
constexpr int TILE_WIDE = 0, TILE_CKPT = 1, TILE_CHUNKED = 2;

// error bits (the chunked kernel uses the low byte)
constexpr uint32_t ERR_PRODUCER = 1u << 8, ERR_MMA = 2u << 8, ERR_CONVERT = 4u << 8,
                   ERR_EPILOGUE = 8u << 8, ERR_TEARDOWN = 16u << 8, ERR_SCHED = 32u << 8;

struct __align__(1024) Smem {
  uint8_t b[B_SLOTS][SS][B_KBLOCK_BYTES];  // this CTA's activation half, per k-block
  uint8_t w[W_SLOTS][W_BOX_BYTES];       // INT8 weights: 128-byte rows, 128-byte swizzle
  uint64_t full_b[B_SLOTS];              // a slot's activation half has landed
  uint64_t full_w[W_SLOTS];              // a slot's INT8 weights have landed
  uint64_t empty_w[W_SLOTS];             // the converters have read them
  uint64_t full_a[A_SLOTS];              // (even CTA) both CTAs' A and B are in place
  uint64_t empty_ss[B_SLOTS];            // the pair MMAs of super-stage s are done
  uint64_t dfull;                        // the tile's accumulator is complete
  uint64_t dempty;                       // (even CTA) both epilogues have copied it out
  uint64_t mma_done;
  uint64_t q_full[SQ], q_empty[SQ];      // tile queue
  uint64_t cp_slot[CLUSTER * NUM_EPI_WARPS];  // (even CTA) per epilogue warp at a checkpoint:
                                             // event tag << 32 | max |accumulator| of its block
  int q_tile[SQ];                        // cluster tile index, or -1: no more tiles
  uint32_t q_ckpt[SQ];                   // bit s: the accumulator is checked before segment s
  uint32_t q_aw[SQ][2 * NSEG];           // the tile's per-segment norm maxima (tokens, channels)
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + slack for 1024-byte alignment

// The weight maps and output pointers of the Linears of a call (they share
// the activations).
struct WMaps {
  CUtensorMap m[kMaxGroup];
};
struct Outs {
  const float* sw[kMaxGroup];
  const uint16_t* bias[kMaxGroup];
  uint16_t* y[kMaxGroup];
  int32_t* acc[kMaxGroup];
  const float2* ab[kMaxGroup];            // (affine mode) per channel and group: step, offset
};

struct Shape {
  int G;              // Linears
  int M, N, K;
  int KB;             // k-blocks
  int NSS;            // super-stages per tile
  int mt, nt;         // 256-token blocks, 128-channel blocks
  int mt128;          // 128-token blocks (the chunked kernel's tiles)
  int ntc;            // channel-block pairs
  int tiles;          // cluster tiles: G * mt * ntc
  int list_cap;       // entries of one Linear's fallback list
  int seg_ss;         // super-stages per norm segment
  uint64_t wmax2;     // 128^2 K: no weight row's sum of squares exceeds it
  int panel;          // raster panel: token blocks (wpanel 0) or channel-block pairs (1)
  int wpanel;
};

// A TILE_CKPT tile's plan: where the accumulator is checked, and the largest
// per-segment sums of squares of its token rows (aw[0..3]) and channel rows
// (aw[4..7]).
struct TilePlan {
  uint32_t ckpt;
  uint32_t aw[2 * NSEG];
};

// Cluster tile t -> Linear g, token block mb (256 tokens) and channel-block
// pair.  The Linears alternate fastest, so concurrent tiles of different
// Linears read the same activation tiles.  The tiles are walked in panels:
// either `panel` token blocks at a time, with every channel-block pair of
// them before the next panel (the panel's activations stay in L2 while the
// weights stream past), or `panel` channel-block pairs at a time, with every
// token block of them (the panel's weights stay, the activations stream).
// Within a panel its own index runs fastest, so the concurrent tiles of a
// round share the streamed operand's tiles too.
__device__ __forceinline__ void tile_coords(const Shape& s, int t, int& g, int& mb, int& pair) {
  g = t % s.G;
  t /= s.G;
  const int span = s.wpanel ? s.ntc : s.mt;    // the panel's dimension
  const int across = s.wpanel ? s.mt : s.ntc;  // walked once per panel
  const int per_group = s.panel * across;
  const int grp = t / per_group;
  const int first = grp * s.panel;
  const int gp = min(s.panel, span - first);
  const int r = t - grp * per_group;
  const int a = first + r % gp, b = r / gp;
  mb = s.wpanel ? b : a;
  pair = s.wpanel ? a : b;
}

// Warp-collective: tile_path past its first test.  Lanes 0-15 read the pair's 16
// weight partial maxima; failing the whole-K test, the per-segment maxima
// (lanes 0-15 segments 0-1, lanes 16-31 segments 2-3 of the same partial
// maxima) give the checkpoint plan: runs of segments grow while
// sqrt(A_r W_r) <= kRunLimit, and a segment that alone exceeds it sends the
// tile to the chunked kernel.  Every lane returns the same plan.
__device__ __forceinline__ int tile_path_norms(const Shape& s, uint64_t a, const uint32_t* aseg,
                                            const uint32_t* nwpart, const uint32_t* nwseg, int mb,
                                            int pair, int lane, TilePlan& plan) {
  const int p = pair * CLUSTER * kNormParts + (lane & (CLUSTER * kNormParts - 1));
  const bool p_ok = p < s.nt * kNormParts;
  uint32_t w = (lane < CLUSTER * kNormParts && p_ok) ? nwpart[p] : 0u;
#pragma unroll
  for (int o = 16; o; o >>= 1) w = max(w, __shfl_xor_sync(0xFFFFFFFFu, w, o));
  if (uint64_t(w) * a <= kExactBound) return TILE_WIDE;
  static_assert(CLUSTER * kNormParts == 16 && NSEG == 4, "two segments per half-warp");
  const int sg = 2 * (lane >> 4);
  uint32_t w0 = p_ok ? nwseg[p * NSEG + sg] : 0u, w1 = p_ok ? nwseg[p * NSEG + sg + 1] : 0u;
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    w0 = max(w0, __shfl_xor_sync(0xFFFFFFFFu, w0, o));
    w1 = max(w1, __shfl_xor_sync(0xFFFFFFFFu, w1, o));
  }
  plan.aw[NSEG + 0] = __shfl_sync(0xFFFFFFFFu, w0, 0);
  plan.aw[NSEG + 1] = __shfl_sync(0xFFFFFFFFu, w1, 0);
  plan.aw[NSEG + 2] = __shfl_sync(0xFFFFFFFFu, w0, 16);
  plan.aw[NSEG + 3] = __shfl_sync(0xFFFFFFFFu, w1, 16);
#pragma unroll
  for (int i = 0; i < NSEG; ++i) plan.aw[i] = aseg[mb * NSEG + i];
  // every sum below is at most 127^2 K < 2^32 and every product < 2^64
  const uint64_t lim2 = uint64_t(kRunLimit) * kRunLimit;
  uint64_t ra = 0, rw = 0;
  uint32_t ck = 0;
#pragma unroll
  for (int i = 0; i < NSEG; ++i) {
    if (i * s.seg_ss >= s.NSS) break;               // empty trailing segments
    const uint64_t na = ra + plan.aw[i], nw = rw + plan.aw[NSEG + i];
    if (na * nw <= lim2) {
      ra = na;
      rw = nw;
      continue;
    }
    if (i == 0 || uint64_t(plan.aw[i]) * plan.aw[NSEG + i] > lim2) return TILE_CHUNKED;
    ck |= 1u << i;
    ra = plan.aw[i];
    rw = plan.aw[NSEG + i];
  }
  plan.ckpt = ck;
  // no checkpoint: the segment maxima bound the whole K within 2^24 after all
  return ck ? TILE_CKPT : TILE_WIDE;
}

// Warp-collective: how a cluster tile is computed.  TILE_WIDE when every
// (token, channel) of the tile has |a|^2 |w|^2 <= 2^48: the token block's
// maximum against the largest possible weight row settles most tiles;
// otherwise tile_path_norms decides, from the weight norms.
__device__ __forceinline__ int tile_path(const Shape& s, const uint32_t* amax,
                                         const uint32_t* aseg, const uint32_t* nwpart,
                                         const uint32_t* nwseg, int mb, int pair, int lane,
                                         TilePlan& plan) {
  const uint64_t a = amax[mb];
  if (a * s.wmax2 <= kExactBound) return TILE_WIDE;
  return tile_path_norms(s, a, aseg, nwpart, nwseg, mb, pair, lane, plan);
}

// Warp-collective take (with the entry's checkpoint bits, or its whole
// checkpoint plan); one arrival for the warp.
__device__ __forceinline__ bool pop_tile_warp(Smem& sm, uint32_t& nq, volatile int* abort_flag,
                                              uint32_t* err, uint32_t code, int& t, int lane,
                                              uint32_t* ckpt = nullptr, TilePlan* plan = nullptr) {
  const uint32_t q = nq % SQ;
  if (!P::mbar_wait_warp(&sm.q_full[q], (nq / SQ) & 1u, abort_flag, err, code)) return false;
  t = sm.q_tile[q];
  if (ckpt) *ckpt = sm.q_ckpt[q];
  if (plan) {
    plan->ckpt = sm.q_ckpt[q];
    if (plan->ckpt)
      for (int i = 0; i < 2 * NSEG; ++i) plan->aw[i] = sm.q_aw[q][i];
  }
  __syncwarp();
  if (lane == 0) P::mbar_arrive(&sm.q_empty[q]);
  ++nq;
  return true;
}

__device__ __forceinline__ bool push_tile(Smem& sm, uint32_t& nq, int t, const TilePlan* plan,
                                          volatile int* abort_flag, uint32_t* err) {
  const uint32_t q = nq % SQ;
  if (!P::mbar_wait(&sm.q_empty[q], ((nq / SQ) & 1u) ^ 1u, abort_flag, err, ERR_SCHED))
    return false;
  sm.q_tile[q] = t;
  sm.q_ckpt[q] = plan ? plan->ckpt : 0u;
  if (plan) {
#pragma unroll
    for (int i = 0; i < 2 * NSEG; ++i) sm.q_aw[q][i] = plan->aw[i];
  }
  P::mbar_arrive(&sm.q_full[q]);
  ++nq;
  return true;
}

// Lists a 256 x 256 cluster tile for the chunked kernel, as one or two
// 128-token tiles.
__device__ __forceinline__ void list_for_chunked(const Shape& shp, uint32_t* status, uint2* list,
                                                 int g, int mb, int pair) {
  const int n128 = min(2, shp.mt128 - 2 * mb);
  const uint32_t i = atomicAdd(status + 2 + g, uint32_t(n128));
  atomicAdd(status + 1, uint32_t(n128));
  for (int h = 0; h < n128; ++h)
    list[g * shp.list_cap + i + h] = make_uint2(uint32_t(2 * mb + h), uint32_t(pair));
}

// A4 for 32 consecutive tokens of this lane's channel row n: lane l holds the
// scale of token mbase + l in sa_l (sa_all is the whole scale vector), and d[j]
// the accumulator of token mbase + j, an exact integer |t| <= 2^24 as an FP32
// value.
//
// The epilogue's instructions compete for issue slots with the converter
// warps, which are on the critical path right after a tile's accumulator is
// released, so the common case is kept short (and runs two tokens per
// instruction where it can).  Per element: c = RN(s_a s_w) and
// v = RN(t c + bias), one FMA; the error argument is epilogue_value's
// (h3q_epilogue.cuh): whenever |v| >= 2^-10 |bias| (a threshold formed once
// per channel), one BF16 rounding of v is within one ulp of the exact value,
// and t = 0 gives v = bias exactly.  An element that fails the check (deep
// cancellation with the bias) takes the error-free path.  Blocks with scales
// outside the checked ranges, ragged token tails and the raw INT32 output
// take the general per-element path.
__device__ __forceinline__ int lane_id() { return int(threadIdx.x & 31u); }

__device__ __forceinline__ void emit_block(const uint32_t (&d)[32], float sa_l, int mbase,
                                           float swn, float bn, int n, bool n_ok,
                                           const Shape& shp, uint16_t* __restrict__ Y,
                                           int32_t* __restrict__ ACC, const float* __restrict__ sa_all) {
  // every token's scales in the cheap path's range: the paired form of
  // epilogue_value, bit for bit
  const bool s_in = epilogue_scales_in_range(sa_l, swn);
  if (__all_sync(0xFFFFFFFFu, s_in) && !ACC && Y && mbase + 32 <= shp.M) {
    // adjacent lanes pair up: after one exchange, the even lane stores channels n, n + 1 of
    // token j and the odd lane those of token j + 1, as one 4-byte store each (even N only,
    // which keeps every pair 4-byte aligned)
    const bool pairs = (shp.N & 1) == 0;
    const int odd = lane_id() & 1;
    const uint32_t sel = odd ? 0x3276u : 0x5410u;
    uint16_t* yp = pairs ? Y + int64_t(mbase + odd) * shp.N + (n - odd)
                         : Y + int64_t(mbase) * shp.N + n;
    const bool pair_ok = (n - odd) < shp.N;
    const float* sa_ptr = sa_all + mbase;
    // two tokens at a time with the paired FP32 instructions (the same IEEE
    // operations as the scalar ones, half the instructions)
    const uint64_t sw2 = (uint64_t(__float_as_uint(swn)) << 32) | __float_as_uint(swn);
    const uint64_t b2 = (uint64_t(__float_as_uint(bn)) << 32) | __float_as_uint(bn);
    const float bthr = fabsf(bn) * 0x1p-10f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      // both tokens' scales in one broadcast load (every lane reads the same 8 bytes)
      const float2 sab = __ldg(reinterpret_cast<const float2*>(sa_ptr + j));
      const float sa_a = sab.x, sa_b = sab.y;
      const uint64_t sa2 = (uint64_t(__float_as_uint(sa_b)) << 32) | __float_as_uint(sa_a);
      const uint64_t t2 = (uint64_t(d[j + 1]) << 32) | d[j];
      uint64_t c2, v2;
      asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c2) : "l"(sa2), "l"(sw2));
      asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(v2) : "l"(t2), "l"(c2), "l"(b2));
      float va = __uint_as_float(uint32_t(v2)), vb = __uint_as_float(uint32_t(v2 >> 32));
      if (!(fabsf(va) >= bthr))
        va = epilogue_value_careful(__float2int_rn(__uint_as_float(d[j])), sa_a, swn, bn);
      if (!(fabsf(vb) >= bthr))
        vb = epilogue_value_careful(__float2int_rn(__uint_as_float(d[j + 1])), sa_b, swn, bn);
      uint32_t h2;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h2) : "f"(vb), "f"(va));
      if (pairs) {
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, h2, 1);
        uint32_t out;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(out) : "r"(h2), "r"(other), "r"(sel));
        if (pair_ok) *reinterpret_cast<uint32_t*>(yp + int64_t(j) * shp.N) = out;
      } else if (n_ok) {
        yp[int64_t(j) * shp.N] = uint16_t(h2);
        yp[int64_t(j + 1) * shp.N] = uint16_t(h2 >> 16);
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float saj = __shfl_sync(0xFFFFFFFFu, sa_l, j);
    const int m = mbase + j;
    const int a = __float2int_rn(__uint_as_float(d[j]));
    if (n_ok && m < shp.M) {
      const int64_t off = int64_t(m) * shp.N + n;
      if (ACC) ACC[off] = a;
      if (Y) Y[off] = float_to_bf16_bits(epilogue_value(a, saj, swn, bn));
    }
  }
}

// The MMA issuer's checkpoint before norm segment `seg` (out of line and
// outside the issue loop, whose speed it would otherwise cost; called by the
// elected lane that issued the MMAs, since its commit must follow them).  The MMAs
// issued so far complete into the accumulator, the
// epilogues read it (exact so far) and each reports the largest magnitude of
// its block, tagged with this event's number (gt + 1); then the run that
// starts here (segments up to the next checkpoint) is checked against 2^24.
// Returns 0 if it holds, 1 if not (or a report is missing), -1 if a wait
// gave up.
__device__ __noinline__ int mma_checkpoint(Smem& sm, const TilePlan& pl, int seg, uint32_t gt,
                                           volatile int* abort_flag, uint32_t* err) {
  P::mma_commit_pair_mc(&sm.dfull, CLUSTER_MASK);
  if (!P::mbar_wait_cluster(&sm.dempty, ((gt + 1) & 1u) ^ 1u, abort_flag, err, ERR_MMA))
    return -1;
  P::tc_fence_after();
  uint32_t obs = 0;
  for (int i = 0; i < CLUSTER * NUM_EPI_WARPS; ++i) {
    const uint64_t word = *reinterpret_cast<volatile uint64_t*>(&sm.cp_slot[i]);
    if (uint32_t(word >> 32) != gt + 1) return 1;
    obs = max(obs, uint32_t(word));
  }
  uint64_t ra = 0, rw = 0;
  bool in_run = true;
#pragma unroll
  for (int i = 0; i < NSEG; ++i) {
    if (i > seg && ((pl.ckpt >> i) & 1u)) in_run = false;
    if (i >= seg && in_run) {
      ra += pl.aw[i];
      rw += pl.aw[NSEG + i];
    }
  }
  return (obs > kAccExact || uint64_t(kAccExact - obs) * (kAccExact - obs) < ra * rw) ? 1 : 0;
}

constexpr uint32_t kNoEvent = 0xFFFFFFFFu;

// An epilogue warp's part of a tile's checkpoints (warp-collective): at each,
// the largest |accumulator| of the warp's 32 x 64 block (TMEM address d_tmem)
// goes into the warp's own slot in the even CTA, tagged with the event's
// number, and lane 0 arrives with a cluster-scope release (the MMA issuer
// waits with a cluster-scope acquire).  (A single word updated by 64-bit
// atomic maxima from both CTAs was seen to lose updates, hence one slot per
// warp.)  Returns the event count after them, or kNoEvent when a wait gave
// up.
__device__ __forceinline__ uint32_t epilogue_checkpoints(Smem& sm, uint32_t ckpt, uint32_t gt,
                                                         volatile int* abort_flag, uint32_t* err,
                                                         uint32_t d_tmem, uint32_t slot_pair,
                                                         uint32_t dempty_pair, int lane) {
  for (; ckpt; ckpt &= ckpt - 1u) {
    if (!P::mbar_wait_warp(&sm.dfull, gt & 1u, abort_flag, err, ERR_EPILOGUE)) return kNoEvent;
    P::tc_fence_after();
    uint32_t d0[32], d1[32];
    P::tmem_ld32(d_tmem, d0);
    P::tmem_ld32(d_tmem + 32, d1);
    P::tmem_wait_ld();
    P::tc_fence_before();
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(d0[j])), fabsf(__uint_as_float(d1[j]))));
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0) {
      // float -> unsigned conversion saturates
      P::st_cluster_u64(slot_pair, (uint64_t(gt + 1) << 32) | __float2uint_ru(mx));
      P::fence_acq_rel_cluster();
      P::mbar_arrive_cluster_release(dempty_pair);
    } else {
      P::mbar_arrive_cluster(dempty_pair);
    }
    ++gt;
  }
  return gt;
}

// Affine mode (the group-wise weight-only comparison scheme): A2 absent, B is
// the BF16 activations themselves, the weights are 8-bit codes dequantised
// by the converters (one group of 64 per k-block), the accumulation is the
// plain FP32 one of a BF16 GEMM (no exactness test, every tile wide), and the
// epilogue is y = BF16(acc + bias).  Only the A2-free path shares the
// pipeline; what W8A8 computes is unchanged (the mode is a template
// parameter, so its branches compile out).
//
// A4 for 32 consecutive tokens of this lane's channel row n in affine mode.
__device__ __forceinline__ void emit_block_affine(const uint32_t (&d)[32], int mbase, float bn,
                                                  int n, bool n_ok, const Shape& shp,
                                                  uint16_t* __restrict__ Y) {
  if (!n_ok) return;
  uint16_t* yp = Y + int64_t(mbase) * shp.N + n;
  const uint64_t b2 = (uint64_t(__float_as_uint(bn)) << 32) | __float_as_uint(bn);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t t2 = (uint64_t(d[j + 1]) << 32) | d[j];
    uint64_t v2;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(v2) : "l"(t2), "l"(b2));
    uint32_t h2;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(h2)
        : "f"(__uint_as_float(uint32_t(v2 >> 32))), "f"(__uint_as_float(uint32_t(v2))));
    if (mbase + j < shp.M) yp[int64_t(j) * shp.N] = uint16_t(h2);
    if (mbase + j + 1 < shp.M) yp[int64_t(j + 1) * shp.N] = uint16_t(h2 >> 16);
  }
}

// 23 warps: at most 6 per SM sub-partition, so 80 registers a thread.
template <bool kAffine>
__global__ void __launch_bounds__(THREADS, 1)
gemm_wide_kernel(const __grid_constant__ CUtensorMap act_map, const __grid_constant__ WMaps wmaps,
                 const float* __restrict__ sa, const __grid_constant__ Outs outs, const Shape shp,
                 const uint32_t* __restrict__ amax, const uint32_t* __restrict__ nwpart,
                 uint32_t* __restrict__ status, uint2* __restrict__ list) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm.abort_flag;
  uint32_t* err = status;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_SLOTS; ++i) {
      P::mbar_init(&sm.full_w[i], 1);
      P::mbar_init(&sm.empty_w[i], NUM_CONV_WARPS * 32);
    }
    for (int i = 0; i < B_SLOTS; ++i) {
      P::mbar_init(&sm.full_b[i], 1);
      P::mbar_init(&sm.empty_ss[i], 1);           // the pair's commit
    }
    for (int i = 0; i < A_SLOTS; ++i)
      P::mbar_init(&sm.full_a[i], CLUSTER * NUM_CONV_WARPS * 32);
    for (int i = 0; i < SQ; ++i) {
      P::mbar_init(&sm.q_full[i], 1);
      P::mbar_init(&sm.q_empty[i], QUEUE_READERS);
    }
    P::mbar_init(&sm.dfull, 1);
    P::mbar_init(&sm.dempty, CLUSTER * NUM_EPI_WARPS * 32);
    P::mbar_init(&sm.mma_done, 1);
    for (int i = 0; i < CLUSTER * NUM_EPI_WARPS; ++i) sm.cp_slot[i] = 0;
    sm.abort_flag = 0;
    P::fence_mbar_init();
  }
  if (warp == MMA_WARP) P::tmem_alloc_pair(&sm.tmem_base, TM_COLS);   // one warp per CTA
  P::tc_fence_before();
  __syncthreads();
  P::cluster_sync();                              // the peer's barriers exist before any arrive
  P::tc_fence_after();
  // The set-up above overlaps the tail of the previous kernel on the stream
  // (programmatic dependent launch); nothing it wrote is read before here.
  P::grid_dependency_wait();
  P::allow_dependent_launch();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t rank = P::cluster_rank();
  const int cid = int(P::cluster_id_x()), ncl = int(P::num_clusters_x());
  // the even CTA's barriers that both CTAs arrive on
  const uint32_t full_a_pair = P::mapa_shared(P::smem_u32(&sm.full_a[0]), 0);
  const uint32_t dempty_pair = P::mapa_shared(P::smem_u32(&sm.dempty), 0);
  // the norm maxima per segment follow the whole-row ones
  const uint32_t* aseg = amax + shp.mt;
  const uint32_t* nwseg = nwpart + shp.G * shp.nt * kNormParts;

  if (warp == 0) {
    // ---------------- TMA producer: activation tiles ----------------
    // warp-uniform, like the MMA issuer: one elected lane issues the copies
    const uint32_t leader = P::elect_one();
    if (leader) P::tma_prefetch_desc(&act_map);
    uint32_t gs = 0, gb = 0, nq = 0;
    bool ok = true;
    for (;;) {
      int t;
      if (!pop_tile_warp(sm, nq, abort_flag, err, ERR_PRODUCER, t, lane) || t < 0) break;
      int g, mb, pair;
      tile_coords(shp, t, g, mb, pair);
      const int row0 = mb * BN + int(rank) * BNH;
      for (int ss = 0; ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % B_SLOTS;
        // the slot is free once the pair MMAs of its previous super-stage are done
        if (!P::mbar_wait_warp(&sm.empty_ss[slot], ((gs / B_SLOTS) & 1u) ^ 1u, abort_flag, err,
                               ERR_PRODUCER)) {
          ok = false;
          break;
        }
        // this CTA's 128 tokens of the super-stage's two k-blocks
        if (leader) {
          P::mbar_arrive_expect_tx(&sm.full_b[slot], SS * B_KBLOCK_BYTES);
          P::tma_load_3d(P::smem_u32(sm.b[slot][0]), &act_map, &sm.full_b[slot], 0, row0,
                         ss * SS);
        }
        __syncwarp();
        gb = gs + 1;
      }
      if (!ok) break;
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (leader) {
      int no_abort = 0;
      volatile int* never = &no_abort;   // this drain does not follow the abort flag
      for (uint32_t i = gb > B_SLOTS ? gb - B_SLOTS : 0; i < gb; ++i)
        P::mbar_wait(&sm.full_b[i % B_SLOTS], (i / B_SLOTS) & 1u, never, err, ERR_TEARDOWN);
    }
    __syncwarp();
  } else if (warp == SCHED_WARP) {
    // ---------------- scheduler + TMA producer: INT8 weight tiles ----------------
    if (lane < shp.G) P::tma_prefetch_desc(&wmaps.m[lane]);
    const uint32_t wleader = P::elect_one();
    uint32_t gs = 0, gw = 0, nq = 0;
    bool ok = true;
    for (int t = cid; t < shp.tiles; t += ncl) {
      int g, mb, pair;
      tile_coords(shp, t, g, mb, pair);
      TilePlan plan;
      const int path = kAffine ? TILE_WIDE
                               : tile_path(shp, amax, aseg, nwpart + g * shp.nt * kNormParts,
                                           nwseg + g * shp.nt * kNormParts * NSEG, mb, pair,
                                           lane, plan);
      if (path == TILE_CHUNKED) {
        // the chunked kernel takes it (both CTAs reach the same verdict; the
        // even one lists it)
        if (rank == 0 && lane == 0) list_for_chunked(shp, status, list, g, mb, pair);
        continue;
      }
      if (lane == 0) {
        ok = push_tile(sm, nq, t, path == TILE_CKPT ? &plan : nullptr, abort_flag, err);
        if (ok && path == TILE_CKPT && rank == 0) atomicAdd(status + 6, 1u);
      }
      ok = __shfl_sync(0xFFFFFFFFu, int(ok), 0) != 0;
      // the weight copies: warp-uniform waits, one elected lane issues
      const int wrow = min(2 * pair + int(rank), shp.nt - 1) * BM;
      for (int ss = 0; ok && ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % W_SLOTS;
        if (!P::mbar_wait_warp(&sm.empty_w[slot], ((gs / W_SLOTS) & 1u) ^ 1u, abort_flag, err,
                               ERR_SCHED)) {
          ok = false;
          break;
        }
        if (wleader) {
          P::mbar_arrive_expect_tx(&sm.full_w[slot], W_BOX_BYTES);
          P::tma_load_2d(P::smem_u32(sm.w[slot]), &wmaps.m[g], &sm.full_w[slot], ss * SS * BK,
                         wrow);
        }
        __syncwarp();
        gw = gs + 1;
      }
      if (!ok) break;
    }
    if (lane == 0) {
      if (ok) push_tile(sm, nq, -1, nullptr, abort_flag, err);
      int no_abort = 0;
      volatile int* never = &no_abort;
      for (uint32_t i = gw > W_SLOTS ? gw - W_SLOTS : 0; i < gw; ++i)
        P::mbar_wait(&sm.full_w[i % W_SLOTS], (i / W_SLOTS) & 1u, never, err, ERR_TEARDOWN);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ---------------- MMA issuer (even CTA): one wait and one commit per 8 MMAs ----------------
    // The whole warp runs the loop, so that its waits, addresses and
    // descriptors are warp-uniform, and one elected lane issues every MMA and
    // commit.  (A loop run by one lane alone loses issue slots to the other
    // warps of its SM sub-partition -- here a converter and four epilogue
    // warps -- and the tensor pipe then waits for its MMAs.)
    if (rank == 0) {
      uint32_t leader_lane;
      const uint32_t leader = P::elect_one(&leader_lane);
      uint32_t gs = 0, gt = 0, nq = 0;
      bool ok = true;
      for (;;) {
        int t;
        TilePlan pl;
        if (!pop_tile_warp(sm, nq, abort_flag, err, ERR_MMA, t, lane, nullptr, &pl) || t < 0)
          break;
        // both epilogues have copied out the previous tile's accumulator
        if (!P::mbar_wait_warp(&sm.dempty, (gt & 1u) ^ 1u, abort_flag, err, ERR_MMA)) break;
        bool check_failed = false;
        uint32_t pending = pl.ckpt;                 // checkpoints still ahead
        // the super-stages run by run, a checkpoint between runs (the inner
        // loop is kept free of the checkpoint code)
        for (int ss = 0;;) {
          const int ss_end = pending ? (__ffs(pending) - 1) * shp.seg_ss : shp.NSS;
          for (; ss < ss_end; ++ss, ++gs) {
            const uint32_t slot = gs % B_SLOTS, aslot = gs % A_SLOTS;
            if (!P::mbar_wait_warp(&sm.full_a[aslot], (gs / A_SLOTS) & 1u, abort_flag, err,
                                   ERR_MMA)) {
              ok = false;
              break;
            }
            P::tc_fence_after();
            const uint32_t a_tmem = tmem + TM_A + aslot * (SS * 32);
            const int nkb = min(SS, shp.KB - ss * SS);
            const uint64_t bdesc0 = P::smem_desc_sw128(P::smem_u32(sm.b[slot][0]));
            const uint64_t bdesc1 = P::smem_desc_sw128(P::smem_u32(sm.b[slot][1]));
            if (leader) {
#pragma unroll
              for (int j = 0; j < SS; ++j) {
                if (j >= nkb) break;
                const uint64_t bdesc = j ? bdesc1 : bdesc0;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                  P::mma_f16_ts_pair(tmem + TM_D, a_tmem + j * 32 + kk * 8,
                                     bdesc + uint64_t(kk * 2), kAffine ? IDESC_BF16 : IDESC,
                                     (ss > 0 || j > 0 || kk > 0) ? 1u : 0u);
              }
              P::mma_commit_pair_mc(&sm.empty_ss[slot], CLUSTER_MASK);
            }
            __syncwarp();
          }
          if (!ok || !pending) break;
          const int seg = __ffs(pending) - 1;
          pending &= pending - 1u;
          int r = 0;
          if (leader) r = mma_checkpoint(sm, pl, seg, gt, abort_flag, err);
          r = __shfl_sync(0xFFFFFFFFu, r, int(leader_lane));
          ++gt;
          if (r < 0) {
            ok = false;
            break;
          }
          check_failed = check_failed || r > 0;
        }
        if (!ok) break;
        if (leader) P::mma_commit_pair_mc(&sm.dfull, CLUSTER_MASK);
        ++gt;
        if (check_failed && leader) {
          // its outputs are rewritten by the chunked kernel, which runs after
          // this grid has completed
          int g, mb, pair;
          tile_coords(shp, t, g, mb, pair);
          list_for_chunked(shp, status, list, g, mb, pair);
          atomicAdd(status + 7, 1u);
        }
        __syncwarp();
      }
      // every MMA the leader issued has finished before TMEM is freed
      if (leader) {
        P::mma_commit_pair_mc(&sm.mma_done, 1);
        int no_abort = 0;
        volatile int* never = &no_abort;
        P::mbar_wait(&sm.mma_done, 0, never, err, ERR_TEARDOWN);
      }
    } else {
      // the odd CTA issues nothing; its MMA warp takes the tiles from the
      // queue like every other role so that the queue slots are released
      uint32_t nq = 0;
      for (;;) {
        int t;
        if (!pop_tile_warp(sm, nq, abort_flag, err, ERR_MMA, t, lane) || t < 0) break;
      }
    }
    __syncwarp();
  } else if (warp < EPI_WARP0) {
    // ---------------- converters: INT8 weights -> FP16 -> TMEM ----------------
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int r = 32 * q + lane;                  // channel row within the tile
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    // this row's 16-byte chunks in a 128-byte-swizzled INT8 box (two k-blocks),
    // precomputed: the converters' instructions are on the critical path
    const uint32_t row_off = uint32_t(r) * 128u, xr = uint32_t(r & 7);
    uint32_t coff[4 * SS];
#pragma unroll
    for (int k = 0; k < 4 * SS; ++k) coff[k] = row_off + ((uint32_t(k) ^ xr) << 4);
    uint32_t gs = 0, nq = 0;
    bool ok = true;
    while (ok) {
      int t;
      if (!pop_tile_warp(sm, nq, abort_flag, err, ERR_CONVERT, t, lane) || t < 0) break;
      // (affine mode) this lane's channel row and its groups' steps and offsets
      const float2* ab_row = nullptr;
      if constexpr (kAffine) {
        int g, mb, pair;
        tile_coords(shp, t, g, mb, pair);
        const int n = (2 * pair + int(rank)) * BM + r;
        ab_row = n < shp.N ? outs.ab[g] + int64_t(n) * shp.KB : nullptr;
      }
      for (int ss = 0; ss < shp.NSS; ++ss, ++gs) {
        const uint32_t slot = gs % B_SLOTS, aslot = gs % A_SLOTS;
        const uint32_t wslot = gs % W_SLOTS;
        const int nkb = min(SS, shp.KB - ss * SS);
        float2 abk[SS];
        if constexpr (kAffine) {
          // loaded before the wait below, which hides their latency
#pragma unroll
          for (int j = 0; j < SS; ++j)
            abk[j] = (ab_row && j < nkb) ? __ldg(ab_row + ss * SS + j) : make_float2(0.f, 0.f);
        }
        if (!P::mbar_wait_warp(&sm.full_w[wslot], (gs / W_SLOTS) & 1u, abort_flag, err,
                               ERR_CONVERT)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < SS; ++j) {
          if (j >= nkb) break;
          const uint8_t* box = sm.w[wslot];
          uint4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = *reinterpret_cast<const uint4*>(box + coff[4 * j + i]);
          uint32_t h[32];
          if constexpr (kAffine) {
            const uint64_t a2 = (uint64_t(__float_as_uint(abk[j].x)) << 32) |
                                __float_as_uint(abk[j].x);
            const uint64_t b2 = (uint64_t(__float_as_uint(abk[j].y)) << 32) |
                                __float_as_uint(abk[j].y);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              P::u8x4_affine_to_bf16x4(v[i].x, a2, b2, h[8 * i + 0], h[8 * i + 1]);
              P::u8x4_affine_to_bf16x4(v[i].y, a2, b2, h[8 * i + 2], h[8 * i + 3]);
              P::u8x4_affine_to_bf16x4(v[i].z, a2, b2, h[8 * i + 4], h[8 * i + 5]);
              P::u8x4_affine_to_bf16x4(v[i].w, a2, b2, h[8 * i + 6], h[8 * i + 7]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              P::s8x4_to_f16x4(v[i].x, h[8 * i + 0], h[8 * i + 1]);
              P::s8x4_to_f16x4(v[i].y, h[8 * i + 2], h[8 * i + 3]);
              P::s8x4_to_f16x4(v[i].z, h[8 * i + 4], h[8 * i + 5]);
              P::s8x4_to_f16x4(v[i].w, h[8 * i + 6], h[8 * i + 7]);
            }
          }
          // the A slot is free once the pair MMAs of super-stage gs - A_SLOTS are done
          if (j == 0 && gs >= A_SLOTS) {
            const uint32_t prev = gs - A_SLOTS;
            if (!P::mbar_wait_warp(&sm.empty_ss[prev % B_SLOTS], (prev / B_SLOTS) & 1u,
                                   abort_flag, err, ERR_CONVERT)) {
              ok = false;
              break;
            }
            P::tc_fence_after();
          }
          P::tmem_st32(tmem + lane_base + TM_A + aslot * (SS * 32) + uint32_t(j) * 32, h);
        }
        if (!ok) break;
        P::mbar_arrive(&sm.empty_w[wslot]);       // this slot's INT8 weights may be refilled
        // forward the readiness of this CTA's activation half to the MMA thread
        if (!P::mbar_wait_warp(&sm.full_b[slot], (gs / B_SLOTS) & 1u, abort_flag, err,
                               ERR_CONVERT)) {
          ok = false;
          break;
        }
        P::tmem_wait_st();
        P::tc_fence_before();
        P::mbar_arrive_cluster(full_a_pair + aslot * 8u);
      }
    }
    P::tmem_wait_st();
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                       // TMEM lane quarter
    const int cq = (warp - EPI_WARP0) >> 2;       // token columns [64*cq, +64)
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const uint32_t cp_slot_pair = P::mapa_shared(
        P::smem_u32(&sm.cp_slot[int(rank) * NUM_EPI_WARPS + (warp - EPI_WARP0)]), 0);
    uint32_t gt = 0, nq = 0;
    for (;;) {
      int t;
      uint32_t ckpt;
      if (!pop_tile_warp(sm, nq, abort_flag, err, ERR_EPILOGUE, t, lane, &ckpt) || t < 0) break;
      if (ckpt) {
        gt = epilogue_checkpoints(sm, ckpt, gt, abort_flag, err, tmem + lane_base + TM_D + 64 * cq,
                                  cp_slot_pair, dempty_pair, lane);
        if (gt == kNoEvent) break;
      }
      int g, mb, pair;
      tile_coords(shp, t, g, mb, pair);
      const int n = (2 * pair + int(rank)) * BM + 32 * q + lane;
      const bool n_ok = n < shp.N;
      // (affine mode: no scales)
      const float swn = (!kAffine && n_ok) ? outs.sw[g][n] : 0.f;
      const uint16_t* bias = outs.bias[g];
      const float bn = (n_ok && bias) ? bias_value(bias[n]) : 0.f;
      const int m0 = mb * BN + 64 * cq;
      const float sa0 = (!kAffine && m0 + lane < shp.M) ? sa[m0 + lane] : 0.f;
      const float sa1 = (!kAffine && m0 + 32 + lane < shp.M) ? sa[m0 + 32 + lane] : 0.f;
      if (!P::mbar_wait_warp(&sm.dfull, gt & 1u, abort_flag, err, ERR_EPILOGUE)) break;
      P::tc_fence_after();
      uint32_t d0[32], d1[32];
      P::tmem_ld32(tmem + lane_base + TM_D + 64 * cq, d0);
      P::tmem_ld32(tmem + lane_base + TM_D + 64 * cq + 32, d1);
      P::tmem_wait_ld();
      P::tc_fence_before();
      P::mbar_arrive_cluster(dempty_pair);        // the MMAs of the next tile may start
      ++gt;
      if constexpr (kAffine) {
        emit_block_affine(d0, m0, bn, n, n_ok, shp, outs.y[g]);
        emit_block_affine(d1, m0 + 32, bn, n, n_ok, shp, outs.y[g]);
      } else {
        emit_block(d0, sa0, m0, swn, bn, n, n_ok, shp, outs.y[g], outs.acc[g], sa);
        emit_block(d1, sa1, m0 + 32, swn, bn, n, n_ok, shp, outs.y[g], outs.acc[g], sa);
      }
    }
  }

  P::tc_fence_before();
  __syncthreads();
  P::cluster_sync();                              // both CTAs are done with TMEM
  if (warp == MMA_WARP) {
    P::tc_fence_after();
    P::tmem_dealloc_pair(tmem, TM_COLS);
  }
  P::cluster_sync();                              // no peer still signals or writes here
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The raster's panel.  By default, panels of 8 token blocks with every
// channel-block pair of them (measured best for the grouped attention call,
// fc1 and fc2: larger token panels, channel-pair panels and evict-first L2
// hints on the streamed operand all read more from DRAM, because the
// persistent clusters drift apart in time and a shared tile leaves L2 before
// its last reader comes).  When the weights of all G Linears (one byte per
// element in both modes) fit in kAllWeightsBytes, one panel holds every
// channel-block pair: the weights stay in L2 and each token block is read
// once (a single attention Linear: 212 -> 139 MB read per launch).
constexpr int kTokenPanel = 8;
constexpr double kAllWeightsBytes = 48.0 * (1 << 20);

void choose_raster(Shape& s) {
  const double weights = double(s.G) * double(s.N) * double(s.K);
  s.wpanel = weights <= kAllWeightsBytes ? 1 : 0;
  s.panel = s.wpanel ? s.ntc : kTokenPanel;
}

// Both modes: act is [M, ld] 16-bit (ld a multiple of 64), viewed as
// (64-element chunk, row, chunk index); one box is two k-blocks of 128 rows.
// ab (affine mode only): per Linear the [N, K/64] (step, offset) pairs.
template <bool kAffine>
cudaError_t launch_wide(const uint16_t* act, int64_t ld, const float* sa, const LinearGroup& grp,
                        const float* const* ab, int64_t M, int64_t N, int64_t K,
                        const uint32_t* amax, const uint32_t* nwpart, uint32_t* status,
                        uint2* list, cudaStream_t s) {
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[3] = {cuuint64_t(BK), cuuint64_t(M), cuuint64_t(ld / BK)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2u, cuuint64_t(BK) * 2u};
  const cuuint32_t box[3] = {BK, BNH, SS};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&map, kAffine ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
          const_cast<uint16_t*>(act), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // weights: [N, K] INT8 per Linear, boxes of 128 rows x 128 bytes (two k-blocks)
  WMaps wmaps;
  Outs outs = {};
  const cuuint64_t wdims[2] = {cuuint64_t(K), cuuint64_t(N)};
  const cuuint64_t wstrides[1] = {cuuint64_t(K)};
  const cuuint32_t wbox[2] = {SS * BK, BM};
  for (int g = 0; g < kMaxGroup; ++g) {
    // unused entries repeat the first Linear's map (never read)
    const int src = g < grp.G ? g : 0;
    if (enc(&wmaps.m[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(grp.wq[src]),
            wdims, wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    outs.sw[g] = grp.ws[src];
    outs.ab[g] = ab ? reinterpret_cast<const float2*>(ab[src]) : nullptr;
    outs.bias[g] = grp.bias[src];
    outs.y[g] = grp.y[src];
    outs.acc[g] = grp.acc[src];
  }

  Shape shp;
  shp.G = grp.G;
  shp.M = int(M);
  shp.N = int(N);
  shp.K = int(K);
  shp.KB = int((K + BK - 1) / BK);
  shp.NSS = (shp.KB + SS - 1) / SS;
  shp.mt = int((M + BN - 1) / BN);
  shp.mt128 = int((M + 127) / 128);
  shp.nt = int((N + BM - 1) / BM);
  shp.ntc = (shp.nt + CLUSTER - 1) / CLUSTER;
  shp.tiles = shp.G * shp.mt * shp.ntc;
  shp.list_cap = int(fallback_list_capacity(M, N));
  shp.seg_ss = norm_segment_len(K) / kSegQuantum;
  shp.wmax2 = uint64_t(128 * 128) * uint64_t(K);
  choose_raster(shp);

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_wide_kernel<kAffine>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int clusters = shp.tiles < sms / CLUSTER ? shp.tiles : sms / CLUSTER;
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
  // may start while the weight-norm pre-pass finishes
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_wide_kernel<kAffine>, map, wmaps, sa, outs, shp, amax,
                            nwpart, status, list);
}

}  // namespace

cudaError_t launch_gemm_wide(const uint16_t* act_f16, const float* sa, const LinearGroup& grp,
                             int64_t M, int64_t N, int64_t K, const uint32_t* amax,
                             const uint32_t* nwpart, uint32_t* status, uint2* list,
                             cudaStream_t s) {
  return launch_wide<false>(act_f16, gemm_tc_coded_ld(K), sa, grp, nullptr, M, N, K, amax,
                            nwpart, status, list, s);
}

cudaError_t launch_gemm_affine(const uint16_t* x, const LinearGroup& grp, const float* const* ab,
                               int64_t M, int64_t N, int64_t K, uint32_t* status,
                               cudaStream_t s) {
  return launch_wide<true>(x, K, nullptr, grp, ab, M, N, K, nullptr, nullptr, status, nullptr, s);
}

}  // namespace h3q
