// h3q_quant.cu -- A1 (weight) and A2 (activation) symmetric per-row INT8
// quantisers, and the INT8 -> FP16-coded-integer expansion.
//
// Rule (readings of "feat(mps): support MiniMax-H3 INT8 inference on Apple M5",
// LightX2V #1672, sections Validation and Summary by CodeRabbit):
//   a = max_k |x[k]|;  s = a / 127 (IEEE FP32 division, round to nearest even);
//   s = 1 when a == 0;  s = 2^-149 when a > 0 but a / 127 underflows to 0;
//   q[k] = clamp(rint(x[k] / s), -127, 127) with an IEEE FP32 division.
// The division is __fdiv_rn so that every q matches an IEEE-754 evaluation
// bit for bit; the build never uses fast-math or flush-to-zero.
#include <cuda_fp16.h>

#include "h3q_internal.cuh"
#include "h3q_tc_ptx.cuh"

namespace h3q {
namespace {

constexpr int kWarps = 8;        // rows per block: one warp per row
constexpr int kRegVecs = 24;     // 16-byte vectors per lane kept in registers

__device__ __forceinline__ float row_scale(float amax) {
  if (amax == 0.f) return 1.f;
  const float s = __fdiv_rn(amax, 127.f);
  return s == 0.f ? __int_as_float(1) : s;   // 2^-149, the smallest positive FP32
}

__device__ __forceinline__ int quant1(float x, float s) {
  const int q = __float2int_rn(__fdiv_rn(x, s));
  return max(-kQMax, min(kQMax, q));
}

__device__ __forceinline__ uint32_t pack2_f16(int a, int b) {
  return uint32_t(__half_as_ushort(__int2half_rn(a))) |
         (uint32_t(__half_as_ushort(__int2half_rn(b))) << 16);
}

__device__ __forceinline__ uint32_t pack2_f16f(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// |bf16| maximum of the 8 values in a 16-byte vector, as a 16-bit magnitude
// pattern: for finite BF16 values the order of |x| is the order of (bits & 0x7fff).
__device__ __forceinline__ uint32_t vec_absmax_bits(uint4 v) {
  uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                        __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  return (uint64_t(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }

// The fast path of quant_store8 gives the same integer as quant1(x, s), as
// an integer-valued float, cheaper.
// With r = RN(1/s) (s normal) and t = RN(x * r): t = (x/s)(1 + e1)(1 + e2),
// |e1|, |e2| <= 2^-24, and |x/s| <= 127 (1 + 2^-23), so |t - x/s| < 1.6e-5;
// the FP32 quotient RN(x/s) is within 2^-18 of x/s.  Hence |t - RN(x/s)| <
// 2^-15, and unless t lies within 2^-15 of a half-integer, RN(x/s) and t
// round to the same integer, with no tie.  Near a half-integer (about 6e-5 of
// inputs) the IEEE division decides.  Rounding t to an integer adds and
// subtracts 1.5 * 2^23: for |t| < 2^22 the sum's last place is 1, so the
// addition itself rounds t to nearest, ties to even.  `fast` is false for
// rows whose scale is too small for a normal reciprocal; those always divide.
// |x| <= absmax makes |q| <= 127 without a clamp.
//
// The rounding sum u = RN(t + 1.5 * 2^23) of an integer n in [-127, 127] is
// the FP32 pattern 0x4B400000 + n (its last place is 1), so u's low byte is
// n's two's-complement byte: the INT8 output is packed from those bytes with
// byte permutes, with no further conversion.
//
// Quantises 8 values, stores them, and returns the sum of their squares
// (exact: at most 8 * 127^2).  The work runs two values at a time on the
// paired FP32 instructions (each half the same IEEE operation as the scalar
// one), and the fallback is taken per vector: the fast results stand when
// every one of the eight passes its test, else all eight take the IEEE
// division, which gives the same integer wherever the test passes.  One
// branch per vector instead of one per value: the quantiser is bound by
// instruction issue otherwise.
template <bool kQ8, bool kF16>
__device__ __forceinline__ uint32_t quant_store8(uint4 v, float s, float r, bool fast,
                                                 int8_t* q8, uint16_t* qh, int64_t elem,
                                                 int64_t helem) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint64_t r2 = pack_f2(r, r);
  const uint64_t c2 = pack_f2(12582912.0f, 12582912.0f);
  const float lim = 0.5f - 0x1p-15f;
  // the low bytes of a pair's rounding sums: the pair's two INT8 codes
  const auto bytes2 = [](uint64_t u2) {
    uint32_t b;
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(b) : "r"(uint32_t(u2)), "r"(uint32_t(u2 >> 32)));
    return b;
  };
  uint64_t q2[4];
  uint32_t p[4];
  bool ok = fast;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // elements 2j (low half of w[j]) and 2j + 1 (high half), widened exactly
    const uint64_t x2 = (uint64_t(w[j] & 0xFFFF0000u) << 32) | (w[j] << 16);
    uint64_t t2, u2, d2;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t2) : "l"(x2), "l"(r2));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(u2) : "l"(t2), "l"(c2));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(q2[j]) : "l"(u2), "l"(c2));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d2) : "l"(t2), "l"(q2[j]));
    ok = ok && fabsf(lo_f(d2)) < lim && fabsf(hi_f(d2)) < lim;
    if constexpr (kQ8) p[j] = bytes2(u2);
  }
  if (!ok) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      q2[j] = pack_f2(float(quant1(__uint_as_float(w[j] << 16), s)),
                      float(quant1(__uint_as_float(w[j] & 0xFFFF0000u), s)));
      if constexpr (kQ8) {
        uint64_t u2;
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(u2) : "l"(q2[j]), "l"(c2));   // exact
        p[j] = bytes2(u2);
      }
    }
  }
  if constexpr (kQ8) {
    // elements 0..7 in order
    uint2 o;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o.x) : "r"(p[0]), "r"(p[1]));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o.y) : "r"(p[2]), "r"(p[3]));
    *reinterpret_cast<uint2*>(q8 + elem) = o;
  }
  if constexpr (kF16) {
    uint4 o;   // integers of magnitude <= 127 are exact in FP16
    o.x = pack2_f16f(lo_f(q2[0]), hi_f(q2[0]));
    o.y = pack2_f16f(lo_f(q2[1]), hi_f(q2[1]));
    o.z = pack2_f16f(lo_f(q2[2]), hi_f(q2[2]));
    o.w = pack2_f16f(lo_f(q2[3]), hi_f(q2[3]));
    *reinterpret_cast<uint4*>(qh + helem) = o;
  }
  uint64_t ss2 = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(ss2) : "l"(q2[j]), "l"(ss2));
  return uint32_t(lo_f(ss2)) + uint32_t(hi_f(ss2));
}

// A row's sums of q^2, one per norm segment.  Every sum is exact: it is at
// most 127^2 K < 2^32 for every supported K.
static_assert(kNormSegs == 4, "the segment selects below are written out for four");
struct SegSq {
  uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
  // v into the segment of element k (selects, so no register is indexed)
  __device__ __forceinline__ void add(int k, int seg_len, uint32_t v) {
    const int g = int(k >= seg_len) + int(k >= 2 * seg_len) + int(k >= 3 * seg_len);
    s0 += g == 0 ? v : 0u;
    s1 += g == 1 ? v : 0u;
    s2 += g == 2 ? v : 0u;
    s3 += g == 3 ? v : 0u;
  }
  __device__ __forceinline__ void warp_sum() {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, o);
      s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, o);
      s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
      s3 += __shfl_xor_sync(0xFFFFFFFFu, s3, o);
    }
  }
  __device__ __forceinline__ void store(uint4* p) const { *p = make_uint4(s0, s1, s2, s3); }
  __device__ __forceinline__ void add(const uint4& v) {
    s0 += v.x;
    s1 += v.y;
    s2 += v.z;
    s3 += v.w;
  }
};

// Folds a row's sums of squares of q into the running maxima of its block of
// 256 token rows: the whole row's sum into blk_max[block], each segment's
// into seg_max[block][segment] (read by the GEMM to decide whether a tile's
// FP32 sums stay exact without splitting K).
__device__ __forceinline__ void record_row_sq(uint32_t* blk_max, uint32_t* seg_max, int64_t row,
                                              const SegSq& q) {
  if (!blk_max) return;
  const int64_t b = row >> 8;
  atomicMax(blk_max + b, q.s0 + q.s1 + q.s2 + q.s3);
  uint32_t* sm = seg_max + b * kNormSegs;
  if (q.s0) atomicMax(sm + 0, q.s0);
  if (q.s1) atomicMax(sm + 1, q.s1);
  if (q.s2) atomicMax(sm + 2, q.s2);
  if (q.s3) atomicMax(sm + 3, q.s3);
}

// One warp per token row.  kRegs: the whole row (<= 32 * kRegVecs vectors)
// stays in registers between the absmax pass and the quantise pass, so X is
// read from memory once; otherwise the second pass re-reads the row.
template <bool kRegs, bool kQ8, bool kF16>
__global__ void __launch_bounds__(kWarps * 32)
quant_act_kernel(const uint16_t* __restrict__ x, int64_t M, int K, int8_t* __restrict__ q8,
                 float* __restrict__ scale, uint16_t* __restrict__ qh, int ldh,
                 uint32_t* __restrict__ sq_max, uint32_t* __restrict__ seg_max, int seg_len) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const int nvec = K >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * int64_t(K));
  const int64_t base = row * int64_t(K), hbase = row * int64_t(ldh);
  uint32_t mbits = 0;
  if constexpr (kF16) {   // zero the row's padding up to the coded row stride
    for (int j = nvec + lane; j < (ldh >> 3); j += 32)
      *reinterpret_cast<uint4*>(qh + hbase + 8 * int64_t(j)) = make_uint4(0, 0, 0, 0);
  }
  if constexpr (kRegs) {
    uint4 v[kRegVecs];
#pragma unroll
    for (int i = 0; i < kRegVecs; ++i) {
      const int j = lane + 32 * i;
      if (j < nvec) {
        v[i] = ld_stream(xr + j);
        mbits = max(mbits, vec_absmax_bits(v[i]));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mbits = max(mbits, __shfl_xor_sync(0xFFFFFFFFu, mbits, o));
    const float s = row_scale(__uint_as_float(mbits << 16));
    const float r = __frcp_rn(s);
    const bool fast = s >= 0x1p-120f;
    SegSq sq;
#pragma unroll
    for (int i = 0; i < kRegVecs; ++i) {
      const int j = lane + 32 * i;
      if (j < nvec)
        sq.add(8 * j, seg_len,
               quant_store8<kQ8, kF16>(v[i], s, r, fast, q8, qh, base + 8 * int64_t(j),
                                       hbase + 8 * int64_t(j)));
    }
    sq.warp_sum();
    if (lane == 0) {
      scale[row] = s;
      record_row_sq(sq_max, seg_max, row, sq);
    }
  } else {
    int j = lane;
    for (; j + 96 < nvec; j += 128) {
      const uint4 a = __ldg(xr + j), b = __ldg(xr + j + 32), c = __ldg(xr + j + 64),
                  d = __ldg(xr + j + 96);
      mbits = max(max(mbits, vec_absmax_bits(a)), vec_absmax_bits(b));
      mbits = max(max(mbits, vec_absmax_bits(c)), vec_absmax_bits(d));
    }
    for (; j < nvec; j += 32) mbits = max(mbits, vec_absmax_bits(__ldg(xr + j)));
#pragma unroll
    for (int o = 16; o; o >>= 1) mbits = max(mbits, __shfl_xor_sync(0xFFFFFFFFu, mbits, o));
    const float s = row_scale(__uint_as_float(mbits << 16));
    const float r = __frcp_rn(s);
    const bool fast = s >= 0x1p-120f;
    SegSq sq;
    for (j = lane; j < nvec; j += 32)
      sq.add(8 * j, seg_len,
             quant_store8<kQ8, kF16>(ld_stream(xr + j), s, r, fast, q8, qh,
                                     base + 8 * int64_t(j), hbase + 8 * int64_t(j)));
    sq.warp_sum();
    if (lane == 0) {
      scale[row] = s;
      record_row_sq(sq_max, seg_max, row, sq);
    }
  }
}

// One 256-thread block per token row, each thread holding kVPT 16-byte vectors
// of it in registers: X is read once, a row needs only a few registers per
// thread, so many rows are in flight per SM.
constexpr int kRowThreads = 256;

// Running maximum of |x| over the BF16 pairs of w: max.xorsign.abs keeps
// max(|a|, |b|) per half (with the XOR of the signs, dropped at the end).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w));
  return r;
}

// The row kernels keep their per-element work short, since a row's work is
// spread over 256 threads and any per-row step is repeated by all 8 warps:
//   - the absmax takes one paired BF16 instruction per 32-bit word;
//   - one warp turns the block's maximum into the scale s and its reciprocal
//     and publishes them through shared memory (the IEEE division and
//     reciprocal run once per row, not once per warp);
//   - with norm maxima requested (kSq), each thread stores the sum of q^2 of
//     each of its vectors in shared memory, and four warps then add up one
//     norm segment each while a fifth adds up the whole row.
template <int kVPT, bool kSq>
struct RowSmem {
  uint32_t red[kRowThreads / 32];
  float2 sr;
  uint32_t vsq[kSq ? kRowThreads * kVPT : 1];   // per-vector sums of q^2
};

// This thread's vectors of row `row` (j = threadIdx.x + 256 i), streamed past L1.
template <int kVPT>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ x, int64_t row, int K,
                                         int nvec, uint4 (&v)[kVPT]) {
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * int64_t(K));
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int j = int(threadIdx.x) + kRowThreads * i;
    if (j < nvec) v[i] = ld_stream(xr + j);
  }
}

// Block-collective: quantise one row held in registers (v, as load_row left
// it).  Three block barriers (two without kSq).
template <int kVPT, bool kQ8, bool kF16, bool kSq>
__device__ __forceinline__ void quant_row(RowSmem<kVPT, kSq>& sm, const uint4 (&v)[kVPT],
                                          int64_t row, int K, int nvec,
                                          int8_t* __restrict__ q8, float* __restrict__ scale,
                                          uint16_t* __restrict__ qh, int ldh,
                                          uint32_t* __restrict__ sq_max,
                                          uint32_t* __restrict__ seg_max, int seg_len) {
  constexpr int kWarpsPerRow = kRowThreads / 32;
  static_assert(kWarpsPerRow > kNormSegs, "a warp per norm segment and one for the row");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base = row * int64_t(K), hbase = row * int64_t(ldh);
  if constexpr (kF16) {   // zero the row's padding up to the coded row stride
    for (int j = nvec + int(threadIdx.x); j < (ldh >> 3); j += kRowThreads)
      *reinterpret_cast<uint4*>(qh + hbase + 8 * int64_t(j)) = make_uint4(0, 0, 0, 0);
  }
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    if (int(threadIdx.x) + kRowThreads * i < nvec) {
      m2 = bf16x2_absmax(bf16x2_absmax(m2, v[i].x), v[i].y);
      m2 = bf16x2_absmax(bf16x2_absmax(m2, v[i].z), v[i].w);
    }
  }
  uint32_t mbits = max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);
#pragma unroll
  for (int o = 16; o; o >>= 1) mbits = max(mbits, __shfl_xor_sync(0xFFFFFFFFu, mbits, o));
  if (lane == 0) sm.red[warp] = mbits;
  __syncthreads();
  if (warp == 0) {
    uint32_t m = lane < kWarpsPerRow ? sm.red[lane] : 0u;
#pragma unroll
    for (int o = kWarpsPerRow / 2; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) {
      const float sc = row_scale(__uint_as_float(m << 16));
      sm.sr = make_float2(sc, __frcp_rn(sc));
      scale[row] = sc;
    }
  }
  __syncthreads();
  const float s = sm.sr.x, r = sm.sr.y;
  const bool fast = s >= 0x1p-120f;
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int j = int(threadIdx.x) + kRowThreads * i;
    if (j < nvec) {
      const uint32_t sq = quant_store8<kQ8, kF16>(v[i], s, r, fast, q8, qh,
                                                  base + 8 * int64_t(j), hbase + 8 * int64_t(j));
      if constexpr (kSq) sm.vsq[j] = sq;
    }
  }
  if constexpr (kSq) {
    __syncthreads();
    // every sum below is exact: a row's sum of q^2 is at most 127^2 K < 2^32
    if (warp <= kNormSegs) {
      const int segv = seg_len >> 3;                  // vectors per norm segment
      const int j0 = warp < kNormSegs ? warp * segv : 0;
      const int j1 = warp < kNormSegs ? min(nvec, j0 + segv) : nvec;
      uint32_t t = 0;
      for (int j = j0 + lane; j < j1; j += 32) t += sm.vsq[j];
#pragma unroll
      for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
      if (lane == 0) {
        const int64_t b = row >> 8;
        if (warp == kNormSegs)
          atomicMax(sq_max + b, t);
        else if (t)
          atomicMax(seg_max + b * kNormSegs + warp, t);
      }
    }
  }
}

// One block per row: eight resident per SM for short rows (32 registers a
// thread), two for rows of up to 12 * 256 vectors.  (With INT8 codes out the
// short-row kernel spills 24 bytes at 32 registers; measured, eight blocks
// with the spill beat six without it: 24.9 against 25.8 us at 8192 x 5376.)
template <int kVPT, bool kQ8, bool kF16, bool kSq>
__global__ void __launch_bounds__(kRowThreads, kVPT <= 3 ? 8 : 2)
quant_act_row_kernel(const uint16_t* __restrict__ x, int K, int8_t* __restrict__ q8,
                     float* __restrict__ scale, uint16_t* __restrict__ qh, int ldh,
                     uint32_t* __restrict__ sq_max, uint32_t* __restrict__ seg_max,
                     int seg_len) {
  __shared__ RowSmem<kVPT, kSq> sm;
  // with programmatic dependent launch: let the next grid be scheduled once
  // every block has started, and wait for the previous grid's writes before
  // reading X (both return at once without the launch attribute)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nvec = K >> 3;
  uint4 v[kVPT];
  load_row<kVPT>(x, blockIdx.x, K, nvec, v);
  quant_row<kVPT, kQ8, kF16, kSq>(sm, v, blockIdx.x, K, nvec, q8, scale, qh, ldh, sq_max,
                                  seg_max, seg_len);
}

// The same per-row work for long rows (K up to 24576), staged in shared
// memory: a persistent
// grid (two 256-thread blocks per SM), each block taking rows b, b + G,
// b + 2G, ...  Thread 0 keeps `ring` rows in flight with untiled bulk copies
// (one mbarrier per ring slot), so HBM latency is covered by the copies
// rather than by the number of resident blocks, and a block passes one
// barrier per row: the absmax partials of a row and the sum-of-squares
// partials of the row before share it (double-buffered by row parity), and
// a slot is refilled as soon as every thread has its vectors in registers.
// Every wait is bounded; on a timeout the block records an error bit in
// *err and stops.
constexpr int kStagedThreads = 256;
constexpr int kStagedSmem = 104 * 1024;   // row ring of a block: two blocks fit an SM
constexpr uint32_t kErrQuantWait = 1u << 16;

template <int kVPT, bool kQ8, bool kF16>
__global__ void __launch_bounds__(kStagedThreads, 2)
quant_act_staged_kernel(const uint16_t* __restrict__ x, int64_t M, int K, int ring, int slot_bytes,
                        int8_t* __restrict__ q8, float* __restrict__ scale,
                        uint16_t* __restrict__ qh, int ldh, uint32_t* __restrict__ sq_max,
                        uint32_t* __restrict__ seg_max, int seg_len, uint32_t* __restrict__ err) {
  namespace P = ptx;
  extern __shared__ __align__(128) uint8_t rows_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(rows_smem + size_t(ring) * slot_bytes);
  __shared__ uint32_t red[2][kStagedThreads / 32];
  __shared__ uint4 red_sq[2][kStagedThreads / 32];
  __shared__ int give_up;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t G = gridDim.x;
  const uint32_t row_bytes = uint32_t(K) * 2u;
  const int nvec = K >> 3;
  if (tid == 0) {
    for (int i = 0; i < ring; ++i) P::mbar_init(&full[i], 1);
    P::fence_mbar_init();
    give_up = 0;
    for (int i = 0; i < ring; ++i) {
      const int64_t row = blockIdx.x + int64_t(i) * G;
      if (row >= M) break;
      P::mbar_arrive_expect_tx(&full[i], row_bytes);
      P::bulk_load(P::smem_u32(rows_smem + size_t(i) * slot_bytes), x + row * int64_t(K),
                   row_bytes, &full[i]);
    }
  }
  __syncthreads();
  int64_t it = 0;
  for (;; ++it) {
    const int64_t row = blockIdx.x + it * G;
    if (row >= M) break;
    const int slot = int(it % ring);
    const int par = int(it & 1);
    // this row's copy (bounded wait; a thread that gives up flags the block,
    // which stops together after the barrier below)
    const uint32_t bar = P::smem_u32(&full[slot]);
    const uint32_t phase = uint32_t(it / ring) & 1u;
    bool ok = P::mbar_test(bar, phase);
    if (!ok) {
      const uint64_t t0 = P::globaltimer();
      while (!(ok = P::mbar_test(bar, phase))) {
        if (P::globaltimer() - t0 > P::kWaitTimeoutNs) {
          give_up = 1;
          if (err) atomicOr(err, kErrQuantWait);
          break;
        }
      }
    }
    const uint4* xr = reinterpret_cast<const uint4*>(rows_smem + size_t(slot) * slot_bytes);
    uint4 v[kVPT];
    uint32_t mbits = 0;
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
      const int j = tid + kStagedThreads * i;
      v[i] = (ok && j < nvec) ? xr[j] : make_uint4(0, 0, 0, 0);
      mbits = max(mbits, vec_absmax_bits(v[i]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mbits = max(mbits, __shfl_xor_sync(0xFFFFFFFFu, mbits, o));
    if (lane == 0) red[par][warp] = mbits;
    __syncthreads();
    if (give_up) break;
    if (tid == 0) {
      // the slot's vectors are in registers: refill it
      const int64_t nrow = row + int64_t(ring) * G;
      if (nrow < M) {
        P::mbar_arrive_expect_tx(&full[slot], row_bytes);
        P::bulk_load(P::smem_u32(rows_smem + size_t(slot) * slot_bytes), x + nrow * int64_t(K),
                     row_bytes, &full[slot]);
      }
      // the previous row's sums of squares
      if (sq_max && it > 0) {
        SegSq t;
#pragma unroll
        for (int w = 0; w < kStagedThreads / 32; ++w) t.add(red_sq[par ^ 1][w]);
        record_row_sq(sq_max, seg_max, row - G, t);
      }
    }
#pragma unroll
    for (int w = 0; w < kStagedThreads / 32; ++w) mbits = max(mbits, red[par][w]);
    const float s = row_scale(__uint_as_float(mbits << 16));
    const float r = __frcp_rn(s);
    const bool fast = s >= 0x1p-120f;
    const int64_t base = row * int64_t(K), hbase = row * int64_t(ldh);
    if constexpr (kF16) {   // zero the row's padding up to the coded row stride
      for (int j = nvec + tid; j < (ldh >> 3); j += kStagedThreads)
        *reinterpret_cast<uint4*>(qh + hbase + 8 * int64_t(j)) = make_uint4(0, 0, 0, 0);
    }
    SegSq sq;
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
      const int j = tid + kStagedThreads * i;
      if (j < nvec)
        sq.add(8 * j, seg_len,
               quant_store8<kQ8, kF16>(v[i], s, r, fast, q8, qh, base + 8 * int64_t(j),
                                       hbase + 8 * int64_t(j)));
    }
    if (tid == 0) scale[row] = s;
    if (sq_max) {
      sq.warp_sum();
      if (lane == 0) sq.store(&red_sq[par][warp]);
    }
  }
  // the last row's sums of squares
  __syncthreads();
  if (tid == 0 && sq_max && it > 0 && !give_up) {
    SegSq t;
#pragma unroll
    for (int w = 0; w < kStagedThreads / 32; ++w) t.add(red_sq[(it - 1) & 1][w]);
    record_row_sq(sq_max, seg_max, blockIdx.x + (it - 1) * G, t);
  }
}

// Weight rows: FP32 or BF16.  Not on the timed path; plain two-pass loops,
// plus a finiteness check (a row with Inf/NaN gets a NaN scale).
template <typename T>
__device__ __forceinline__ float load_w(const T* p, int64_t i);
template <>
__device__ __forceinline__ float load_w<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_w<uint16_t>(const uint16_t* p, int64_t i) {
  return __uint_as_float(uint32_t(p[i]) << 16);
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
quant_weight_kernel(const T* __restrict__ w, int64_t N, int K, int8_t* __restrict__ q8,
                    float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= N) return;
  const T* wr = w + row * int64_t(K);
  float amax = 0.f;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    const float a = fabsf(load_w<T>(wr, k));
    bad |= !(a <= 3.4028234663852886e38f);   // Inf or NaN
    amax = fmaxf(amax, a);
  }
  bad = __any_sync(0xFFFFFFFFu, bad);
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float s = row_scale(amax);
  int8_t* qr = q8 + row * int64_t(K);
  for (int k = lane; k < K; k += 32) qr[k] = int8_t(bad ? 0 : quant1(load_w<T>(wr, k), s));
  if (lane == 0) scale[row] = bad ? __int_as_float(0x7FC00000) : s;
}

// Group-wise affine quantisation of weight rows (the comparison scheme;
// offline, plain): one warp per row, one group of 64 at a time, two values
// per lane.  With L = 2^bits - 1 levels (255 or 15), per group: lo, hi = min,
// max; step = RN(RN(hi - lo) / L) (1 for a constant group, the smallest
// positive FP32 if it underflows); offset = lo; q = clamp(rint(RN(RN(w - lo) /
// step)), 0, L), one code per byte.  A group with Inf or NaN gets a NaN step
// and zero codes.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
quant_weight_affine_kernel(const T* __restrict__ w, int64_t N, int K, int levels,
                           uint8_t* __restrict__ q, float2* __restrict__ ab) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= N) return;
  const T* wr = w + row * int64_t(K);
  const int groups = K / 64;
  for (int gi = 0; gi < groups; ++gi) {
    const int k0 = gi * 64 + lane, k1 = k0 + 32;
    const float v0 = load_w<T>(wr, k0), v1 = load_w<T>(wr, k1);
    bool bad = !(fabsf(v0) <= 3.4028234663852886e38f) || !(fabsf(v1) <= 3.4028234663852886e38f);
    bad = __any_sync(0xFFFFFFFFu, bad);
    float lo = fminf(v0, v1), hi = fmaxf(v0, v1);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    }
    float step = __fdiv_rn(__fsub_rn(hi, lo), float(levels));
    if (hi == lo) step = 1.f;
    else if (step == 0.f) step = __int_as_float(1);
    const auto code = [&](float v) {
      const int c = __float2int_rn(__fdiv_rn(__fsub_rn(v, lo), step));
      return uint8_t(bad ? 0 : max(0, min(levels, c)));
    };
    q[row * int64_t(K) + k0] = code(v0);
    q[row * int64_t(K) + k1] = code(v1);
    if (lane == 0)
      ab[row * groups + gi] = make_float2(bad ? __int_as_float(0x7FC00000) : step, lo);
  }
}

// One 256-thread block per row: INT8 -> FP16-coded integers, rows of stride
// ldh with the padding zeroed, and the row's sum of squares.
__global__ void __launch_bounds__(256)
int8_to_f16_kernel(const int8_t* __restrict__ q, int K, int ldh, uint16_t* __restrict__ out,
                   uint32_t* __restrict__ sq_max, uint32_t* __restrict__ seg_max, int seg_len) {
  __shared__ uint4 red[8];
  const int64_t row = blockIdx.x;
  const int groups = ldh >> 4;                      // 16-element groups of a coded row
  SegSq sq;
  for (int grp = threadIdx.x; grp < groups; grp += 256) {
    uint4* dst = reinterpret_cast<uint4*>(out + row * ldh + 16 * int64_t(grp));
    if (16 * grp >= K) {
      dst[0] = make_uint4(0, 0, 0, 0);
      dst[1] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + row * K + 16 * int64_t(grp)));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
    uint32_t g2 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b0 = int(int8_t(w[j])), b1 = int(int8_t(w[j] >> 8));
      const int b2 = int(int8_t(w[j] >> 16)), b3 = int(int8_t(w[j] >> 24));
      o[2 * j] = pack2_f16(b0, b1);
      o[2 * j + 1] = pack2_f16(b2, b3);
      g2 = uint32_t(__dp4a(int(w[j]), int(w[j]), int(g2)));
    }
    sq.add(16 * grp, seg_len, g2);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  if (sq_max) {
    sq.warp_sum();
    if ((threadIdx.x & 31) == 0) sq.store(&red[threadIdx.x >> 5]);
    __syncthreads();
    if (threadIdx.x == 0) {
      SegSq t;
#pragma unroll
      for (int w = 0; w < 8; ++w) t.add(red[w]);
      record_row_sq(sq_max, seg_max, row, t);
    }
  }
}

// Weight-row norms for the GEMM's exactness test.  Every block first checks
// whether any block of 256 tokens could fail the test against the largest
// possible weight row (sum q^2 <= 128^2 K); if none can, the GEMM never reads
// the norms and the block returns at once.  Otherwise, for each group b of 16
// weight rows (16b .. 16b+15; the blocks stride over the groups), the block's
// 16 warps sum q^2 with DP4A on 16-byte loads, per norm segment, and write the
// largest whole-row sum to part[b] and the largest sum of each segment s to
// part[nblocks + b * kNormSegs + s].  The sums are
// taken modulo 2^32, which is exact: K * 128^2 < 2^32 for every supported K.
constexpr int kNormRows = 16;

struct WeightPtrs {
  const int8_t* w[kMaxGroup];
};

__global__ void __launch_bounds__(32 * kNormRows)
weight_norm_kernel(const WeightPtrs wqs, int64_t N, int K, int blocks_per_linear, int nblocks,
                   const uint32_t* __restrict__ amax, int mt2, uint32_t* __restrict__ part,
                   int seg_len) {
  // the quantiser that wrote amax may still be finishing (programmatic
  // dependent launch): wait for it, then let the GEMM be scheduled
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint4 red[kNormRows];
  __shared__ int needed;
  if (threadIdx.x == 0) needed = 0;
  __syncthreads();
  const uint64_t wmax2 = uint64_t(128 * 128) * uint64_t(K);
  for (int i = threadIdx.x; i < mt2; i += blockDim.x)
    if (uint64_t(amax[i]) * wmax2 > (uint64_t(1) << 48)) needed = 1;
  __syncthreads();
  if (!needed) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid-stride over the row groups: group b covers rows 16 (b mod
  // blocks_per_linear) .. + 15 of Linear b / blocks_per_linear (a small grid,
  // so that the early return above costs one wave of blocks)
  for (int b = blockIdx.x; b < nblocks; b += gridDim.x) {
    const int g = b / blocks_per_linear;
    const int8_t* __restrict__ wq = wqs.w[g];
    const int64_t n = int64_t(b - g * blocks_per_linear) * kNormRows + warp;
    SegSq sq;
    if (n < N) {
      // a 16-byte vector never straddles two segments (they are multiples of 128)
      const uint4* row = reinterpret_cast<const uint4*>(wq + n * K);
      const int nv = K >> 4;
      int i = lane;
      for (; i + 96 < nv; i += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(row + i + 32 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t t = uint32_t(__dp4a(int(v[u].x), int(v[u].x), 0));
          t = uint32_t(__dp4a(int(v[u].y), int(v[u].y), int(t)));
          t = uint32_t(__dp4a(int(v[u].z), int(v[u].z), int(t)));
          t = uint32_t(__dp4a(int(v[u].w), int(v[u].w), int(t)));
          sq.add(16 * (i + 32 * u), seg_len, t);
        }
      }
      for (; i < nv; i += 32) {
        const uint4 v = __ldg(row + i);
        uint32_t t = uint32_t(__dp4a(int(v.x), int(v.x), 0));
        t = uint32_t(__dp4a(int(v.y), int(v.y), int(t)));
        t = uint32_t(__dp4a(int(v.z), int(v.z), int(t)));
        t = uint32_t(__dp4a(int(v.w), int(v.w), int(t)));
        sq.add(16 * i, seg_len, t);
      }
    }
    sq.warp_sum();
    if (lane == 0) sq.store(&red[warp]);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t m = 0;
      uint4 ms = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int w = 0; w < kNormRows; ++w) {
        const uint4 r = red[w];
        m = max(m, r.x + r.y + r.z + r.w);
        ms = make_uint4(max(ms.x, r.x), max(ms.y, r.y), max(ms.z, r.z), max(ms.w, r.w));
      }
      part[b] = m;
      reinterpret_cast<uint4*>(part + nblocks)[b] = ms;
    }
    __syncthreads();                              // red[] is rewritten next round
  }
}

// The per-segment activation norm maxima follow the per-block ones.
uint32_t* seg_maxima(uint32_t* sq_max, int64_t M) {
  return sq_max ? sq_max + (M + kNormTokens - 1) / kNormTokens : nullptr;
}

template <bool kRegs>
cudaError_t launch_act(const uint16_t* x, int64_t M, int K, int8_t* q, float* s, uint16_t* qh,
                       int ldh, uint32_t* sqm, cudaStream_t st) {
  const dim3 grid(unsigned((M + kWarps - 1) / kWarps)), block(kWarps * 32);
  uint32_t* sgm = seg_maxima(sqm, M);
  const int sl = norm_segment_len(K);
  if (q && qh)
    quant_act_kernel<kRegs, true, true><<<grid, block, 0, st>>>(x, M, K, q, s, qh, ldh, sqm,
                                                                sgm, sl);
  else if (q)
    quant_act_kernel<kRegs, true, false><<<grid, block, 0, st>>>(x, M, K, q, s, qh, ldh, sqm,
                                                                 sgm, sl);
  else
    quant_act_kernel<kRegs, false, true><<<grid, block, 0, st>>>(x, M, K, q, s, qh, ldh, sqm,
                                                                 sgm, sl);
  return cudaGetLastError();
}

template <int kVPT, bool kQ8, bool kF16>
cudaError_t launch_rows_sq(dim3 grid, cudaStream_t st, const uint16_t* x, int K, int8_t* q,
                           float* s, uint16_t* qh, int ldh, uint32_t* sqm, uint32_t* sgm,
                           int sl) {
  if (sqm) {
    quant_act_row_kernel<kVPT, kQ8, kF16, true><<<grid, kRowThreads, 0, st>>>(x, K, q, s, qh,
                                                                             ldh, sqm, sgm, sl);
    return cudaGetLastError();
  }
  // Where the quantiser runs on its own (h3q_quantize_act), it is launched
  // with programmatic dependent launch: its blocks may be scheduled while the
  // previous kernel on the stream finishes, and they wait for that kernel's
  // writes (griddepcontrol.wait) before they read X.  Back to back, that
  // overlaps each launch's ramp with the previous launch's tail: 24.95 ->
  // 22.7 us at 8192 x 5376 in steady state.  (Inside a Linear call the
  // quantiser follows the memset of the workspace's status block, which this
  // attribute does not overlap.)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kRowThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_act_row_kernel<kVPT, kQ8, kF16, false>, x, K, q, s, qh,
                            ldh, sqm, sgm, sl);
}

template <int kVPT>
cudaError_t launch_rows(const uint16_t* x, int64_t M, int K, int8_t* q, float* s, uint16_t* qh,
                        int ldh, uint32_t* sqm, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(M));
  uint32_t* sgm = seg_maxima(sqm, M);
  const int sl = norm_segment_len(K);
  if (q && qh) return launch_rows_sq<kVPT, true, true>(grid, st, x, K, q, s, qh, ldh, sqm, sgm, sl);
  if (q) return launch_rows_sq<kVPT, true, false>(grid, st, x, K, q, s, qh, ldh, sqm, sgm, sl);
  return launch_rows_sq<kVPT, false, true>(grid, st, x, K, q, s, qh, ldh, sqm, sgm, sl);
}

template <int kVPT, bool kQ8, bool kF16>
cudaError_t launch_staged_one(const uint16_t* x, int64_t M, int K, int8_t* q, float* s,
                              uint16_t* qh, int ldh, uint32_t* sqm, uint32_t* err,
                              cudaStream_t st) {
  const int slot = (2 * K + 127) / 128 * 128;
  const int ring = max(2, min(8, kStagedSmem / slot));
  const size_t smem = size_t(ring) * slot + size_t(ring) * sizeof(uint64_t);
  auto kern = quant_act_staged_kernel<kVPT, kQ8, kF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int64_t blocks = M < 2 * int64_t(sms) ? M : 2 * int64_t(sms);
  kern<<<unsigned(blocks), kStagedThreads, smem, st>>>(x, M, K, ring, slot, q, s, qh, ldh, sqm,
                                                      seg_maxima(sqm, M), norm_segment_len(K),
                                                      err);
  return cudaGetLastError();
}

template <int kVPT>
cudaError_t launch_staged(const uint16_t* x, int64_t M, int K, int8_t* q, float* s,
                          uint16_t* qh, int ldh, uint32_t* sqm, uint32_t* err, cudaStream_t st) {
  if (q && qh) return launch_staged_one<kVPT, true, true>(x, M, K, q, s, qh, ldh, sqm, err, st);
  if (q) return launch_staged_one<kVPT, true, false>(x, M, K, q, s, qh, ldh, sqm, err, st);
  return launch_staged_one<kVPT, false, true>(x, M, K, q, s, qh, ldh, sqm, err, st);
}

}  // namespace

cudaError_t launch_quantize_act(const uint16_t* x, int64_t M, int64_t K, int8_t* q,
                                float* scale, uint16_t* q_f16, int64_t ldh, uint32_t* sq_max,
                                cudaStream_t s, uint32_t* err) {
  const int64_t nvec = K / 8;
  // Short rows: one block per row, with enough blocks resident to keep HBM
  // busy (a persistent grid that loads the next row while it quantises the
  // current one measured slower: 26.6 against 25.9 us alone, 33.5 against
  // 30.3 us in a call).  Longer rows (measured at K = 21504: 525 against 559
  // us), when the call has a status word for the bounded waits: rows staged
  // in shared memory.
  if (nvec <= kRowThreads * 3)
    return launch_rows<3>(x, M, int(K), q, scale, q_f16, int(ldh), sq_max, s);
  if (err && nvec <= kStagedThreads * 12)
    return launch_staged<12>(x, M, int(K), q, scale, q_f16, int(ldh), sq_max, err, s);
  if (nvec <= kRowThreads * 12)
    return launch_rows<12>(x, M, int(K), q, scale, q_f16, int(ldh), sq_max, s);
  return launch_act<false>(x, M, int(K), q, scale, q_f16, int(ldh), sq_max, s);
}

cudaError_t launch_quantize_weights(const void* w, int w_dtype, int64_t N, int64_t K,
                                    int8_t* q, float* scale, cudaStream_t s) {
  const dim3 grid(unsigned((N + kWarps - 1) / kWarps)), block(kWarps * 32);
  if (w_dtype == H3Q_DTYPE_F32)
    quant_weight_kernel<float><<<grid, block, 0, s>>>(static_cast<const float*>(w), N, int(K),
                                                      q, scale);
  else
    quant_weight_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t*>(w), N,
                                                         int(K), q, scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights_affine(const void* w, int w_dtype, int bits, int64_t N,
                                           int64_t K, uint8_t* q, float* ab, cudaStream_t s) {
  const dim3 grid(unsigned((N + kWarps - 1) / kWarps)), block(kWarps * 32);
  float2* ab2 = reinterpret_cast<float2*>(ab);
  const int levels = (1 << bits) - 1;
  if (w_dtype == H3Q_DTYPE_F32)
    quant_weight_affine_kernel<float><<<grid, block, 0, s>>>(static_cast<const float*>(w), N,
                                                             int(K), levels, q, ab2);
  else
    quant_weight_affine_kernel<uint16_t><<<grid, block, 0, s>>>(
        static_cast<const uint16_t*>(w), N, int(K), levels, q, ab2);
  return cudaGetLastError();
}

cudaError_t launch_weight_norms(const LinearGroup& grp, int64_t N, int64_t K,
                                const uint32_t* amax, int64_t M, uint32_t* nwpart,
                                cudaStream_t s) {
  static_assert(128 / kNormRows == kNormParts, "partial maxima per 128-channel block");
  WeightPtrs wqs = {};
  for (int g = 0; g < grp.G; ++g) wqs.w[g] = grp.wq[g];
  const int per = static_cast<int>((N + 127) / 128 * kNormParts);
  const int nblocks = per * grp.G;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // one wave of resident blocks (four of 512 threads per SM)
  cfg.gridDim = dim3(static_cast<unsigned>(nblocks < 4 * sms ? nblocks : 4 * sms));
  cfg.blockDim = dim3(32 * kNormRows);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int mt2 = static_cast<int>((M + kNormTokens - 1) / kNormTokens);
  return cudaLaunchKernelEx(&cfg, weight_norm_kernel, wqs, N, static_cast<int>(K), per, nblocks,
                            amax, mt2, nwpart, norm_segment_len(K));
}

cudaError_t launch_int8_to_f16(const int8_t* q, int64_t M, int64_t K, int64_t ldh,
                               uint16_t* out, uint32_t* sq_max, cudaStream_t s) {
  int8_to_f16_kernel<<<static_cast<unsigned>(M), 256, 0, s>>>(
      q, int(K), int(ldh), out, sq_max, seg_maxima(sq_max, M), norm_segment_len(K));
  return cudaGetLastError();
}

}  // namespace h3q
