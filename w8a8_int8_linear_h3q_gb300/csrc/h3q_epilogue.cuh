// h3q_epilogue.cuh -- A4: dequantise, add the bias, round once to BF16.
//
//   y = BF16_RNE(acc * s_a * s_w + bias)
//
// The bias is added before the single rounding of the output ("MLX
// implementation and experiment report", What the default preserves: biased
// BF16 linears use an addmm epilogue).  The value is formed in FP32 with
// error-free transformations (an FMA-exact two-product for s_a * s_w and for
// the product with the accumulator, and a two-sum with the bias) so that its
// error stays far below one BF16 ulp even when the product and the bias
// nearly cancel, and so that no FP32 intermediate overflows or underflows
// unless the exact result does.  The result is within one BF16 ulp of the
// exact value of the expression.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace h3q {

// Exact-transformation path: used where the cheap path below cannot prove
// its error small enough.
static __device__ __noinline__ float epilogue_value_careful(int acc, float sa, float sw, float bias) {
  if (acc == 0) return bias;                       // also covers 0 * (huge scale)
  float sa_ = sa, back = 1.f;
  float p_hi = __fmul_rn(sa_, sw);
  if (p_hi < 0x1p-60f) {                           // keep the two-product exact: rescale by 2^64
    sa_ = __fmul_rn(sa, 0x1p64f);
    p_hi = __fmul_rn(sa_, sw);
    back = 0x1p-64f;
  }
  if (isinf(p_hi)) return acc > 0 ? p_hi : -p_hi;  // |exact| >= FP32 max > BF16 max
  const float p_lo = __fmaf_rn(sa_, sw, -p_hi);    // s_a * s_w == p_hi + p_lo exactly
  const float a_hi = __int2float_rn(acc);
  const float a_lo = __ll2float_rn(static_cast<long long>(acc) - __float2ll_rz(a_hi));
  float t_hi = __fmul_rn(a_hi, p_hi);
  if (isinf(t_hi)) return t_hi;                    // exact result overflows as well
  float t_lo = __fmaf_rn(a_hi, p_hi, -t_hi);       // exact error of t_hi
  t_lo = __fmaf_rn(a_hi, p_lo, t_lo);
  t_lo = __fmaf_rn(a_lo, p_hi, t_lo);              // a_lo * p_lo is below 2^-47 relative
  if (back != 1.f) {
    t_hi = __fmul_rn(t_hi, back);
    t_lo = __fmul_rn(t_lo, back);
  }
  // two-sum of t_hi and the bias, then the low parts
  const float s = __fadd_rn(t_hi, bias);
  const float bv = __fsub_rn(s, t_hi);
  const float err = __fadd_rn(__fsub_rn(t_hi, __fsub_rn(s, bv)), __fsub_rn(bias, bv));
  return __fadd_rn(s, __fadd_rn(err, t_lo));
}

// The scales of the cheap path: s_a zero or in [2^-60, 2^45], s_w in
// [2^-40, 2^45].  Then c = RN(s_a * s_w) is zero or in [2^-100, 2^90], and for
// 1 <= |acc| <= 2^31, P = RN(float(acc) * c) is zero or in [2^-100, 2^121]:
// finite and normal.
__device__ __forceinline__ bool epilogue_scales_in_range(float sa, float sw) {
  return (sa == 0.f || (sa >= 0x1p-60f && sa <= 0x1p45f)) && (sw >= 0x1p-40f && sw <= 0x1p45f);
}

// Cheap path first: c = RN(s_a * s_w), then v = RN(float(acc) * c + bias), one
// fused multiply-add.  float(acc) is exact up to |acc| = 2^24 and within 2^-24
// relative above, and c is within 2^-24 relative, so the FMA's exact argument
// differs from the exact value by at most 2^-23 |acc c|, and its rounding adds
// at most 2^-24 |v|.  When |v| >= 2^-10 |bias|, |acc c| = |v - bias| <= 1025 |v|
// (up to those rounding terms), so the total is below 2^-12 |v|, far under
// half a BF16 ulp (>= 2^-9 |v|), and one BF16 rounding of v lands within one
// ulp of the exact value.  A zero accumulator gives v = bias exactly.
// Cancellation (|v| < 2^-10 |bias|) or scales outside the range above take
// the exact path; with acc != 0 the check also keeps v a normal FP32 number
// (|acc c| >= 2^-100 when the scales are in range).  Every kernel forms y by
// these same operations (the hot kernel's paired FP32 instructions perform
// them two tokens at a time), so y depends on (acc, s_a, s_w, bias) alone: not
// on the kernel, the tile or the call that produced the accumulator.
__device__ __forceinline__ float epilogue_value(int acc, float sa, float sw, float bias) {
  if (epilogue_scales_in_range(sa, sw)) {
    const float v = __fmaf_rn(__int2float_rn(acc), __fmul_rn(sa, sw), bias);
    if (fabsf(v) >= fabsf(bias) * 0x1p-10f) return v;
  }
  if (acc == 0) return bias;
  return epilogue_value_careful(acc, sa, sw, bias);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

// A bias element as the epilogue uses it: its FP32 value, with -0 taken as +0
// (adding +0 leaves every other value unchanged).  A zero accumulator then
// gives v = +0 + bias with the same bits whether the accumulator is held as
// the integer 0 or as an FP32 sum that came out -0.
__device__ __forceinline__ float bias_value(uint16_t b) {
  return __fadd_rn(bf16_bits_to_float(b), 0.f);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

}  // namespace h3q
