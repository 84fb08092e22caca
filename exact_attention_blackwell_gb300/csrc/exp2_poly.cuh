// exp2_poly.cuh — 2^x evaluated on the FMA pipe instead of the special-function
// unit (FlashAttention-4 paper summary, section 2.B: the exponential is emulated
// with FMA instructions, using a polynomial of degree 3 to 5 for the fractional
// part, in parallel with the hardware unit).
//
// Method (Cody & Waite style range reduction, in base 2 where it is exact):
//   j = rint(x) is obtained by adding 1.5*2^23 (the sum's low mantissa bits are
//   then the integer), f = x - j lies in [-1/2, 1/2] and is exact;
//   2^f ~= 1 + f (C1 + f (C2 + f C3)), a minimax fit of relative error made by
//   fit_exp2.py (coefficients in exp2_poly_coeffs.h);
//   2^j is put into the exponent field with one integer add.
// The shift constant carries an extra +64 so that the integer add never leaves
// the normal range; one exact multiply by 2^-64 then takes the result back,
// rounding correctly into the subnormal range for x in [-150, -126).
#pragma once

#include "exp2_poly_coeffs.h"
#include "ptx.cuh"

namespace fa {

__device__ __forceinline__ float mul_rn_noftz(float a, float b) {
  float r;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// 2^x for x <= 63 (2^(j+64) must stay below the fp32 exponent limit);
// x < -150 (including -inf) returns +0.
__device__ __forceinline__ float exp2_poly(float x) {
  constexpr float kShift = 12582912.0f + 64.0f;  // 1.5 * 2^23 + 64
  x = fmaxf(x, -150.0f);
  const float t = __fadd_rn(x, kShift);  // mantissa low bits: j + 64, j = rint(x)
  const float j = __fsub_rn(t, kShift);  // rint(x), exact
  const float f = __fsub_rn(x, j);       // exact, |f| <= 1/2
  const float p = __fmaf_rn(__fmaf_rn(__fmaf_rn(FA_EXP2_C3, f, FA_EXP2_C2), f, FA_EXP2_C1), f, 1.0f);
  const int bits = __float_as_int(p) + (__float_as_int(t) << 23);  // p * 2^(j + 64)
  return mul_rn_noftz(__int_as_float(bits), 0x1p-64f);
}

// Two values with f32x2 arithmetic: the same operations as exp2_poly, each
// rounded once (x - j as fma(j, -1, x)), so each result equals exp2_poly of its
// input bit for bit in half the floating-point instructions.
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float &y0, float &y1) {
  constexpr float kShift = 12582912.0f + 64.0f;
  x0 = fmaxf(x0, -150.0f);
  x1 = fmaxf(x1, -150.0f);
  float t0, t1, j0, j1, f0, f1, p0, p1;
  fadd2(t0, t1, x0, x1, kShift, kShift);
  fadd2(j0, j1, t0, t1, -kShift, -kShift);
  ffma2(f0, f1, j0, j1, -1.0f, -1.0f, x0, x1);
  ffma2(p0, p1, FA_EXP2_C3, FA_EXP2_C3, f0, f1, FA_EXP2_C2, FA_EXP2_C2);
  ffma2(p0, p1, p0, p1, f0, f1, FA_EXP2_C1, FA_EXP2_C1);
  ffma2(p0, p1, p0, p1, f0, f1, 1.0f, 1.0f);
  const int b0 = __float_as_int(p0) + (__float_as_int(t0) << 23);
  const int b1 = __float_as_int(p1) + (__float_as_int(t1) << 23);
  fmul2(y0, y1, __int_as_float(b0), __int_as_float(b1), 0x1p-64f, 0x1p-64f);
}

}  // namespace fa
