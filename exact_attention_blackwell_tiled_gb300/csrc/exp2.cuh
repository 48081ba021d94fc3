// exp2.cuh -- the two exponential paths of the softmax.
//
// The FlashAttention-4 pages (key contribution #2) spread the softmax
// exponentials over two units: the hardware exp2 (MUFU) and a degree-3
// polynomial evaluated on the FMA pipe, stated to be accurate enough for bf16.
// The pages give neither coefficients nor range reduction; this file supplies
// both:
//   x = n + f,  n = round-to-nearest(x),  f in [-1/2, 1/2]
//   2^x = 2^n * p(f),  p = minimax (Remez, relative error) cubic for 2^f on
//   [-1/2, 1/2]; fitted by fit_exp2_poly.py, max relative error 7.5e-5 in fp32,
//   far below the bf16 half-ulp 2^-9.
// n is obtained by adding 1.5 * 2^23 (the sum's low mantissa bits then hold
// round(x) in two's complement), and 2^n is applied by adding n << 23 to the
// bits of p(f) -- an integer add, so the path uses FMA and ALU pipes only.
// Inputs are clamped to >= -125 so the exponent field never underflows; the
// result there is 2^-125, negligible against a softmax row whose largest term
// is >= 1.
#pragma once

#include <cstdint>

namespace fa {

constexpr float kExp2C0 = 0x1.fff692p-1f;  // 0.999928057
constexpr float kExp2C1 = 0x1.62f31ap-1f;  // 0.693260968
constexpr float kExp2C2 = 0x1.f0de1ap-3f;  // 0.242611125
constexpr float kExp2C3 = 0x1.c3f76p-5f;   // 0.0551716685

__device__ __forceinline__ float ex2_poly(float x) {
  x = fmaxf(x, -125.0f);
  const float kShift = 12582912.0f;  // 1.5 * 2^23
  const float y = __fadd_rn(x, kShift);
  const float n = __fsub_rn(y, kShift);
  const float f = __fsub_rn(x, n);
  float p = __fmaf_rn(kExp2C3, f, kExp2C2);
  p = __fmaf_rn(p, f, kExp2C1);
  p = __fmaf_rn(p, f, kExp2C0);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(y) << 23));
}

// The same steps for two inputs at once on the packed fp32 pipe: one packed
// instruction per add / FMA for both lanes (the clamp and the exponent add
// stay scalar).
__device__ __forceinline__ float2 ex2_poly2(float2 x) {
  x.x = fmaxf(x.x, -125.0f);
  x.y = fmaxf(x.y, -125.0f);
  const float2 y = __fadd2_rn(x, make_float2(12582912.0f, 12582912.0f));
  const float2 n = __fadd2_rn(y, make_float2(-12582912.0f, -12582912.0f));
  const float2 f = __ffma2_rn(n, make_float2(-1.0f, -1.0f), x);  // x - n, exact
  float2 p = __ffma2_rn(make_float2(kExp2C3, kExp2C3), f, make_float2(kExp2C2, kExp2C2));
  p = __ffma2_rn(p, f, make_float2(kExp2C1, kExp2C1));
  p = __ffma2_rn(p, f, make_float2(kExp2C0, kExp2C0));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(y.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(y.y) << 23)));
}

}  // namespace fa
