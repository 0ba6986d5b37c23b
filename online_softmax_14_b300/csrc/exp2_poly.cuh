// 2^x on the FMA pipe, two values at a time, for the part of the softmax
// exponentials that the kernels take off the special-function unit.
//
// Method: Cody and Waite's range reduction ("Software Manual for the Elementary
// Functions", 1980): x = n + f with n = round(x) and f = x - n in [-1/2, 1/2], so
// 2^x = 2^n * 2^f.  2^f is a degree-3 polynomial, the minimax fit of the relative
// error on [-1/2, 1/2] found by the Remez exchange in exp2_poly_fit.py (relative
// error below 7.5e-5 before float32 rounding; a probability then goes to bfloat16,
// whose rounding alone is up to 2^-9 = 2e-3).  2^n is built directly as the float
// whose exponent field is n + 127.
//
// Range: x is clamped below at -127, where 2^n's exponent field is 0, so every
// x <= -127 (and -inf, a masked score) gives exactly 0, as ex2.approx.ftz does
// for results below 2^-126.  x must be below 128.
#pragma once
#include "ptx.cuh"

namespace fa {

// p(f) = C0 + C1 f + C2 f^2 + C3 f^3 ~ 2^f on [-1/2, 1/2] (float32 values of the fit)
constexpr float kExp2C0 = 0x1.fff692p-1f;
constexpr float kExp2C1 = 0x1.62f31ap-1f;
constexpr float kExp2C2 = 0x1.f0de1ap-3f;
constexpr float kExp2C3 = 0x1.c3f76p-5f;
// 1.5 * 2^23: adding it rounds a float of magnitude < 2^22 to an integer held in
// the low mantissa bits (round to nearest even).
constexpr float kRoundMagic = 12582912.0f;

__device__ __forceinline__ uint64_t f2_add_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// (2^x0, 2^x1) for the packed pair x2 = (x0, x1).
__device__ __forceinline__ uint64_t exp2_fma2(uint64_t x2) {
  float x0, x1;
  f2_unpack(x2, x0, x1);
  const uint64_t x = f2_pack(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
  const uint64_t magic = f2_pack(kRoundMagic, kRoundMagic);
  const uint64_t t = f2_add_rn(x, magic);            // n in the low mantissa bits
  const uint64_t f = f2_sub_rn(x, f2_sub_rn(t, magic));  // x - n, exact
  uint64_t p = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  p = f2_fma(p, f, f2_pack(kExp2C1, kExp2C1));
  p = f2_fma(p, f, f2_pack(kExp2C0, kExp2C0));
  float t0, t1;
  f2_unpack(t, t0, t1);
  // (bits(t) + 127) << 23 is (n + 127) << 23: the high bits of t shift out
  const uint32_t e0 = (__float_as_uint(t0) + 127u) << 23, e1 = (__float_as_uint(t1) + 127u) << 23;
  return f2_mul(p, f2_pack(__uint_as_float(e0), __uint_as_float(e1)));
}

}  // namespace fa
