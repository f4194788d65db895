// Exponential helpers of the softmax in the exp2 domain: the SFU's
// ex2.approx, a three-input max, and a polynomial 2^x on the FMA pipes (used
// for part of the exponentials so that the SFU is not the only unit doing
// them).
#pragma once

#include "common.cuh"

namespace pkv {

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x for a pair of floats, on the FMA/ALU pipes, for x <= 8 (the
// softmax's stale-max bound).  Method: Cody-Waite style range reduction,
// x = n + f with n = round-to-nearest(x) (adding and subtracting 1.5 * 2^23
// rounds a float to an integer) and f in [-1/2, 1/2]; 2^f from a cubic in
// f, evaluated by Horner's rule, whose coefficients were fitted to keep the
// relative error on [-1/2, 1/2] below 2.2e-4 (the largest error sits at
// f = +1/2; bf16 P resolves 2^-8); n is added to the exponent field.  x is
// clamped at -125 so that the result stays a normal float: a masked, -inf
// score gives about 2^-125 instead of 0, below 2^-100 of the row sum, which
// holds at least one term >= 2^-8.
__device__ __forceinline__ uint64_t poly_exp2x2(uint64_t x) {
  float x0, x1;
  f2_split(x, x0, x1);
  const uint64_t xc = f2(fmaxf(x0, -125.f), fmaxf(x1, -125.f));
  const uint64_t kMagic = f2(12582912.f, 12582912.f);  // 1.5 * 2^23
  const uint64_t tt = f2_add(xc, kMagic);
  const uint64_t f = f2_sub(xc, f2_sub(tt, kMagic));
  uint64_t p = f2_fma(f2(0.05286737531423569f, 0.05286737531423569f), f,
                      f2(0.24215202033519745f, 0.24215202033519745f));
  p = f2_fma(p, f, f2(0.6935867667198181f, 0.6935867667198181f));
  p = f2_fma(p, f, f2(0.9999627470970154f, 0.9999627470970154f));
  float t0, t1, p0, p1;
  f2_split(tt, t0, t1);
  f2_split(p, p0, p1);
  const int n0 = __float_as_int(t0) - 0x4B400000;
  const int n1 = __float_as_int(t1) - 0x4B400000;
  return f2(__int_as_float(__float_as_int(p0) + (n0 << 23)),
            __int_as_float(__float_as_int(p1) + (n1 << 23)));
}

}  // namespace pkv
