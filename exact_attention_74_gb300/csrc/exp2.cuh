// exp2.cuh -- the two ways the softmax stage takes 2^x.
//
// ex2_hw:    the hardware ex2 unit (MUFU), approximate, flush-to-zero.
// ex2_poly3: the FMA-pipe emulation of "論文解説: FlashAttention-4 —
//            Algorithm and Kernel Pipelining Co-Design for Asymmetric
//            Hardware Scaling", ソフトウェア指数関数エミュレーション:
//            2^x = 2^n * 2^f with n = floor(x), f = x - n in [0, 1), 2^f from
//            the printed cubic by Horner's rule, and n added to the exponent
//            field with an integer operation.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Valid for x <= 127; inputs below -126 return 2^-126 (x is clamped), so a
// masked score (-inf) yields a value that is negligible against any row sum.
__device__ __forceinline__ float ex2_poly3(float x) {
  x = fmaxf(x, -126.0f);
  // Adding 1.5 * 2^23 with rounding toward -inf leaves floor(x) in the low
  // mantissa bits of t (its unit in the last place is 1 there), so
  // bits(t) = 0x4B400000 + floor(x) and, shifted left by 23, exactly
  // floor(x) << 23 modulo 2^32.
  const float kShift = 12582912.0f;
  const float t = __fadd_rd(x, kShift);
  const float n = t - kShift;          // floor(x), exact
  const float f = x - n;               // [0, 1)
  const float p = fmaf(fmaf(fmaf(0.0771f, f, 0.2276f), f, 0.6951f), f, 1.0f);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(t) << 23));
}

}  // namespace fa
