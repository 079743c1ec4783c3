// FP8 (e4m3) quantisation helpers: UE8M0 (power-of-two) scales per group of
// 128 values.
//
// SGLang chapter 17, section "prefll 侧的一个必要步骤:per-token-group 量化":
// hidden states are quantised in groups of 128 consecutive features of one
// token, with UE8M0 scale factors for a 1x128 fine-grained-scaled GEMM.
// A group's scale is the smallest power of two 2^e with amax <= 448 * 2^e
// (448 is the largest e4m3 value; e = 0 for an all-zero group), stored as the
// byte e + 127; each value becomes e4m3(x / 2^e), rounded to nearest with ties
// to even and saturating at +-448.
#pragma once

#include <stdint.h>

namespace moe {

// Exact 2^n for n in [-149, 127].
__device__ __forceinline__ float pow2i(int n) {
  return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(1 << (n + 149));
}

// Scale exponent of a group with largest magnitude amax (see above), clamped
// to [-127, 127].  amax = f * 2^E with f in [0.5, 1) and 448 = 0.875 * 2^9.
__device__ __forceinline__ int fp8_scale_exp(float amax) {
  if (!(amax > 0.0f)) return 0;
  int E;
  const float f = frexpf(amax, &E);
  int e = E - 9 + (f > 0.875f ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Four values -> four e4m3 codes, first value in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  // the first source lands in the upper byte of each pair
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Largest magnitude over the 4 lanes of an aligned lane quad.
__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

}  // namespace moe
