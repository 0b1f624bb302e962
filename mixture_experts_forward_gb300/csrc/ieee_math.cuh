// exp evaluated by a fixed sequence of IEEE binary32 operations (round-to-
// nearest multiply and fused multiply-add), so its result is the same on every
// device and matches a host restatement of the same steps bit for bit; shared
// by the router (softmax weights, softcap tanh) and the SwiGLU of the FP8
// gated FFN.  Not a libdevice call:
//   n = rint(x * log2e); r = fma(-n, ln2_hi, x); r = fma(-n, ln2_lo, r);
//   p = sum_{j<=7} r^j / j! by Horner with fma; exp = p * 2^n
//   (Cody & Waite argument reduction); x < -87 -> 0, x > 88 -> +inf.
#pragma once

#include <cstdint>

namespace moe {

__device__ __forceinline__ float f32_bits(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float exp_ieee(float x) {
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return __int_as_float(0x7f800000);
  const float log2e = f32_bits(0x3fb8aa3bu);
  const float ln2_hi = f32_bits(0x3f317218u);
  const float ln2_lo = f32_bits(0xb102e308u);
  float n = rintf(__fmul_rn(x, log2e));
  float r = __fmaf_rn(-n, ln2_hi, x);
  r = __fmaf_rn(-n, ln2_lo, r);
  // 1/j!, j = 7 down to 0
  float p = f32_bits(0x39500d01u);
  p = __fmaf_rn(p, r, f32_bits(0x3ab60b61u));
  p = __fmaf_rn(p, r, f32_bits(0x3c088889u));
  p = __fmaf_rn(p, r, f32_bits(0x3d2aaaabu));
  p = __fmaf_rn(p, r, f32_bits(0x3e2aaaabu));
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  int ni = static_cast<int>(n);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

}  // namespace moe
