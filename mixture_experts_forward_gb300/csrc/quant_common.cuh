// Blockwise E4M3 quantisation of 16 consecutive bf16 elements per thread,
// shared by the standalone quantise+gather kernel and the fused routing
// kernel.  "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Baseline:
// 7 kernels" item 4: per 1x128 block amax, scale = amax/448, element-wise
// E4M3; IEEE binary32 arithmetic (s = amax / 448, inv = 1 / s,
// q = cvt.rn.satfinite(x * inv)); amax == 0 gives s = 0 and all-zero codes.
#pragma once

#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantises elements [16c, 16c+16) of `row` (bf16).  The 8 threads of one
// 128-element block must be lanes l, l^1, l^2, l^4 of the same warp, and every
// lane of the warp must call this (invalid lanes pass valid = false).
// Returns the 16 codes (byte i = code of element 16c+i) and the block scale.
__device__ __forceinline__ void quantize16(const __nv_bfloat16* row, int c, bool valid, uint4& q,
                                           float& scale) {
  uint4 raw0 = make_uint4(0u, 0u, 0u, 0u), raw1 = raw0;
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(row + 16 * c);
    raw0 = __ldg(src);
    raw1 = __ldg(src + 1);
  }
  float v[16];
  {
    const uint32_t w[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);              // element 2i (low half)
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);  // element 2i+1
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  q = make_uint4(0u, 0u, 0u, 0u);
  scale = 0.0f;
  if (amax > 0.0f) {
    scale = __fdiv_rn(amax, 448.0f);
    const float inv = __fdiv_rn(1.0f, scale);
    uint32_t words[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint16_t c01 = cvt_e4m3x2(__fmul_rn(v[4 * w + 0], inv), __fmul_rn(v[4 * w + 1], inv));
      const uint16_t c23 = cvt_e4m3x2(__fmul_rn(v[4 * w + 2], inv), __fmul_rn(v[4 * w + 3], inv));
      words[w] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
    }
    q = make_uint4(words[0], words[1], words[2], words[3]);
  }
}

}  // namespace moe
