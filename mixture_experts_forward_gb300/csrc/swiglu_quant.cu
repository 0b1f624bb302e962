// SwiGLU + FP8 re-quantisation between the two projections of the FP8 gated
// FFN: the two-layer expert MLP (gate+up projection, SiLU, down projection)
// that "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)" compares against in its
// closing section "Reference: vLLM full MLP", with both projections in the
// page's FP8 format ("Baseline: 7 kernels", item 6).
//
// The up projection stores gu (f32 [R, 2I]: gate columns [0, I), up columns
// [I, 2I)).  For every routed row s and 1x128 block b of h:
//   h = silu(g) * u = (g / (1 + exp(-g))) * u    (IEEE binary32 operations,
//       exp by the same fixed sequence as the router),
//   amax = max |h|, scale = amax / 448, q = E4M3_rn_satfinite(h * (1/scale))
//   (the 1x128 rule of item 4; amax = 0 gives scale 0 and zero codes),
// written as h_q (u8 [R, I]) and h_scales (f32 [I/128, R], block-major like
// the activations' scales) for the FP8 down projection.
//
// One warp per (row, block): each lane loads 4 gate and 4 up values (16-byte
// loads), the block amax is a warp max, each lane stores its 4 codes (one
// 128-byte line per warp) and lane 0 the block's scale.  Consecutive warps
// take consecutive rows of one block, so the block-major scale stores of a
// CTA are contiguous.  Bound by HBM: 8 bytes read and 1 + 4/128 written per
// element of h.
#include "ieee_math.cuh"
#include "moe_internal.cuh"
#include "quant_common.cuh"

namespace moe {
namespace {

constexpr int kSqWarps = 8;

__device__ __forceinline__ float swiglu_ieee(float g, float u) {
  const float e = exp_ieee(-g);              // 0 for g > 87, +inf for g < -88
  const float d = __fadd_rn(1.0f, e);
  return __fmul_rn(__fdiv_rn(g, d), u);      // g / +inf = -0 for very negative g
}

__global__ void __launch_bounds__(kSqWarps * 32)
    swiglu_quant_kernel(const float4* __restrict__ gu, int R, int I,
                        uint32_t* __restrict__ h_q, float* __restrict__ h_scales,
                        long long items) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long stride = static_cast<long long>(gridDim.x) * kSqWarps;
  const size_t row4 = static_cast<size_t>(I) / 2;   // float4s per gu row (2I floats)
  const size_t up4 = static_cast<size_t>(I) / 4;    // float4 offset of the up columns
  for (long long it = static_cast<long long>(blockIdx.x) * kSqWarps + (threadIdx.x >> 5);
       it < items; it += stride) {
    const int b = static_cast<int>(it / R);
    const int s = static_cast<int>(it - static_cast<long long>(b) * R);
    const size_t g4 = static_cast<size_t>(s) * row4 + static_cast<size_t>(b) * 32 + lane;
    const float4 g = __ldcs(gu + g4);
    const float4 u = __ldcs(gu + g4 + up4);
    const float h0 = swiglu_ieee(g.x, u.x), h1 = swiglu_ieee(g.y, u.y);
    const float h2 = swiglu_ieee(g.z, u.z), h3 = swiglu_ieee(g.w, u.w);
    float amax = fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint32_t codes = 0u;
    float scale = 0.0f;
    if (amax > 0.0f) {
      scale = __fdiv_rn(amax, 448.0f);
      const float inv = __fdiv_rn(1.0f, scale);
      const uint32_t c01 = cvt_e4m3x2(__fmul_rn(h0, inv), __fmul_rn(h1, inv));
      const uint32_t c23 = cvt_e4m3x2(__fmul_rn(h2, inv), __fmul_rn(h3, inv));
      codes = c01 | (c23 << 16);
    }
    h_q[static_cast<size_t>(s) * (I / 4) + static_cast<size_t>(b) * 32 + lane] = codes;
    if (lane == 0) h_scales[static_cast<size_t>(b) * R + s] = scale;
  }
}

}  // namespace

cudaError_t launch_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales,
                                int num_sms, cudaStream_t stream, bool pdl) {
  const long long items = static_cast<long long>(R) * (I / 128);
  long long blocks = (items + kSqWarps - 1) / kSqWarps;
  const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t err = prefer_max_shared(swiglu_quant_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      make_cfg(dim3(static_cast<unsigned>(blocks)), dim3(kSqWarps * 32), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, swiglu_quant_kernel, reinterpret_cast<const float4*>(gu), R, I,
                            reinterpret_cast<uint32_t*>(h_q), h_scales, items);
}

}  // namespace moe
