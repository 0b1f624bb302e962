// Quantise + sort/gather ("QSG").
//
// "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Baseline: 7
// kernels" item 4 (per 1x128 block: amax, scale = amax/448, element-wise
// E4M3 quantisation) and section "Fusion 2" (one pass quantises a token and
// copies its codes and scales to every routed slot), with the refinements of
// sections "QSG scatter vectorisation" (16-byte stores), "QSG load
// pipelining" (all loads issued before the reductions) and "Fused Memset"
// (the output accumulator is zeroed in the same pass).
//
// Layout: G = K/16 threads per token; thread c owns elements [16c, 16c+16):
// two 16-byte bf16 loads, one 16-byte E4M3 store per slot.  The 8 threads of a
// 128-element block are consecutive lanes, so amax is a 3-step xor shuffle.
// Arithmetic is IEEE binary32: s = amax / 448, inv = 1 / s, q = cvt.rn.satfinite
// (x * inv); amax == 0 gives s = 0 and all-zero codes.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(1024) quant_gather_kernel(
    const __nv_bfloat16* __restrict__ x, int M, int K, int k, const int32_t* __restrict__ route_slot,
    uint8_t* __restrict__ a_q, float* __restrict__ a_scales, float* __restrict__ zero_acc,
    int zero_cols) {
  const int G = K >> 4;                            // threads per token
  const int tpc = max(1, static_cast<int>(blockDim.x) / G);  // tokens per CTA
  const int t = blockIdx.x * tpc + threadIdx.x / G;
  const int c = threadIdx.x % G;
  const int R = M * k;
  // Idle threads (past the last token) still take part in the shuffles.
  const bool valid = threadIdx.x < tpc * G && t < M;

  // let the grouped GEMM's CTAs start their setup now; they wait for this grid
  pdl_launch_dependents();
  pdl_wait();

  if (valid && zero_acc != nullptr) {
    float4* row = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t) * zero_cols);
    for (int i = c; i < (zero_cols >> 2); i += G) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  uint4 raw0 = make_uint4(0u, 0u, 0u, 0u), raw1 = raw0;
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * K + 16 * c);
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
  // the 8 threads of one 128-element block are lanes l, l^1, l^2, l^4
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  if (!valid) return;

  uint4 q = make_uint4(0u, 0u, 0u, 0u);
  float s = 0.0f;
  if (amax > 0.0f) {
    s = __fdiv_rn(amax, 448.0f);
    const float inv = __fdiv_rn(1.0f, s);
    uint32_t words[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // byte i of the store is the code of element i
      uint16_t c01 = cvt_e4m3x2(__fmul_rn(v[4 * w + 0], inv), __fmul_rn(v[4 * w + 1], inv));
      uint16_t c23 = cvt_e4m3x2(__fmul_rn(v[4 * w + 2], inv), __fmul_rn(v[4 * w + 3], inv));
      words[w] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
    }
    q = make_uint4(words[0], words[1], words[2], words[3]);
  }

  const int b = c >> 3;  // 128-element block of this thread
  for (int j = 0; j < k; ++j) {
    const int slot = __ldg(route_slot + static_cast<size_t>(t) * k + j);
    if (slot < 0 || slot >= R) continue;
    *reinterpret_cast<uint4*>(a_q + static_cast<size_t>(slot) * K + 16 * c) = q;
    if ((c & 7) == 0) a_scales[static_cast<size_t>(b) * R + slot] = s;
  }
}

}  // namespace

cudaError_t launch_quant_gather(const void* x, int M, int K, int k, const int32_t* route_slot,
                                uint8_t* a_q, float* a_scales, float* zero_acc, int zero_cols,
                                cudaStream_t stream, bool pdl) {
  const int G = K / 16;
  int threads, tpc;
  if (G <= 256) {
    threads = 256;
    tpc = 256 / G;
  } else {
    threads = (G + 31) / 32 * 32;  // K <= 16384
    tpc = 1;
  }
  cudaError_t err = prefer_max_shared(quant_gather_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + tpc - 1) / tpc);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_gather_kernel, static_cast<const __nv_bfloat16*>(x), M, K,
                            k, route_slot, a_q, a_scales, zero_acc, zero_cols);
}

}  // namespace moe
