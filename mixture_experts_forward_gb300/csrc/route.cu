// Router: softcapped softmax top-k, one warp per token.
//
// "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Baseline: 7
// kernels", item 1: softcapping (tanh) and softmax over the experts, then
// top-k by warp-shuffle reduction, one warp per token with E/32 values per
// lane.  Ties go to the lower expert id.  Selection uses the capped logits z
// (before exp), and the weights are the softmax over the selected experts.
//
// exp and tanh are not libdevice calls: they are evaluated by a fixed
// sequence of IEEE binary32 operations (round-to-nearest multiply, add,
// divide and fused multiply-add) so the result is the same on every device
// and on the host:
//   exp(x):  n = rint(x * log2e); r = fma(-n, ln2_hi, x); r = fma(-n, ln2_lo, r);
//            p = sum_{j<=7} r^j / j! by Horner with fma; exp = p * 2^n
//            (Cody & Waite argument reduction); x < -87 -> 0, x > 88 -> inf.
//   tanh(t): |t| < 0.5: a + (a*s)*q(s), s = a*a, q the odd Taylor series of
//            tanh to degree 17 by Horner in s; 0.5 <= |t| < 10:
//            1 - 2/(exp(2|t|) + 1); |t| >= 10: 1; sign of t restored.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxPerLane = 32;  // E <= 1024

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

__device__ __forceinline__ float tanh_ieee(float t) {
  float a = fabsf(t);
  float y;
  if (a >= 10.0f) {
    y = 1.0f;
  } else if (a < 0.5f) {
    float s = __fmul_rn(a, a);
    // tanh Taylor coefficients of t^17 down to t^3
    float q = f32_bits(0x3a1aac12u);
    q = __fmaf_rn(q, s, f32_bits(0xbabed1b2u));
    q = __fmaf_rn(q, s, f32_bits(0x3b6b69e8u));
    q = __fmaf_rn(q, s, f32_bits(0xbc11371bu));
    q = __fmaf_rn(q, s, f32_bits(0x3cb327a4u));
    q = __fmaf_rn(q, s, f32_bits(0xbd5d0dd1u));
    q = __fmaf_rn(q, s, f32_bits(0x3e088889u));
    q = __fmaf_rn(q, s, f32_bits(0xbeaaaaabu));
    y = __fmaf_rn(__fmul_rn(a, s), q, a);
  } else {
    float e = exp_ieee(__fadd_rn(a, a));
    y = __fsub_rn(1.0f, __fdiv_rn(2.0f, __fadd_rn(e, 1.0f)));
  }
  return signbit(t) ? -y : y;
}

// (value desc, id asc) ordering
__device__ __forceinline__ bool better(float za, int ia, float zb, int ib) {
  return za > zb || (za == zb && ia < ib);
}

__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int M,
                                                    int E, int k, float softcap, int renorm,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ weights) {
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (t >= M) return;
  const float* row = logits + static_cast<size_t>(t) * E;
  const int per_lane = (E + 31) >> 5;

  float z[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    int e = lane + 32 * i;
    float v = -__int_as_float(0x7f800000);
    if (i < per_lane && e < E) {
      v = __ldg(row + e);
      if (softcap > 0.0f) v = __fmul_rn(softcap, tanh_ieee(__fdiv_rn(v, softcap)));
    }
    z[i] = v;
  }

  uint32_t taken = 0;
  float my_z = 0.0f;  // lane j keeps the j-th selected value
  int my_id = 0;
  float z0 = 0.0f;
  for (int j = 0; j < k; ++j) {
    float bz = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      int e = lane + 32 * i;
      if (i < per_lane && e < E && !((taken >> i) & 1u) && better(z[i], e, bz, bi)) {
        bz = z[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float oz = __shfl_xor_sync(0xffffffffu, bz, off);
      int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(oz, oi, bz, bi)) {
        bz = oz;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_z = bz;
      my_id = bi;
    }
    if (j == 0) z0 = bz;
  }

  float my_e = 0.0f;
  if (lane < k) my_e = exp_ieee(__fsub_rn(my_z, z0));
  float s = 0.0f;
  if (renorm) {
    for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, my_e, j));
  } else {
    // sum over all experts in expert-id order
    for (int e = 0; e < E; ++e) {
      float mine = 0.0f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (i == (e >> 5)) mine = z[i];
      float ze = __shfl_sync(0xffffffffu, mine, e & 31);
      s = __fadd_rn(s, exp_ieee(__fsub_rn(ze, z0)));
    }
  }
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_id;
    weights[static_cast<size_t>(t) * k + lane] = __fdiv_rn(my_e, s);
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                         int32_t* ids, float* weights, cudaStream_t stream, bool pdl) {
  const int warps = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + warps - 1) / warps);
  cfg.blockDim = dim3(32 * warps);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel, logits, M, E, k, softcap, renorm, ids, weights);
}

}  // namespace moe
