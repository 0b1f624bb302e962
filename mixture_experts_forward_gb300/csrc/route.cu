// Router: softcapped softmax top-k, one warp per token.
//
// "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Baseline: 7
// kernels", item 1: softcapping (tanh) and softmax over the experts, then
// top-k by warp-shuffle reduction, one warp per token with E/32 values per
// lane.  Ties go to the lower expert id.  Selection uses the capped logits z
// (before exp), and the weights are the softmax over the selected experts.
// Each lane keeps its best remaining expert; a selection round is one
// warp-wide max over order-preserving keys (redux.sync), one min over the
// ids that hold it, and a rescan by the winning lane only.
//
// exp and tanh are not libdevice calls: they are evaluated by a fixed
// sequence of IEEE binary32 operations (round-to-nearest multiply, add,
// divide and fused multiply-add) so the result is the same on every device
// and on the host:
//   exp(x):  exp_ieee (ieee_math.cuh): Cody & Waite reduction, degree-7 Taylor.
//   tanh(t): |t| < 0.5: a + (a*s)*q(s), s = a*a, q the odd Taylor series of
//            tanh to degree 17 by Horner in s; 0.5 <= |t| < 10:
//            1 - 2/(exp(2|t|) + 1); |t| >= 10: 1; sign of t restored.
#include "ieee_math.cuh"
#include "layout_block.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

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

// Order-preserving map of a binary32 value to an unsigned key: larger value,
// larger key.  -0.0 is first made +0.0 so that the two zeros tie (and the
// lower expert id wins), as they do under floating-point comparison.
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t u = __float_as_uint(z == 0.0f ? 0.0f : z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Routes one token with one warp.  NPL = experts per lane (E <= 32 * NPL);
// lane l owns experts l, l+32, ...
template <int NPL>
__device__ __forceinline__ int route_token(const float* __restrict__ row, int E, int k,
                                           float softcap, int renorm, int32_t* __restrict__ ids,
                                           float* __restrict__ weights) {
  const int lane = threadIdx.x & 31;
  float z[NPL];
  uint32_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    z[i] = e < E ? __ldg(row + e) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (softcap > 0.0f) z[i] = __fmul_rn(softcap, tanh_ieee(__fdiv_rn(z[i], softcap)));
    key[i] = e < E ? order_key(z[i]) : 0u;  // key 0: below every real value
  }

  // this lane's best remaining expert (largest key; the first one wins ties,
  // which is the lowest id because ids grow with i)
  uint32_t hk = 0u;
  int hi = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (key[i] > hk) {
      hk = key[i];
      hi = i;
    }

  float my_z = 0.0f;  // lane j keeps the j-th selected value and id
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t best = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t cand =
        (hk == best && best != 0u) ? static_cast<uint32_t>(lane + 32 * hi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    const int owner = static_cast<int>(win & 31u);
    float zv = 0.0f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i == hi) zv = z[i];
    zv = __shfl_sync(0xffffffffu, zv, owner);
    if (lane == j) {
      my_z = zv;
      my_id = static_cast<int>(win);
    }
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (i == hi) key[i] = 0u;
      hk = 0u;
      hi = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (key[i] > hk) {
          hk = key[i];
          hi = i;
        }
    }
  }
  const float z0 = __shfl_sync(0xffffffffu, my_z, 0);

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
      for (int i = 0; i < NPL; ++i)
        if (i == (e >> 5)) mine = z[i];
      const float ze = __shfl_sync(0xffffffffu, mine, e & 31);
      s = __fadd_rn(s, exp_ieee(__fsub_rn(ze, z0)));
    }
  }
  if (lane < k) {
    ids[lane] = my_id;
    weights[lane] = __fdiv_rn(my_e, s);
  }
  return my_id;  // lane j < k: the j-th selected expert
}

template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int M,
                                                    int E, int k, float softcap, int renorm,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ weights) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= M) return;
  route_token<NPL>(logits + static_cast<size_t>(t) * E, E, k, softcap, renorm,
                   ids + static_cast<size_t>(t) * k, weights + static_cast<size_t>(t) * k);
}

// Large batches: route + per-CTA ranking, and in the last CTA the expert
// offsets.  Every CTA routes 32 tokens (a warp each).  The k experts of one
// token are distinct, so the rank of route (t, j) among this CTA's routes to
// its expert e is the number of earlier tokens of the CTA that chose e: a
// per-warp 0/1 row of a [32][E] shared table, prefix-summed over the warps.
// The CTA publishes its per-expert totals (cta_hist[cta][E]) and the ranks
// (local_rank[R]), then takes an arrival number from an acq_rel counter.  The
// last S = ceil(E / 32) CTAs to arrive scan the totals, each for its own
// block of up to 32 experts: they wait (bounded) until every CTA has arrived —
// the others have all finished or are still running, so the wait ends — and
// turn their experts' columns into per-CTA bases (cta_base[cta][E], exclusive
// over the CTAs) and counts.  The last of them to finish (a second counter)
// scans the counts over the experts into offsets and tile offsets.  The
// quantise/gather kernel then places route r of expert e at
// offsets[e] + cta_base[cta(r)][e] + local_rank[r] — the stable layout by
// route id.
// Bound on the scanning CTAs' wait for the other CTAs' totals.
constexpr uint64_t kScanWaitNs = 2000000000ull;

// Two CTAs per SM where E is small (the router keeps few registers);
// 32-token groups with many experts keep one CTA per SM and 64 registers.
template <int NPL>
__global__ void __launch_bounds__(kLayoutThreads, NPL <= 4 ? 2 : 1)
    route_rank_kernel(const float* __restrict__ logits, int M, int E, int k, float softcap,
                      int renorm, int32_t* ids, float* __restrict__ weights, int block_m,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ tile_offsets, Ctrl* ctrl, int32_t* local_rank,
                      int32_t* cta_hist, int32_t* __restrict__ cta_base) {
  extern __shared__ int s_tab[];  // [32][E] ranking table (at least 1024 ints: the scanners' [32][32] sums)
  __shared__ int s_last;
  __shared__ int s_wa[32], s_wb[32];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int t = blockIdx.x * 32 + w;
  int e_sel = -1;
  if (t < M) {
    const int id = route_token<NPL>(logits + static_cast<size_t>(t) * E, E, k, softcap, renorm,
                                    ids + static_cast<size_t>(t) * k,
                                    weights + static_cast<size_t>(t) * k);
    if (lane < k) e_sel = id;
  }
  for (int i = tid; i < 32 * E; i += kLayoutThreads) s_tab[i] = 0;
  __syncthreads();
  if (e_sel >= 0) s_tab[w * E + e_sel] = 1;
  __syncthreads();
  for (int e = tid; e < E; e += kLayoutThreads) {
    int run = 0;
    for (int ww = 0; ww < 32; ++ww) {
      const int v = s_tab[ww * E + e];
      s_tab[ww * E + e] = run;
      run += v;
    }
    cta_hist[static_cast<size_t>(blockIdx.x) * E + e] = run;
  }
  __syncthreads();
  if (e_sel >= 0) local_rank[static_cast<size_t>(t) * k + lane] = s_tab[w * E + e_sel];
  __syncthreads();
  if (tid == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(&ctrl->route_done)
                 : "memory");
    s_last = static_cast<int>(prev);  // arrival number
  }
  __syncthreads();
  const int nC = gridDim.x;
  const int S = min(nC, (E + 31) / 32);  // column-scanning CTAs
  const int scan = s_last - (nC - S);    // this CTA's scanner index, or < 0
  if (scan < 0) return;

  // ---- scanners: wait until every CTA has published its totals
  if (tid == 0) {
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&ctrl->route_done) : "memory");
      if (v >= static_cast<unsigned>(nC)) break;
      if (global_timer_ns() - t0 > kScanWaitNs) { ok = 0; break; }
      __nanosleep(64);
    }
    if (!ok) set_error(ctrl, MOE_ERR_TIMEOUT, 6);
    s_wa[0] = ok;
  }
  __syncthreads();
  if (!s_wa[0]) return;

  // Experts [e0, e1) of this scanner, 32 at a time: lane = expert, warp w
  // takes a contiguous run of CTAs (rows) and sums it; the exclusive prefix
  // of the run sums over the warps gives each run's start; a second pass over
  // the run writes the bases.  Row loads are 128-byte coalesced.
  const int per = (E + S - 1) / S;
  const int e0 = scan * per, e1 = min(E, e0 + per);
  const int L = (nC + 31) / 32;  // rows per warp
  const int r0 = min(nC, w * L), r1 = min(nC, r0 + L);
  int* s_sum = s_tab;            // [32 warps][32 lanes]
  for (int eb = e0; eb < e1; eb += 32) {
    const int e = eb + lane;
    const bool act = e < e1;
    int part = 0;
    if (act)
      for (int r = r0; r < r1; ++r) part += __ldcg(cta_hist + static_cast<size_t>(r) * E + e);
    s_sum[w * 32 + lane] = part;
    __syncthreads();
    int run = 0;
    for (int ww = 0; ww < w; ++ww) run += s_sum[ww * 32 + lane];
    if (act) {
      for (int r = r0; r < r1; ++r) {
        const int v = __ldcg(cta_hist + static_cast<size_t>(r) * E + e);
        cta_base[static_cast<size_t>(r) * E + e] = run;
        run += v;
      }
      if (w == 31) counts[e] = run;  // warp 31 holds the column total
    }
    __syncthreads();
  }

  // ---- the last scanner: offsets and tile offsets over all experts
  __syncthreads();
  if (tid == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(&ctrl->scan_done)
                 : "memory");
    s_last = prev == static_cast<unsigned>(S - 1);
  }
  __syncthreads();
  if (!s_last) return;
  int cnt = 0, ntile = 0;
  if (tid < E) {
    cnt = __ldcg(counts + tid);
    ntile = (cnt + block_m - 1) / block_m;
  }
  int inc_c = cnt, inc_t = ntile;
  block_scan2(inc_c, inc_t, s_wa, s_wb);
  if (tid < E) {
    offsets[tid] = inc_c - cnt;
    tile_offsets[tid] = inc_t - ntile;
    if (tid == E - 1) {
      offsets[E] = inc_c;
      tile_offsets[E] = inc_t;
    }
  }
  if (tid == 0) {
    ctrl->queue = 0;
    ctrl->done = 0;
    ctrl->queue2 = 0;
    ctrl->done2 = 0;
    ctrl->route_done = 0u;
    ctrl->scan_done = 0u;
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                         int32_t* ids, float* weights, cudaStream_t stream, bool pdl) {
  const int warps = 8;
  cudaError_t err = prefer_max_shared(route_kernel<1>);
  if (err == cudaSuccess) err = prefer_max_shared(route_kernel<2>);
  if (err == cudaSuccess) err = prefer_max_shared(route_kernel<4>);
  if (err == cudaSuccess) err = prefer_max_shared(route_kernel<8>);
  if (err == cudaSuccess) err = prefer_max_shared(route_kernel<16>);
  if (err == cudaSuccess) err = prefer_max_shared(route_kernel<32>);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + warps - 1) / warps);
  cfg.blockDim = dim3(32 * warps);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int npl = (E + 31) / 32;
  if (npl <= 1) return cudaLaunchKernelEx(&cfg, route_kernel<1>, logits, M, E, k, softcap, renorm, ids, weights);
  if (npl <= 2) return cudaLaunchKernelEx(&cfg, route_kernel<2>, logits, M, E, k, softcap, renorm, ids, weights);
  if (npl <= 4) return cudaLaunchKernelEx(&cfg, route_kernel<4>, logits, M, E, k, softcap, renorm, ids, weights);
  if (npl <= 8) return cudaLaunchKernelEx(&cfg, route_kernel<8>, logits, M, E, k, softcap, renorm, ids, weights);
  if (npl <= 16) return cudaLaunchKernelEx(&cfg, route_kernel<16>, logits, M, E, k, softcap, renorm, ids, weights);
  return cudaLaunchKernelEx(&cfg, route_kernel<32>, logits, M, E, k, softcap, renorm, ids, weights);
}


template <int NPL>
cudaError_t launch_route_rank_t(const float* logits, int M, int E, int k, float softcap,
                                int renorm, int32_t* ids, float* weights, int block_m,
                                int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                                Ctrl* ctrl, int32_t* local_rank, int32_t* cta_hist,
                                int32_t* cta_base, cudaStream_t stream, bool pdl) {
  // [32][E] ranking table; the scanning CTAs reuse it for [32][32] run sums
  const int n_ctas = (M + 31) / 32;
  const int ints = 32 * E > 1024 ? 32 * E : 1024;
  const size_t smem = static_cast<size_t>(ints) * sizeof(int);
  cudaError_t err = cudaFuncSetAttribute(route_rank_kernel<NPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err == cudaSuccess) err = prefer_max_shared(route_rank_kernel<NPL>);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(kLayoutThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_rank_kernel<NPL>, logits, M, E, k, softcap, renorm, ids,
                            weights, block_m, counts, offsets, tile_offsets, ctrl, local_rank,
                            cta_hist, cta_base);
}

cudaError_t launch_route_rank(const float* logits, int M, int E, int k, float softcap, int renorm,
                              int32_t* ids, float* weights, int block_m, int32_t* counts,
                              int32_t* offsets, int32_t* tile_offsets, Ctrl* ctrl,
                              int32_t* local_rank, int32_t* cta_hist, int32_t* cta_base,
                              cudaStream_t stream, bool pdl) {
  const int npl = (E + 31) / 32;
#define MOE_RR(N)                                                                           \
  return launch_route_rank_t<N>(logits, M, E, k, softcap, renorm, ids, weights, block_m,    \
                                counts, offsets, tile_offsets, ctrl, local_rank, cta_hist,  \
                                cta_base, stream, pdl)
  if (npl <= 1) MOE_RR(1);
  if (npl <= 2) MOE_RR(2);
  if (npl <= 4) MOE_RR(4);
  if (npl <= 8) MOE_RR(8);
  if (npl <= 16) MOE_RR(16);
  MOE_RR(32);
#undef MOE_RR
}


}  // namespace moe
