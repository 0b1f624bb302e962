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
#include "moe_internal.cuh"
#include "quant_common.cuh"

namespace moe {
namespace {

// Slot of route r (see Placement); writes route_slot / sorted_route_ids when placing.
__device__ __forceinline__ int route_slot_of(int r, int t, const int32_t* route_slot_in,
                                             int32_t* route_slot, const Placement& pl, int R) {
  if (pl.cta_base == nullptr) return __ldg(route_slot_in + r);
  const int e = __ldg(pl.ids + r);
  if (e < 0 || e >= pl.E) return -1;
  const int slot = __ldg(pl.offsets + e) +
                   __ldg(pl.cta_base + static_cast<size_t>(t / kRankTokensPerCta) * pl.E + e) +
                   __ldg(pl.local_rank + r);
  if (slot < 0 || slot >= R) return -1;
  route_slot[r] = slot;
  pl.sorted_route_ids[slot] = r;
  return slot;
}

// token_major = 1 (the grouped GEMM gathers rows itself): each token's codes
// and scales are written once, token-major (a_q [M, K], a_scales [K/128, M]),
// before the wait for the router; after it the kernel only places the routes
// (route_slot, sorted_route_ids).
__global__ void __launch_bounds__(1024) quant_gather_kernel(
    const __nv_bfloat16* __restrict__ x, int M, int K, int k, int32_t* route_slot,
    uint8_t* __restrict__ a_q, float* __restrict__ a_scales, float* __restrict__ zero_acc,
    int zero_cols, const Placement pl, int token_major) {
  __shared__ int s_slot[1024];
  const int G = K >> 4;                            // threads per token
  const int tpc = max(1, static_cast<int>(blockDim.x) / G);  // tokens per CTA
  const int lt = static_cast<int>(threadIdx.x) / G;
  const int t = blockIdx.x * tpc + lt;
  const int c = threadIdx.x % G;
  const int R = M * k;
  // Idle threads (past the last token) still take part in the shuffles.
  const bool valid = threadIdx.x < tpc * G && t < M;

  // let the grouped GEMM's CTAs start their setup now; they wait for this grid
  pdl_launch_dependents();
  // x does not depend on the previous kernel: clear the accumulator rows and
  // quantise before waiting for it
  if (valid && zero_acc != nullptr) {
    float4* row = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t) * zero_cols);
    for (int i = c; i < (zero_cols >> 2); i += G) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint4 q;
  float s;
  quantize16(x + static_cast<size_t>(valid ? t : 0) * K, c, valid, q, s);
  if (token_major) {
    if (valid) {
      *reinterpret_cast<uint4*>(a_q + static_cast<size_t>(t) * K + 16 * c) = q;
      if ((c & 7) == 0) a_scales[static_cast<size_t>(c >> 3) * M + t] = s;
    }
    pdl_wait();
    // a token has G threads and top_k routes (top_k may exceed G): strided
    if (valid)
      for (int j = c; j < k; j += G) route_slot_of(t * k + j, t, route_slot, route_slot, pl, R);
    return;
  }
  pdl_wait();

  if (valid)
    for (int j = c; j < k; j += G)
      s_slot[lt * k + j] = route_slot_of(t * k + j, t, route_slot, route_slot, pl, R);
  __syncthreads();
  if (!valid) return;

  const int b = c >> 3;  // 128-element block of this thread
  for (int j = 0; j < k; ++j) {
    const int slot = s_slot[lt * k + j];
    if (slot < 0 || slot >= R) continue;
    *reinterpret_cast<uint4*>(a_q + static_cast<size_t>(slot) * K + 16 * c) = q;
    if ((c & 7) == 0) a_scales[static_cast<size_t>(b) * R + slot] = s;
  }
}

// Exclusive scan of v[0..n) in place over a CTA of any size (a multiple of
// 32, at most 1024 threads); each thread owns a contiguous run of entries.
// Returns the total.  s_tmp: 32 ints of shared memory.
__device__ int block_exclusive_scan(int* v, int n, int* s_tmp) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int b = min(n, static_cast<int>(threadIdx.x) * per), e = min(n, b + per);
  int local = 0;
  for (int i = b; i < e; ++i) local += v[i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) s_tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < static_cast<int>(blockDim.x >> 5) ? s_tmp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_tmp[lane] = w;  // inclusive totals of warps 0..lane
  }
  __syncthreads();
  int run = inc - local + (warp > 0 ? s_tmp[warp - 1] : 0);
  const int total = s_tmp[31];
  for (int i = b; i < e; ++i) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  __syncthreads();
  return total;
}

// Small-batch quantise + layout + gather ("QSG" with the layout folded in):
// each CTA quantises its tokens while the router still runs (x does not
// depend on routing; the wait for the router comes after), then loads every
// route's expert id into shared memory and finds its own routes' slots
// directly: slot(r) = #{routes with a smaller expert id} + #{earlier routes of
// the same expert} — the same stable layout the layout kernel builds, without
// a device-wide handoff.  One extra CTA (the last; it has no tokens) writes
// counts, offsets and tile offsets and re-zeroes the tile-queue counters.
// Used when M * top_k is small.
__global__ void __launch_bounds__(1024) quant_layout_kernel(
    const __nv_bfloat16* __restrict__ x, int M, int K, int k, int E, int block_m,
    const int32_t* __restrict__ ids, uint8_t* __restrict__ a_q, float* __restrict__ a_scales,
    float* __restrict__ zero_acc, int zero_cols, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_route_ids,
    int32_t* __restrict__ route_slot, int32_t* __restrict__ tile_offsets, Ctrl* ctrl) {
  extern __shared__ int s_dyn[];  // [R] ids, then [tpc*k] slots, then [E] counts (CTA 0)
  __shared__ int s_tmp[32];
  __shared__ int s_bad;
  const int G = K >> 4;
  const int tpc = max(1, static_cast<int>(blockDim.x) / G);
  const int t0 = blockIdx.x * tpc;
  const int t = t0 + static_cast<int>(threadIdx.x) / G;
  const int c = threadIdx.x % G;
  const int R = M * k;
  const bool valid = static_cast<int>(threadIdx.x) < tpc * G && t < M;
  int* s_ids = s_dyn;
  int* s_slot = s_dyn + R;
  int* s_cnt = s_slot + tpc * k;

  pdl_launch_dependents();
  // independent of the router: clear the accumulator rows, quantise the tokens
  if (valid && zero_acc != nullptr) {
    float4* row = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t) * zero_cols);
    for (int i = c; i < (zero_cols >> 2); i += G) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint4 q;
  float sc;
  quantize16(x + static_cast<size_t>(valid ? t : 0) * K, c, valid, q, sc);
  if (threadIdx.x == 0) s_bad = 0;

  pdl_wait();
  // all expert ids, every copy in flight before one wait
  if ((R & 3) == 0) {
    for (int i = 4 * threadIdx.x; i < R; i += 4 * blockDim.x) cp_async16(smem_u32(s_ids + i), ids + i);
  } else {
    for (int i = threadIdx.x; i < R; i += blockDim.x) cp_async4(smem_u32(s_ids + i), ids + i);
  }
  cp_async_wait_all();
  __syncthreads();

  // slots of this CTA's routes: one warp per route
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int nr = max(0, min(tpc, M - t0)) * k;
  for (int j = warp; j < nr; j += nwarps) {
    const int r = t0 * k + j;
    const int e = s_ids[r];
    int lt = 0, eq = 0;
    for (int i = lane; i < R; i += 32) {
      const int v = s_ids[i];
      lt += v < e;
      eq += (v == e) & (i < r);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lt += __shfl_xor_sync(0xffffffffu, lt, off);
      eq += __shfl_xor_sync(0xffffffffu, eq, off);
    }
    if (lane == 0) {
      int slot = lt + eq;
      if (e < 0 || e >= E) {
        slot = -1;
        s_bad = 1;
      } else {
        sorted_route_ids[slot] = r;
      }
      s_slot[j] = slot;
      route_slot[r] = slot;
    }
  }
  __syncthreads();

  if (valid) {
    const int b = c >> 3;
    for (int j = 0; j < k; ++j) {
      const int slot = s_slot[(t - t0) * k + j];
      if (slot < 0 || slot >= R) continue;
      *reinterpret_cast<uint4*>(a_q + static_cast<size_t>(slot) * K + 16 * c) = q;
      if ((c & 7) == 0) a_scales[static_cast<size_t>(b) * R + slot] = sc;
    }
  }
  if (threadIdx.x == 0 && s_bad) set_error(ctrl, MOE_ERR_DEVICE_FAULT, 2);

  if (blockIdx.x == gridDim.x - 1) {
    // counts, offsets and tile offsets of all experts (the extra CTA, in
    // parallel with the others' slot search)
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
    if (threadIdx.x == 0 && ctrl != nullptr) {
      ctrl->queue = 0;
      ctrl->done = 0;
      ctrl->queue2 = 0;
      ctrl->done2 = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
      const int e = s_ids[i];
      if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) counts[i] = s_cnt[i];
    __syncthreads();
    const int total = block_exclusive_scan(s_cnt, E, s_tmp);
    for (int i = threadIdx.x; i < E; i += blockDim.x) offsets[i] = s_cnt[i];
    if (threadIdx.x == 0) offsets[E] = total;
    // tiles per expert: recompute from the offsets (entries e and e+1)
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      const int cnt = (i + 1 < E ? s_cnt[i + 1] : total) - s_cnt[i];
      s_ids[i] = (cnt + block_m - 1) / block_m;  // s_ids is no longer needed
    }
    __syncthreads();
    const int tiles = block_exclusive_scan(s_ids, E, s_tmp);
    for (int i = threadIdx.x; i < E; i += blockDim.x) tile_offsets[i] = s_ids[i];
    if (threadIdx.x == 0) tile_offsets[E] = tiles;
  }
}

}  // namespace

cudaError_t launch_quant_gather(const void* x, int M, int K, int k, int32_t* route_slot,
                                uint8_t* a_q, float* a_scales, float* zero_acc, int zero_cols,
                                const Placement& pl, cudaStream_t stream, bool pdl,
                                bool token_major) {
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
                            k, route_slot, a_q, a_scales, zero_acc, zero_cols, pl,
                            token_major ? 1 : 0);
}

bool quant_layout_fits(int M, int K, int k, int E) {
  const int R = M * k;
  if (R > kQuantLayoutMaxRoutes || E > 1024 || K > 16384) return false;
  return true;
}

cudaError_t launch_quant_layout(const void* x, int M, int K, int k, int E, int block_m,
                                const int32_t* ids, uint8_t* a_q, float* a_scales, float* zero_acc,
                                int zero_cols, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_route_ids, int32_t* route_slot,
                                int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl) {
  const int G = K / 16;
  int threads, tpc;
  if (G <= 256) {
    threads = 256;
    tpc = 256 / G;
  } else {
    threads = (G + 31) / 32 * 32;
    tpc = 1;
  }
  const int R = M * k;
  const size_t smem = static_cast<size_t>(R + tpc * k + E) * sizeof(int);
  cudaError_t err = cudaFuncSetAttribute(quant_layout_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err == cudaSuccess) err = prefer_max_shared(quant_layout_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + tpc - 1) / tpc + 1);  // + the counts / offsets CTA
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_layout_kernel, static_cast<const __nv_bfloat16*>(x), M, K,
                            k, E, block_m, ids, a_q, a_scales, zero_acc, zero_cols, counts,
                            offsets, sorted_route_ids, route_slot, tile_offsets, ctrl);
}

}  // namespace moe
