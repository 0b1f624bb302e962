// Count + build layout for one CTA of 1024 threads (used by the standalone
// layout kernel and by the last CTA of the fused route kernel).
//
// "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Fusion 3"
// (count_and_build: shared-memory histogram then prefix over the experts) and
// section "Parallel Hillis-Steele Prefix Scan" (no serial scan); the blog
// retelling of "Weave", section 4.3 (histogram -> prefix -> per-expert tiles).
//
// Slot order inside an expert is deterministic: ascending route id
// (t*top_k + j); the pages hand out slots with atomicAdd, in arbitrary order.
//
// Work split: warps 0..nw-1 (nw <= 32) own consecutive route ranges.  Pass 1 counts each
// range into the warp's private row of an [nw][E] shared histogram, grouping
// equal ids of a 32-route step with __match_any_sync (no atomics).  Per expert
// (one thread each), the rows become exclusive per-warp bases; counts and
// ceil(count/block_m) are scanned over the experts with warp shuffles.  Pass 2
// revisits the same routes in the same order and writes each one to
// base + rank-in-step.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kLayoutThreads = 1024;

// Warps that take part in the histogram passes: about 32 routes each, so a
// small layout is one step per warp.
__host__ __device__ inline int layout_warps(int R) {
  int nw = (R + 31) / 32;
  return nw < 1 ? 1 : (nw > 32 ? 32 : nw);
}

// Inclusive block-wide scan of two values per thread (blockDim = 1024).
__device__ __forceinline__ void block_scan2(int& a, int& b, int* s_warp_a, int* s_warp_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int ya = __shfl_up_sync(0xffffffffu, a, off);
    int yb = __shfl_up_sync(0xffffffffu, b, off);
    if (lane >= off) {
      a += ya;
      b += yb;
    }
  }
  if (lane == 31) {
    s_warp_a[warp] = a;
    s_warp_b[warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    int wa = s_warp_a[lane], wb = s_warp_b[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int ya = __shfl_up_sync(0xffffffffu, wa, off);
      int yb = __shfl_up_sync(0xffffffffu, wb, off);
      if (lane >= off) {
        wa += ya;
        wb += yb;
      }
    }
    s_warp_a[lane] = wa;  // inclusive totals of warps 0..lane
    s_warp_b[lane] = wb;
  }
  __syncthreads();
  if (warp > 0) {
    a += s_warp_a[warp - 1];
    b += s_warp_b[warp - 1];
  }
}

// s_hist: [layout_warps(R)][E] ints of shared memory.  Must be called by all
// 1024 threads of the CTA.  ids are read with L2 loads (they may have been
// written by other CTAs of the same grid).
static __device__ void layout_block(const int32_t* ids, int R, int E, int block_m, int32_t* counts,
                             int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                             int32_t* tile_offsets, Ctrl* ctrl, int* s_hist) {
  __shared__ int s_wa[32], s_wb[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = layout_warps(R);

  for (int i = tid; i < nw * E; i += kLayoutThreads) s_hist[i] = 0;
  if (tid == 0) s_bad = 0;
  if (tid == 0 && ctrl != nullptr) {
    ctrl->queue = 0;
    ctrl->done = 0;
    ctrl->queue2 = 0;
    ctrl->done2 = 0;
  }
  __syncthreads();

  const int chunk = (R + nw - 1) / nw;
  const int r_begin = warp < nw ? min(R, warp * chunk) : R;
  const int r_end = warp < nw ? min(R, r_begin + chunk) : R;
  int* my_row = s_hist + (warp < nw ? warp : 0) * E;

  // pass 1: per-warp histogram.  A warp walks its range in steps of 32
  // routes; the ids of kBatch steps are loaded together so their latencies
  // overlap.  When the whole range is one batch (R <= 32 * 32 * kBatch) the
  // ids and match masks stay in registers for pass 2.
  constexpr int kBatch = 8;
  const bool one_batch = r_end - r_begin <= 32 * kBatch;
  int eb[kBatch];
  uint32_t mb[kBatch];
  for (int b0 = r_begin; b0 < r_end; b0 += 32 * kBatch) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int r = b0 + 32 * j + lane;
      eb[j] = r < r_end ? __ldcg(ids + r) : -1;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int r = b0 + 32 * j + lane;
      if (b0 + 32 * j >= r_end) break;  // warp-uniform
      if (r < r_end && (eb[j] < 0 || eb[j] >= E)) {
        s_bad = 1;
        eb[j] = -2;  // excluded from the layout
      }
      mb[j] = __match_any_sync(0xffffffffu, eb[j]);
      if (eb[j] >= 0 && lane == __ffs(mb[j]) - 1) my_row[eb[j]] += __popc(mb[j]);
      __syncwarp();
    }
  }
  __syncthreads();

  // per expert: total count and exclusive per-warp bases
  int cnt = 0, ntile = 0;
  const int e = tid;
  if (e < E) {
    for (int w = 0; w < nw; ++w) {
      const int c = s_hist[w * E + e];
      s_hist[w * E + e] = cnt;
      cnt += c;
    }
    ntile = (cnt + block_m - 1) / block_m;
  }
  int inc_c = cnt, inc_t = ntile;
  block_scan2(inc_c, inc_t, s_wa, s_wb);  // E <= 1024 threads
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = inc_c - cnt;
    tile_offsets[e] = inc_t - ntile;
    if (e == E - 1) {
      offsets[E] = inc_c;
      tile_offsets[E] = inc_t;
    }
    for (int w = 0; w < nw; ++w) s_hist[w * E + e] += inc_c - cnt;
  }
  __syncthreads();

  // pass 2: stable placement
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int b0 = r_begin; b0 < r_end; b0 += 32 * kBatch) {
    if (!one_batch) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int r = b0 + 32 * j + lane;
        int ex = r < r_end ? __ldcg(ids + r) : -1;
        if (r < r_end && (ex < 0 || ex >= E)) ex = -2;
        eb[j] = ex;
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int r = b0 + 32 * j + lane;
      if (b0 + 32 * j >= r_end) break;  // warp-uniform
      const int ex = eb[j];
      const uint32_t same = one_batch ? mb[j] : __match_any_sync(0xffffffffu, ex);
      const int base = ex >= 0 ? my_row[ex] : 0;
      __syncwarp();
      if (ex >= 0) {
        const int slot = base + __popc(same & lt_mask);
        sorted_route_ids[slot] = r;
        route_slot[r] = slot;
        if (lane == __ffs(same) - 1) my_row[ex] = base + __popc(same);
      } else if (ex == -2) {
        route_slot[r] = -1;  // invalid id: the route has no slot
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (tid == 0 && s_bad) set_error(ctrl, MOE_ERR_DEVICE_FAULT, 1);
}

}  // namespace moe
