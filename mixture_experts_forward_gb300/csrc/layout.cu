// Count + build layout in one CTA.
//
// "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section "Fusion 3"
// (count_and_build: shared-memory histogram then prefix over the experts) and
// section "Parallel Hillis-Steele Prefix Scan" (the serial scan replaced by a
// parallel one); the blog retelling of "Weave", section 4.3 (histogram ->
// prefix -> per-expert tiles of the task queue).
//
// Here the slot order inside an expert is made deterministic: routes of an
// expert occupy its segment in ascending route id (t*top_k + j).  The pages
// hand out slots with atomicAdd, whose order is arbitrary.
//
// Work split (1024 threads = 32 warps): warp w owns the routes
// [w*chunk, (w+1)*chunk).  Pass 1 counts them into the warp's private row of a
// [32][E] shared histogram, grouping equal ids of a 32-route step with
// __match_any_sync (no atomics).  Per expert, the rows are turned into
// exclusive per-warp bases; counts and ceil(count/block_m) are scanned over the
// experts with warp shuffles (no serial loop over E).  Pass 2 revisits the same
// routes in the same order and writes each one to base + rank-in-step.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

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

__global__ void __launch_bounds__(kThreads, 1)
    layout_kernel(const int32_t* __restrict__ ids, int R, int E, int block_m,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ sorted_route_ids, int32_t* __restrict__ route_slot,
                  int32_t* __restrict__ tile_offsets, Ctrl* ctrl) {
  extern __shared__ int s_hist[];  // [kWarps][E]
  __shared__ int s_wa[32], s_wb[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_wait();
  for (int i = tid; i < kWarps * E; i += kThreads) s_hist[i] = 0;
  if (tid == 0) s_bad = 0;
  if (tid == 0 && ctrl != nullptr) {
    ctrl->queue = 0;
    ctrl->done = 0;
    ctrl->queue2 = 0;
    ctrl->done2 = 0;
  }
  __syncthreads();

  const int chunk = (R + kWarps - 1) / kWarps;
  const int r_begin = min(R, warp * chunk), r_end = min(R, r_begin + chunk);
  int* my_row = s_hist + warp * E;

  // pass 1: per-warp histogram
  for (int r0 = r_begin; r0 < r_end; r0 += 32) {
    int r = r0 + lane;
    int e = r < r_end ? __ldg(ids + r) : -1;
    if (r < r_end && (e < 0 || e >= E)) {
      s_bad = 1;
      e = -2;  // excluded from the layout
    }
    uint32_t same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(same) - 1) my_row[e] += __popc(same);
    __syncwarp();
  }
  __syncthreads();

  // per expert: total count and exclusive per-warp bases
  int cnt = 0, ntile = 0;
  const int e = tid;
  if (e < E) {
    for (int w = 0; w < kWarps; ++w) {
      int c = s_hist[w * E + e];
      s_hist[w * E + e] = cnt;
      cnt += c;
    }
    ntile = (cnt + block_m - 1) / block_m;
  }
  int inc_c = cnt, inc_t = ntile;
  block_scan2(inc_c, inc_t, s_wa, s_wb);  // requires E <= kThreads
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = inc_c - cnt;
    tile_offsets[e] = inc_t - ntile;
    if (e == E - 1) {
      offsets[E] = inc_c;
      tile_offsets[E] = inc_t;
    }
    for (int w = 0; w < kWarps; ++w) s_hist[w * E + e] += inc_c - cnt;
  }
  __syncthreads();

  // pass 2: stable placement
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int r0 = r_begin; r0 < r_end; r0 += 32) {
    int r = r0 + lane;
    int ex = r < r_end ? __ldg(ids + r) : -1;
    if (r < r_end && (ex < 0 || ex >= E)) ex = -2;
    uint32_t same = __match_any_sync(0xffffffffu, ex);
    int base = ex >= 0 ? my_row[ex] : 0;
    __syncwarp();
    if (ex >= 0) {
      int slot = base + __popc(same & lt_mask);
      sorted_route_ids[slot] = r;
      route_slot[r] = slot;
      if (lane == __ffs(same) - 1) my_row[ex] = base + __popc(same);
    } else if (ex == -2) {
      route_slot[r] = -1;  // invalid id: the route has no slot
    }
    __syncwarp();
  }
  pdl_launch_dependents();
  __syncthreads();
  if (tid == 0 && s_bad) set_error(ctrl, MOE_ERR_DEVICE_FAULT, 1);
}

}  // namespace

size_t layout_smem_bytes(int E) { return static_cast<size_t>(kWarps) * E * sizeof(int); }

cudaError_t launch_layout(const int32_t* ids, int R, int E, int block_m, int32_t* counts,
                          int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                          int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl) {
  const size_t smem = layout_smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, layout_kernel, ids, R, E, block_m, counts, offsets,
                            sorted_route_ids, route_slot, tile_offsets, ctrl);
}

}  // namespace moe
