// Standalone count + build layout kernel (one CTA); the algorithm is in
// layout_block.cuh.
#include "layout_block.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(kLayoutThreads, 1)
    layout_kernel(const int32_t* __restrict__ ids, int R, int E, int block_m,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ sorted_route_ids, int32_t* __restrict__ route_slot,
                  int32_t* __restrict__ tile_offsets, Ctrl* ctrl) {
  extern __shared__ int s_hist[];  // [layout_warps(R)][E]
  pdl_wait();
  pdl_launch_dependents();
  layout_block(ids, R, E, block_m, counts, offsets, sorted_route_ids, route_slot, tile_offsets,
               ctrl, s_hist);
}

}  // namespace

size_t layout_smem_bytes(int R, int E) {
  return static_cast<size_t>(layout_warps(R)) * E * sizeof(int);
}

cudaError_t launch_layout(const int32_t* ids, int R, int E, int block_m, int32_t* counts,
                          int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                          int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl) {
  const size_t smem = layout_smem_bytes(R, E);
  cudaError_t err = cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kLayoutThreads);
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
