// Output-side glue of the forward:
//  - scatter: the unfused weighted scatter of "Fused MoE FP8: 8.09 -> 13.18
//    TFLOPS (1.63x)", section "Baseline: 7 kernels" item 7, written as a
//    deterministic gather per token (sum over j in order, fp32);
//  - gather_rows_bf16: the BF16 path's sort/gather (section "Fusion 2"
//    without quantisation): token rows copied to their expert-compact slots,
//    with the accumulator zeroed in the same pass.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) scatter_kernel(const float* __restrict__ rows,
                                                      const int32_t* __restrict__ route_slot,
                                                      const float* __restrict__ weights, int M,
                                                      int N, int k,
                                                      __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= M) return;
  const int R = M * k;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int slot = __ldg(route_slot + static_cast<size_t>(t) * k + j);
      if (slot < 0 || slot >= R) continue;
      acc = __fmaf_rn(__ldg(weights + static_cast<size_t>(t) * k + j),
                      __ldg(rows + static_cast<size_t>(slot) * N + n), acc);
    }
    out[static_cast<size_t>(t) * N + n] = __float2bfloat16_rn(acc);
  }
}

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int M,
                                                          int row_vecs, int k,
                                                          const int32_t* __restrict__ route_slot,
                                                          uint4* __restrict__ a,
                                                          float* __restrict__ zero_acc,
                                                          int zero_cols,
                                                          unsigned* __restrict__ zero_cnt,
                                                          int cnt_per_token) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= M) return;
  const int R = M * k;
  if (zero_acc != nullptr) {
    float4* row = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t) * zero_cols);
    for (int i = threadIdx.x; i < (zero_cols >> 2); i += blockDim.x)
      row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (zero_cnt != nullptr)
    for (int i = threadIdx.x; i < cnt_per_token; i += blockDim.x)
      zero_cnt[static_cast<size_t>(t) * cnt_per_token + i] = 0u;
  int slots[32];
#pragma unroll
  for (int j = 0; j < 32; ++j)
    slots[j] = j < k ? __ldg(route_slot + static_cast<size_t>(t) * k + j) : -1;
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
    uint4 v = __ldg(x + static_cast<size_t>(t) * row_vecs + i);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < k && slots[j] >= 0 && slots[j] < R) a[static_cast<size_t>(slots[j]) * row_vecs + i] = v;
    }
  }
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t stream, bool pdl,
                            cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_scatter(const float* rows, const int32_t* route_slot, const float* weights,
                           int M, int N, int k, void* out, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(M), dim3(256), stream, false, attr);
  return cudaLaunchKernelEx(&cfg, scatter_kernel, rows, route_slot, weights, M, N, k,
                            static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_gather_rows_bf16(const void* x, int M, int K, int k, const int32_t* route_slot,
                                    void* a, float* zero_acc, int zero_cols, unsigned* zero_cnt,
                                    int cnt_per_token, cudaStream_t stream, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(M), dim3(256), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, static_cast<const uint4*>(x), M, K / 8, k,
                            route_slot, static_cast<uint4*>(a), zero_acc, zero_cols, zero_cnt,
                            cnt_per_token);
}

}  // namespace moe
