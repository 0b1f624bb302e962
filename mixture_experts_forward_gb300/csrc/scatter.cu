// Output-side glue of the forward:
//  - finalize: the fp32 accumulator that the grouped GEMM's scatter epilogue
//    adds into is rounded once to bf16 (round to nearest even).  It is
//    launched as a programmatic dependent of the GEMM, which triggers early,
//    so its CTAs are resident and start converting as soon as the GEMM ends;
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

__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ acc,
                                                       uint2* __restrict__ out, size_t n4) {
  pdl_wait();
  pdl_launch_dependents();
  // four independent 16-byte loads in flight per thread per step
  constexpr int kUnroll = 4;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcg(acc + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      __nv_bfloat162 a = __floats2bfloat162_rn(v[u].x, v[u].y);
      __nv_bfloat162 b = __floats2bfloat162_rn(v[u].z, v[u].w);
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&a);
      o.y = *reinterpret_cast<uint32_t*>(&b);
      out[i + u * stride] = o;
    }
  }
  for (; i < n4; i += stride) {
    const float4 v = __ldcg(acc + i);
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&a);
    o.y = *reinterpret_cast<uint32_t*>(&b);
    out[i] = o;
  }
}

__global__ void __launch_bounds__(256) scatter_kernel(const float* __restrict__ rows,
                                                      const int32_t* __restrict__ route_slot,
                                                      const float* __restrict__ weights, int M,
                                                      int N, int k,
                                                      __nv_bfloat16* __restrict__ out, Ctrl* ctrl) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= M) return;
  const int R = M * k;
  // a route whose slot is out of range adds nothing and is reported once per token
  if (threadIdx.x < k) {
    const int slot = __ldg(route_slot + static_cast<size_t>(t) * k + threadIdx.x);
    if (slot < 0 || slot >= R) set_error(ctrl, MOE_ERR_DEVICE_FAULT, 3);
  }
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

// Weighted reduction of bf16 expert-compact rows back to token order (the
// forward's large-batch form of the weighted scatter): out[t, :] =
// bf16( sum_j weights[t*k+j] * rows[route_slot[t*k+j], :] ), the sum in j order
// in fp32.  One thread per token and 8 columns (16-byte loads and stores).
__global__ void __launch_bounds__(256) reduce_rows_kernel(const uint4* __restrict__ rows,
                                                          const int32_t* __restrict__ route_slot,
                                                          const float* __restrict__ weights,
                                                          int M, int n8, int k,
                                                          uint4* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int R = M * k;
  const size_t total = static_cast<size_t>(M) * n8;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += stride) {
    const int t = static_cast<int>(i / n8);
    const int c = static_cast<int>(i - static_cast<size_t>(t) * n8);
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.0f;
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int slot = __ldg(route_slot + static_cast<size_t>(t) * k + j);
      if (slot < 0 || slot >= R) continue;
      const float w = __ldg(weights + static_cast<size_t>(t) * k + j);
      const uint4 v = __ldcs(rows + static_cast<size_t>(slot) * n8 + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h[u]);
        acc[2 * u] = __fmaf_rn(w, f.x, acc[2 * u]);
        acc[2 * u + 1] = __fmaf_rn(w, f.y, acc[2 * u + 1]);
      }
    }
    uint4 o;
    __nv_bfloat162* ho = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int u = 0; u < 4; ++u) ho[u] = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
    out[i] = o;
  }
}

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int M,
                                                          int row_vecs, int k, int32_t* route_slot,
                                                          uint4* __restrict__ a,
                                                          float* __restrict__ zero_acc,
                                                          int zero_cols, const Placement pl) {
  __shared__ int s_slot[32];
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= M) return;
  const int R = M * k;
  if (zero_acc != nullptr) {
    float4* row = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t) * zero_cols);
    for (int i = threadIdx.x; i < (zero_cols >> 2); i += blockDim.x)
      row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  if (static_cast<int>(threadIdx.x) < k) {
    const int r = t * k + threadIdx.x;
    int slot;
    if (pl.cta_base == nullptr) {
      slot = __ldg(route_slot + r);
    } else {
      const int e = __ldg(pl.ids + r);
      slot = -1;
      if (e >= 0 && e < pl.E) {
        slot = __ldg(pl.offsets + e) +
               __ldg(pl.cta_base + static_cast<size_t>(t / kRankTokensPerCta) * pl.E + e) +
               __ldg(pl.local_rank + r);
        if (slot >= R) slot = -1;
        if (slot >= 0) {
          route_slot[r] = slot;
          pl.sorted_route_ids[slot] = r;
        }
      }
    }
    s_slot[threadIdx.x] = slot;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
    const uint4 v = __ldg(x + static_cast<size_t>(t) * row_vecs + i);
    for (int j = 0; j < k; ++j) {
      const int slot = s_slot[j];
      if (slot >= 0 && slot < R) a[static_cast<size_t>(slot) * row_vecs + i] = v;
    }
  }
}

// Large-batch placement for a GEMM that gathers rows itself: 32 tokens per
// CTA; their accumulator rows are cleared before the wait for the router, then
// each route's slot is placed (route_slot, sorted_route_ids) as
// offsets[e] + cta_base[t / 32][e] + local_rank[r].
__global__ void __launch_bounds__(256) place_routes_kernel(int M, int k, int32_t* route_slot,
                                                           float* __restrict__ zero_acc,
                                                           int zero_cols, const Placement pl) {
  pdl_launch_dependents();
  const int t0 = blockIdx.x * 32;
  const int nt = min(32, M - t0);
  const int R = M * k;
  if (zero_acc != nullptr) {
    const int q = zero_cols >> 2;
    float4* rows = reinterpret_cast<float4*>(zero_acc + static_cast<size_t>(t0) * zero_cols);
    for (int i = threadIdx.x; i < nt * q; i += blockDim.x) rows[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int r = t0 * k + i;
    const int t = r / k;
    const int e = __ldg(pl.ids + r);
    if (e < 0 || e >= pl.E) continue;
    const int slot = __ldg(pl.offsets + e) +
                     __ldg(pl.cta_base + static_cast<size_t>(t / kRankTokensPerCta) * pl.E + e) +
                     __ldg(pl.local_rank + r);
    if (slot < 0 || slot >= R) continue;
    route_slot[r] = slot;
    pl.sorted_route_ids[slot] = r;
  }
}

}  // namespace

cudaError_t launch_finalize(const float* acc, void* out, size_t n, int num_sms,
                            cudaStream_t stream, bool pdl) {
  const size_t n4 = n / 4;
  // up to 8 CTAs of 256 threads per SM; each thread converts >= 4 vectors
  int blocks = static_cast<int>(std::min<size_t>((n4 + 1023) / 1024, static_cast<size_t>(num_sms) * 8));
  if (blocks < 1) blocks = 1;
  cudaError_t err = prefer_max_shared(finalize_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(blocks), dim3(256), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, finalize_kernel, reinterpret_cast<const float4*>(acc),
                            static_cast<uint2*>(out), n4);
}

cudaError_t launch_reduce_rows(const void* rows, const int32_t* route_slot, const float* weights,
                               int M, int N, int k, void* out, int num_sms, cudaStream_t stream,
                               bool pdl) {
  const size_t total = static_cast<size_t>(M) * (N / 8);
  int blocks = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(num_sms) * 8));
  if (blocks < 1) blocks = 1;
  cudaError_t err = prefer_max_shared(reduce_rows_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(blocks), dim3(256), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, reduce_rows_kernel, static_cast<const uint4*>(rows), route_slot,
                            weights, M, N / 8, k, static_cast<uint4*>(out));
}

cudaError_t launch_scatter(const float* rows, const int32_t* route_slot, const float* weights,
                           int M, int N, int k, void* out, Ctrl* ctrl, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(M), dim3(256), stream, false, attr);
  return cudaLaunchKernelEx(&cfg, scatter_kernel, rows, route_slot, weights, M, N, k,
                            static_cast<__nv_bfloat16*>(out), ctrl);
}

cudaError_t launch_place_routes(int M, int k, int32_t* route_slot, float* zero_acc, int zero_cols,
                                const Placement& pl, cudaStream_t stream, bool pdl) {
  cudaError_t err = prefer_max_shared(place_routes_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((M + 31) / 32), dim3(256), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, place_routes_kernel, M, k, route_slot, zero_acc, zero_cols, pl);
}

cudaError_t launch_gather_rows_bf16(const void* x, int M, int K, int k, int32_t* route_slot,
                                    void* a, float* zero_acc, int zero_cols, const Placement& pl,
                                    cudaStream_t stream, bool pdl) {
  cudaError_t err = prefer_max_shared(gather_rows_kernel);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(M), dim3(256), stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, static_cast<const uint4*>(x), M, K / 8, k,
                            route_slot, static_cast<uint4*>(a), zero_acc, zero_cols, pl);
}

}  // namespace moe
