// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include "moe_common.cuh"

namespace moe {

// Parameters of one grouped-GEMM launch (beyond the two TMA descriptors).
struct GemmParams {
  const float* a_scales;        // FP8: [KB, R]
  const float* w_scales;        // FP8: [E, N/128, KB]
  const int32_t* offsets;       // [E+1]
  const int32_t* tile_offsets;  // [E+1]
  const int32_t* sorted_route_ids;
  const float* route_weights;
  void* out;
  Ctrl* ctrl;
  unsigned* queue_ctr;          // tile-queue counter (zero at launch; reset by the last CTA)
  unsigned* done_ctr;
  int E, N, K, R, top_k;
  int KB;                       // K blocks of 128 bytes
  int k_splits, kb_per_split;
  int n_tiles;                  // output tiles of 128 columns
  int sched;
  int num_stages;
  int drop_producer;
  unsigned long long timeout_ns;
  // SCATTER only, optional: when out_bf16 is set, the CTA that adds the last
  // contribution to a (token, 128-column tile) of the fp32 output rounds that
  // segment to bf16 into out_bf16; tile_cnt[M * n_tiles] counts contributions
  // and must be zero at launch (top_k * k_splits arrive per entry).
  void* out_bf16;
  unsigned* tile_cnt;
};

cudaError_t launch_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                         int32_t* ids, float* weights, cudaStream_t stream, bool pdl);
cudaError_t launch_layout(const int32_t* ids, int R, int E, int block_m, int32_t* counts,
                          int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                          int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl);
cudaError_t launch_route_layout(const float* logits, int M, int E, int k, float softcap,
                                int renorm, int32_t* ids, float* weights, int block_m,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_route_ids,
                                int32_t* route_slot, int32_t* tile_offsets, Ctrl* ctrl,
                                cudaStream_t stream, bool pdl);
cudaError_t launch_quant_gather(const void* x, int M, int K, int k, const int32_t* route_slot,
                                uint8_t* a_q, float* a_scales, float* zero_acc, int zero_cols,
                                unsigned* zero_cnt, int cnt_per_token, cudaStream_t stream,
                                bool pdl);
cudaError_t launch_scatter(const float* rows, const int32_t* route_slot, const float* weights,
                           int M, int N, int k, void* out, cudaStream_t stream);
cudaError_t launch_gather_rows_bf16(const void* x, int M, int K, int k, const int32_t* route_slot,
                                    void* a, float* zero_acc, int zero_cols, unsigned* zero_cnt,
                                    int cnt_per_token, cudaStream_t stream, bool pdl);
cudaError_t launch_grouped_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_a,
                                const GemmParams& p, bool fp8, int epi, int bm, int num_ctas,
                                cudaStream_t stream, bool pdl);
int gemm_stage_bytes(bool fp8, int epi, int bm);

}  // namespace moe
