// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include "moe_common.cuh"

namespace moe {

// Small kernels that run next to (or just before) the grouped GEMM ask for
// the largest shared-memory carveout: an SM still holding one of their CTAs
// can then take a GEMM CTA (210 KB of shared memory) without first draining
// to change its L1/shared split.
template <typename F>
inline cudaError_t prefer_max_shared(F* kernel) {
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                              cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// Launch configuration of a plain kernel, as a programmatic dependent of the
// previous launch on `stream` when `pdl` is set (attr: one slot, caller-owned).
inline cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t stream, bool pdl,
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

// Parameters of one grouped-GEMM launch (beyond the two TMA descriptors).
struct GemmParams {
  const float* a_scales;        // FP8: [KB, R]
  const float* w_scales;        // FP8: [E, N/128, KB]
  const int32_t* offsets;       // [E+1]
  const int32_t* tile_offsets;  // [E+1]
  const int32_t* sorted_route_ids;
  const float* route_weights;
  void* out;
  float* out_scales;            // FP8 SwiGLU: h block scales [N/256, R]
  Ctrl* ctrl;
  unsigned* queue_ctr;          // tile-queue counter (zero at launch; reset by the last CTA)
  unsigned* done_ctr;
  int E, N, K, R, top_k;
  int KB;                       // K blocks of 128 bytes
  int k_splits, kb_per_split;
  int n_tiles;                  // output tiles of 128 columns
  int sched;
  int num_stages;
  int sk;                       // K blocks per pipeline stage (1, 2 or 4)
  int w_reuse;                  // experts average more than one row tile: keep weights in L2
  int tail_tiles;               // FP8 scatter, one K split: last tiles split in K parts (the
                                // queue: this many; -G: balanced for G CTA pairs' fixed order)
  int tail_parts;               // 2 or 4 parts per split tile
  int tail_partkb;              // K blocks of each part but the last (a multiple of sk)
  int warm_first;               // before the wait for the layout: L2-prefetch the weight tiles
                                // of this CTA's likely first warm_first tiles (0 = off)
  int wide;                     // BF16 store / scatter: tiles of 256 output columns
  int cta2;                     // FP8 scatter at block_m 128: tiles of 256 weight rows over a
                                // cluster of two CTAs (n_tiles counts 256-row tiles)
  int gather;                   // A rows gathered from token-major rows (see moe_gemm_args)
  int M;                        // gather: rows of the token-major A (tokens)
  int drop_producer;
  unsigned long long timeout_ns;
};

cudaError_t launch_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                         int32_t* ids, float* weights, cudaStream_t stream, bool pdl);
cudaError_t launch_layout(const int32_t* ids, int R, int E, int block_m, int32_t* counts,
                          int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                          int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl);
// Route + per-CTA ranking of 32-token groups; the last CTA writes the per-CTA
// bases, counts, offsets and tile offsets (see Placement).
cudaError_t launch_route_rank(const float* logits, int M, int E, int k, float softcap, int renorm,
                              int32_t* ids, float* weights, int block_m, int32_t* counts,
                              int32_t* offsets, int32_t* tile_offsets, Ctrl* ctrl,
                              int32_t* local_rank, int32_t* cta_hist, int32_t* cta_base,
                              cudaStream_t stream, bool pdl);

// How a gather kernel finds the slot of route r = t*k + j: from route_slot
// (cta_base == nullptr), or — after launch_route_rank — as
// offsets[e] + cta_base[(t / 32) * E + e] + local_rank[r] with e = ids[r], in
// which case the kernel also writes route_slot[r] and sorted_route_ids[slot].
struct Placement {
  const int32_t* ids = nullptr;
  const int32_t* local_rank = nullptr;
  const int32_t* cta_base = nullptr;
  const int32_t* offsets = nullptr;
  int32_t* sorted_route_ids = nullptr;
  int E = 0;
};
constexpr int kRankTokensPerCta = 32;
// Largest M * top_k for which the forward folds the layout into the
// quantise/gather kernel (every CTA scans all routes' expert ids).
constexpr int kQuantLayoutMaxRoutes = 4096;
bool quant_layout_fits(int M, int K, int k, int E);
cudaError_t launch_quant_layout(const void* x, int M, int K, int k, int E, int block_m,
                                const int32_t* ids, uint8_t* a_q, float* a_scales, float* zero_acc,
                                int zero_cols, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_route_ids, int32_t* route_slot,
                                int32_t* tile_offsets, Ctrl* ctrl, cudaStream_t stream, bool pdl);
// SwiGLU of the FP8 gated FFN's up projection (gu f32 [R, 2I], gate columns
// first) re-quantised by the 1x128 rule: h_q u8 [R, I], h_scales f32 [I/128, R].
cudaError_t launch_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales,
                                int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_finalize(const float* acc, void* out, size_t n, int num_sms,
                            cudaStream_t stream, bool pdl);
// token_major: write each token's codes once ([M, K], scales [K/128, M]) and
// only place the routes, for a grouped GEMM that gathers its rows.
cudaError_t launch_quant_gather(const void* x, int M, int K, int k, int32_t* route_slot,
                                uint8_t* a_q, float* a_scales, float* zero_acc, int zero_cols,
                                const Placement& pl, cudaStream_t stream, bool pdl,
                                bool token_major = false);
// Large-batch placement without a row copy (the GEMM gathers rows): zero the
// accumulator rows, then write route_slot and sorted_route_ids.
cudaError_t launch_place_routes(int M, int k, int32_t* route_slot, float* zero_acc, int zero_cols,
                                const Placement& pl, cudaStream_t stream, bool pdl);
// out bf16 [M,N] = weighted sum over each token's k bf16 rows (N % 8 == 0).
cudaError_t launch_reduce_rows(const void* rows, const int32_t* route_slot, const float* weights,
                               int M, int N, int k, void* out, int num_sms, cudaStream_t stream,
                               bool pdl);
cudaError_t launch_scatter(const float* rows, const int32_t* route_slot, const float* weights,
                           int M, int N, int k, void* out, Ctrl* ctrl, cudaStream_t stream);
cudaError_t launch_gather_rows_bf16(const void* x, int M, int K, int k, int32_t* route_slot,
                                    void* a, float* zero_acc, int zero_cols, const Placement& pl,
                                    cudaStream_t stream, bool pdl);
cudaError_t launch_grouped_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_a,
                                const GemmParams& p, bool fp8, int epi, int bm, int num_ctas,
                                cudaStream_t stream, bool pdl);
int gemm_stage_bytes(bool fp8, int epi, int bm, bool wide = false, bool cta2 = false);
// BF16 store / scatter tiles of two adjacent weight tiles (256 output columns)
bool gemm_wide_supported(bool fp8, int epi, int bm);
// FP8 scatter tiles of 256 weight rows computed by a cluster of two CTAs
bool gemm_cta2_supported(bool fp8, int epi, int bm);
int gemm_cta2_max_clusters(bool query = true);
int gemm_meta_bytes(bool fp8, int bm, int kb_per_split, bool pair = false);
int gemm_rows_bytes(bool fp8, int bm);   // the route-id ring of the gathered-rows mode
// shared memory after the tables: the gathered-rows ring, or the FP8 SwiGLU
// epilogue's block-amax exchange
int gemm_extra_bytes(bool fp8, int epi, int bm, bool gather);
bool gemm_gather_supported(bool fp8, int epi);
int gemm_table_bytes(int E);

}  // namespace moe
