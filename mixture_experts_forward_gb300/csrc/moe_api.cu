// C ABI of the fused MoE forward: argument checks, TMA descriptors, workspace
// layout, the launch sequence of the forward and its CUDA-graph cache.
//
// The forward is the serving path of "Fused MoE FP8: 8.09 -> 13.18 TFLOPS
// (1.63x)" (section "Phase 2": no host synchronisation between launches, the
// launch sequence captured once into a CUDA graph and replayed), extended with
// the router in front and a bf16 finalize at the end.  Consecutive kernels are
// chained with programmatic dependent launch (the PDL idea of section 2.3 of
// the Weave retelling): each kernel's prologue overlaps its predecessor's tail
// and its griddepcontrol.wait orders the data.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "moe_internal.cuh"

using namespace moe;

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s
int g_drop_producer = 0;
unsigned long long g_timeout_ns = kDefaultTimeoutNs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D K-major tensor map: rows of `inner` elements, `outer` rows, 128-byte
// swizzle, box = 128 bytes x box_rows; out-of-range rows read as zero.
// Operand view for the grouped GEMM: a row-major [outer, inner] matrix seen
// as 3-D {128-byte K block slice, row, K block}, so one box brings `sk`
// consecutive K blocks of `box_rows` rows ([K block][row][128 B] in shared
// memory, 128-byte swizzle) and each row is read `sk` * 128 bytes at a time.
bool make_tmap(CUtensorMap* m, const void* base, bool fp8, uint64_t inner, uint64_t outer,
               uint32_t box_rows, uint32_t sk) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint32_t esize = fp8 ? 1 : 2;
  const uint64_t kb_elems = 128u / esize;
  cuuint64_t dims[3] = {kb_elems, outer, inner / kb_elems};
  cuuint64_t strides[2] = {inner * esize, 128u};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kb_elems), box_rows, sk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over token-major rows [rows, inner] for the gathered-rows mode:
// one-row boxes of 128 bytes (tile::gather4 loads four rows per copy), with
// the same 128-byte swizzle as the tiled operand boxes.
bool make_tmap_rows(CUtensorMap* m, const void* base, bool fp8, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint32_t esize = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {128u / esize, 1u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

thread_local char g_last_error[256] = "";

moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

int auto_block_m(bool fp8, long long R, int E) {
  const long long avg = (R + E - 1) / E;
  if (avg <= 16) return 16;
  if (avg <= 32) return 32;
  if (avg <= 64) return 64;
  if (fp8 || avg <= 128) return 128;
  return 256;
}

// Host checks shared by moe_grouped_gemm and the forward.
moe_status_t check_gemm(const moe_gemm_args* a) {
  if (a == nullptr) return MOE_ERR_INVALID_ARG;
  const bool fp8 = a->dtype == MOE_DTYPE_FP8_E4M3;
  if (a->dtype != MOE_DTYPE_FP8_E4M3 && a->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (a->epilogue < MOE_EPI_SCATTER || a->epilogue > MOE_EPI_STORE_BF16) return MOE_ERR_INVALID_ARG;
  if (a->sched != MOE_SCHED_QUEUE && a->sched != MOE_SCHED_STATIC) return MOE_ERR_INVALID_ARG;
  if (a->cta_pairs != 0 && a->cta_pairs != -1) return MOE_ERR_INVALID_ARG;
  if (a->E <= 0 || a->N <= 0 || a->K <= 0 || a->R <= 0) return MOE_ERR_INVALID_ARG;
  if (a->a == nullptr || a->w == nullptr || a->offsets == nullptr || a->tile_offsets == nullptr ||
      a->out == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a->a) || !aligned16(a->w) || !aligned16(a->out)) return MOE_ERR_INVALID_ARG;
  if (a->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (a->block_m < 16 || a->block_m > 256 || a->block_m % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if ((a->block_m & (a->block_m - 1)) != 0) return MOE_ERR_UNSUPPORTED;
  if (a->N % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (fp8) {
    if (a->K % 128 != 0 || a->block_m > 128) return MOE_ERR_UNSUPPORTED;
    if (a->a_scales == nullptr || a->w_scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (a->epilogue == MOE_EPI_SWIGLU) {
      // gate + up tiles of 128 h columns each; codes and block scales out
      if (a->N % 256 != 0 || a->gather_rows != 0) return MOE_ERR_UNSUPPORTED;
      if (a->out_scales == nullptr || (reinterpret_cast<uintptr_t>(a->out_scales) & 3u) != 0)
        return MOE_ERR_INVALID_ARG;
    }
  } else {
    if (a->K % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (a->epilogue == MOE_EPI_SWIGLU && a->N % 256 != 0) return MOE_ERR_UNSUPPORTED;
  }
  if (a->epilogue == MOE_EPI_SCATTER) {
    if (a->sorted_route_ids == nullptr || a->route_weights == nullptr) return MOE_ERR_INVALID_ARG;
    if (a->M <= 0 || a->top_k <= 0 || static_cast<long long>(a->M) * a->top_k != a->R)
      return MOE_ERR_INVALID_ARG;
  }
  if (a->k_splits < 0) return MOE_ERR_INVALID_ARG;
  if (a->k_splits > 1 && !(fp8 && a->epilogue == MOE_EPI_SCATTER)) return MOE_ERR_UNSUPPORTED;
  if (a->gather_rows != 0) {
    if (a->gather_rows != 1 || a->sorted_route_ids == nullptr) return MOE_ERR_INVALID_ARG;
    if (!gemm_gather_supported(fp8, a->epilogue)) return MOE_ERR_UNSUPPORTED;
    if (a->M <= 0 || a->top_k <= 0 || static_cast<long long>(a->M) * a->top_k != a->R)
      return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

int pick_k_splits(const moe_gemm_args* a, int sms, int KB) {
  if (a->k_splits > 0) return a->k_splits > KB ? KB : a->k_splits;
  if (!(a->dtype == MOE_DTYPE_FP8_E4M3 && a->epilogue == MOE_EPI_SCATTER)) return 1;
  // Upper bound of the tile count (every row in its own expert's ragged tile).
  const long long tiles =
      ((static_cast<long long>(a->R) + a->block_m - 1) / a->block_m + a->E) * (a->N / 128);
  int ks = 1;
  while (tiles * ks < 4LL * sms && ks * 2 <= KB / 4) ks *= 2;
  return ks;
}

moe_status_t run_gemm(const moe_gemm_args* a, Ctrl* ctrl, bool second, cudaStream_t stream,
                      bool pdl) {
  const bool fp8 = a->dtype == MOE_DTYPE_FP8_E4M3;
  const int sms = device_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.a_scales = a->a_scales;
  p.w_scales = a->w_scales;
  p.offsets = a->offsets;
  p.tile_offsets = a->tile_offsets;
  p.sorted_route_ids = a->sorted_route_ids;
  p.route_weights = a->route_weights;
  p.out = a->out;
  p.out_scales = a->out_scales;
  p.ctrl = ctrl;
  p.queue_ctr = second ? &ctrl->queue2 : &ctrl->queue;
  p.done_ctr = second ? &ctrl->done2 : &ctrl->done;
  p.E = a->E;
  p.N = a->N;
  p.K = a->K;
  p.R = a->R;
  p.top_k = a->top_k;
  p.KB = fp8 ? a->K / 128 : a->K / 64;
  p.k_splits = pick_k_splits(a, sms, p.KB);
  p.kb_per_split = (p.KB + p.k_splits - 1) / p.k_splits;
  // BF16 store / scatter with 128- or 256-row tiles: two adjacent weight
  // tiles per tile (a stage then carries two MMAs per K block)
  p.wide = (gemm_wide_supported(fp8, a->epilogue, a->block_m) && a->gather_rows == 0 &&
            a->N % 256 == 0) ? 1 : 0;
  // FP8 at 128 routed rows, scatter (the same 256-row tiles, a 128-row half on
  // each CTA) and SwiGLU (tiles of 2 x 128 routed rows, 128 on each CTA): a
  // cluster of two CTAs per tile; an even grid of at most the clusters that
  // fit at once
  int ctas = a->num_ctas > 0 ? a->num_ctas : sms;
  const bool swiglu = a->epilogue == MOE_EPI_SWIGLU;
  if (a->cta_pairs == 0 && (p.wide || swiglu) && a->gather_rows == 0 &&
      gemm_cta2_supported(fp8, a->epilogue, a->block_m)) {
    // (the first query per device is kept out of stream captures)
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool capturing =
        cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
    const int max_cl = gemm_cta2_max_clusters(!capturing);
    const int pairs = (ctas < 2 * max_cl ? ctas : 2 * max_cl) / 2;
    if (pairs >= 1) {
      p.cta2 = 1;
      p.wide = 0;
      ctas = 2 * pairs;
    }
  }
  p.n_tiles = (swiglu ? a->N / 2 : a->N) / ((p.wide || (p.cta2 && !swiglu)) ? 256 : 128);
  p.sched = a->sched;
  p.w_reuse = 2LL * a->R >= static_cast<long long>(a->block_m) * a->E ? 1 : 0;
  p.drop_producer = g_drop_producer;
  p.timeout_ns = g_timeout_ns;
  const int stage_bytes = gemm_stage_bytes(fp8, a->epilogue, a->block_m, p.wide != 0, p.cta2 != 0);
  if (stage_bytes <= 0) return MOE_ERR_UNSUPPORTED;
  const bool pair = fp8 && (p.wide != 0 || a->epilogue == MOE_EPI_SWIGLU);
  const int meta_bytes = gemm_meta_bytes(fp8, a->block_m, p.kb_per_split, pair);
  p.gather = a->gather_rows;
  p.M = a->M;
  // FP8 weights read once per expert (no row-tile reuse) through the queue:
  // warm L2 with each CTA's likely first weight tile before the layout is known
  p.warm_first = (fp8 && !p.w_reuse && a->sched == MOE_SCHED_QUEUE && !p.cta2) ? 1 : 0;
  const int rows_bytes = gemm_extra_bytes(fp8, a->epilogue, a->block_m, p.gather != 0);
  // Several K blocks per stage (more bytes per copy instruction, and 128 *
  // sk contiguous bytes of every weight row per copy): the largest of 4, 2, 1
  // that divides a split and still leaves at least three stages.
  const int avail = 232448 - 1024 - 2048 - meta_bytes - gemm_table_bytes(a->E) - rows_bytes;
  p.sk = 1;
  for (int sk = 4; sk >= 2; sk /= 2)
    if (p.kb_per_split % sk == 0 && avail / (sk * stage_bytes) >= 3) { p.sk = sk; break; }
  // FP8 pair tiles of 128 routed rows that store their results feed both
  // weight tiles to one MMA as a single 256-row operand, so a stage holds one
  // K block (the tiles adjacent)
  // (CTA pairs stage one weight tile per CTA, so their stages may be deeper)
  if (pair && a->block_m == 128 && a->epilogue != MOE_EPI_SCATTER && !p.cta2) p.sk = 1;
  int stages = avail / (p.sk * stage_bytes);
  if (stages > 16) stages = 16;
  if (stages < 2) return MOE_ERR_UNSUPPORTED;
  p.num_stages = stages;
  // FP8 scatter through the queue: split the last wave (one tile per CTA) in
  // K parts, so CTAs finish within a part of a tile of one another — quarters
  // where tiles are narrow (block_m <= 32: a cheap epilogue per part), else halves
  p.tail_parts = 2;
  for (int parts = a->block_m <= 32 ? 4 : 2; parts >= 2; parts /= 2) {
    const int partkb = (p.KB / parts) / p.sk * p.sk;
    if (partkb >= p.sk && p.KB - (parts - 1) * partkb >= p.sk) {
      p.tail_parts = parts;
      p.tail_partkb = partkb;
      break;
    }
  }
  // (CTA pairs walk a fixed round-robin list, one tile per pair at a time)
  if (fp8 && a->epilogue == MOE_EPI_SCATTER && p.k_splits == 1 &&
      (a->sched == MOE_SCHED_QUEUE || p.cta2) && p.tail_partkb > 0)
    p.tail_tiles = p.cta2 ? -(ctas / 2) : ctas;   // (negative: the pairs' balanced tail)
  CUtensorMap tw, ta;
  if (!make_tmap(&tw, a->w, fp8, static_cast<uint64_t>(a->K),
                 static_cast<uint64_t>(a->E) * a->N, 128u, static_cast<uint32_t>(p.sk)))
    return MOE_ERR_CUDA;
  if (p.gather) {
    if (!make_tmap_rows(&ta, a->a, fp8, static_cast<uint64_t>(a->K), static_cast<uint64_t>(a->M)))
      return MOE_ERR_CUDA;
  } else if (!make_tmap(&ta, a->a, fp8, static_cast<uint64_t>(a->K), static_cast<uint64_t>(a->R),
                        static_cast<uint32_t>((p.cta2 && !(fp8 && swiglu)) ? a->block_m / 2
                                                                           : a->block_m),
                        static_cast<uint32_t>(p.sk))) {
    return MOE_ERR_CUDA;
  }
  return cuda_status(launch_grouped_gemm(tw, ta, p, fp8, a->epilogue, a->block_m, ctas, stream,
                                         pdl));
}

// ---------------------------------------------------------------------------
// Workspace layout of the forward.
struct WsLayout {
  size_t ctrl, ids, weights, counts, offsets, tile_off, sorted, slot, a, a_scales, acc, h;
  size_t hq, hs;  // FP8 gated FFN: h codes [R, N] and scales [N/128, R] (h: f32 gu [R, 2N])
  size_t local_rank, cta_hist, cta_base;
  size_t st_logits, st_x, st_out;
  size_t total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The FP8 gated FFN (two FP8 projections with h re-quantised between them).
bool fp8_ffn(const moe_forward_args* f) {
  return f->dtype == MOE_DTYPE_FP8_E4M3 && f->gated == 1;
}

// Columns of the forward's output: N for the single FP8 GEMM, K (the token
// feature size) for the gated FFNs.
long long out_cols(const moe_forward_args* f) {
  return (f->dtype == MOE_DTYPE_FP8_E4M3 && f->gated != 1) ? f->N : f->K;
}

bool forward_shape_ok(const moe_forward_args* f) {
  return f != nullptr && f->M > 0 && f->K > 0 && f->N > 0 && f->E > 0 && f->top_k > 0;
}

// The weighted scatter's form: while the fp32 output accumulator fits well
// inside L2 the last GEMM scatter-adds into it (reductions stay on chip and
// one conversion pass follows); a larger accumulator would be read and
// written back to HBM by the reductions, so the GEMM stores each routed row
// in bf16 instead and one kernel reduces every token's rows (streaming).
constexpr long long kAccOnChipBytes = 112ll << 20;
bool rows_path(const moe_forward_args* f) {
  return static_cast<long long>(f->M) * out_cols(f) * 4 > kAccOnChipBytes;
}

// The forward's large-batch path with gather_rows set gathers the routed rows
// inside the first grouped GEMM.
bool forward_gathers(const moe_forward_args* f) {
  const bool fp8 = f->dtype == MOE_DTYPE_FP8_E4M3;
  // the FP8 gated FFN's fused SwiGLU up projection reads compact rows only
  return f->gather_rows == 1 && !(fp8 && quant_layout_fits(f->M, f->K, f->top_k, f->E)) &&
         !fp8_ffn(f);
}

WsLayout ws_layout(const moe_forward_args* f) {
  WsLayout L;
  std::memset(&L, 0, sizeof(L));
  const bool fp8 = f->dtype == MOE_DTYPE_FP8_E4M3;
  const size_t M = f->M, K = f->K, N = f->N, E = f->E, k = f->top_k, R = M * k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.ctrl = take(MOE_CTRL_BYTES);
  L.ids = take(R * 4);
  L.weights = take(R * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.tile_off = take((E + 1) * 4);
  L.sorted = take(R * 4);
  L.slot = take(R * 4);
  const size_t n_rank_ctas = (M + kRankTokensPerCta - 1) / kRankTokensPerCta;
  L.local_rank = take(R * 4);
  L.cta_hist = take(n_rank_ctas * E * 4);
  L.cta_base = take(n_rank_ctas * E * 4);
  // gathered rows (large batches): FP8 codes and scales token-major, BF16 rows
  // read straight from x; otherwise the expert-compact copy
  const bool gather = forward_gathers(f);
  const size_t a_rows = gather ? M : R;
  L.a = (gather && !fp8) ? 0 : take(fp8 ? a_rows * K : a_rows * K * 2);
  L.a_scales = fp8 ? take((K / 128) * a_rows * 4) : 0;
  const size_t cols = static_cast<size_t>(out_cols(f));
  // fp32 accumulator [M, out] for the scatter-add, or bf16 expert-compact rows
  // [R, out] reduced afterwards (see rows_path)
  if (rows_path(f))
    L.acc = take(R * cols * 2);
  else
    L.acc = take(M * cols * 4);
  // gated FFN intermediates: BF16 h [R, N]; FP8 h's codes [R, N] and block
  // scales [N/128, R], written by the up projection's epilogue
  if (!fp8) {
    L.h = take(R * N * 2);
  } else if (fp8_ffn(f)) {
    L.hq = take(R * N);
    L.hs = take((N / 128) * R * 4);
  }
  L.st_logits = take(M * E * 4);
  L.st_x = take(M * K * 2);
  L.st_out = take(M * cols * 2);
  L.total = off;
  return L;
}

moe_status_t check_forward(const moe_forward_args* f) {
  if (!forward_shape_ok(f)) return MOE_ERR_INVALID_ARG;
  if (f->dtype != MOE_DTYPE_FP8_E4M3 && f->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (f->sched != MOE_SCHED_QUEUE && f->sched != MOE_SCHED_STATIC) return MOE_ERR_INVALID_ARG;
  if (f->cta_pairs != 0 && f->cta_pairs != -1) return MOE_ERR_INVALID_ARG;
  if (f->w == nullptr) return MOE_ERR_INVALID_ARG;
  if (f->E > 1024 || f->top_k > 32 || f->top_k > f->E) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(f->M) * f->top_k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (f->K % 128 != 0 || f->N % 128 != 0 || f->K > 16384) return MOE_ERR_UNSUPPORTED;
  if (!(f->softcap >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (f->gather_rows != 0 && f->gather_rows != 1) return MOE_ERR_INVALID_ARG;
  if (f->gated != 0 && f->gated != 1) return MOE_ERR_INVALID_ARG;
  if (f->block_m != 0 && (f->block_m < 16 || f->block_m > 256 || (f->block_m & (f->block_m - 1))))
    return MOE_ERR_UNSUPPORTED;
  if (f->dtype == MOE_DTYPE_FP8_E4M3) {
    if (f->w_scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (f->gated == 1 && (f->w2 == nullptr || f->w2_scales == nullptr)) return MOE_ERR_INVALID_ARG;
    if (f->block_m > 128) return MOE_ERR_UNSUPPORTED;
  } else {
    if (f->w2 == nullptr) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(f->w) || (f->w2 && !aligned16(f->w2))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The launch sequence of one forward (no host synchronisation).
moe_status_t enqueue_forward(const moe_forward_args* f, const float* logits, const void* x,
                             void* out, uint8_t* ws, cudaStream_t stream) {
  const bool fp8 = f->dtype == MOE_DTYPE_FP8_E4M3;
  const WsLayout L = ws_layout(f);
  const int M = f->M, K = f->K, N = f->N, E = f->E, k = f->top_k, R = M * k;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  float* wts = reinterpret_cast<float*>(ws + L.weights);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + L.tile_off);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  int32_t* slot = reinterpret_cast<int32_t*>(ws + L.slot);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  const int bm = f->block_m > 0 ? f->block_m : auto_block_m(fp8, R, E);
  const bool pdl = true;
  cudaError_t e;

  const bool small = fp8 && quant_layout_fits(M, K, k, E);
  const bool rows = !small && rows_path(f);
  // gather_rows: the (first) grouped GEMM gathers its routed rows from the
  // token-major activations, so no expert-compact copy is written
  const bool gather = forward_gathers(f);
  if (small) {
    // small batch: route, then quantise + layout + gather in one kernel
    e = launch_route(logits, M, E, k, f->softcap, f->renorm, ids, wts, stream, false);
  } else {
    e = launch_route_rank(logits, M, E, k, f->softcap, f->renorm, ids, wts, bm, counts, offsets,
                          tile_off, ctrl, reinterpret_cast<int32_t*>(ws + L.local_rank),
                          reinterpret_cast<int32_t*>(ws + L.cta_hist),
                          reinterpret_cast<int32_t*>(ws + L.cta_base), stream, false);
  }
  Placement pl;  // large batches: the gather kernels place the routes
  if (!small) {
    pl.ids = ids;
    pl.local_rank = reinterpret_cast<const int32_t*>(ws + L.local_rank);
    pl.cta_base = reinterpret_cast<const int32_t*>(ws + L.cta_base);
    pl.offsets = offsets;
    pl.sorted_route_ids = sorted;
    pl.E = E;
  }
  if (e != cudaSuccess) return cuda_status(e);
  if (fp8) {
    uint8_t* a_q = ws + L.a;
    float* a_s = reinterpret_cast<float*>(ws + L.a_scales);
    const bool ffn = fp8_ffn(f);
    const int cols = static_cast<int>(out_cols(f));   // zeroed accumulator width
    if (small)
      e = launch_quant_layout(x, M, K, k, E, bm, ids, a_q, a_s, acc, cols, counts, offsets,
                              sorted, slot, tile_off, ctrl, stream, pdl);
    else
      e = launch_quant_gather(x, M, K, k, slot, a_q, a_s, rows ? nullptr : acc, cols, pl, stream,
                              pdl, gather);
    if (e != cudaSuccess) return cuda_status(e);
    moe_gemm_args g;
    std::memset(&g, 0, sizeof(g));
    g.dtype = MOE_DTYPE_FP8_E4M3;
    g.sched = f->sched;
    g.cta_pairs = f->cta_pairs;
    g.block_m = bm;
    g.E = E;
    g.K = K;
    g.R = R;
    g.M = M;
    g.top_k = k;
    g.a = a_q;
    g.a_scales = a_s;
    g.w = f->w;
    g.w_scales = f->w_scales;
    g.offsets = offsets;
    g.tile_offsets = tile_off;
    g.sorted_route_ids = sorted;
    g.route_weights = wts;
    g.gather_rows = gather ? 1 : 0;
    moe_status_t s;
    if (ffn) {
      // up projection (gate and up tiles) with the SwiGLU + 1x128
      // re-quantisation in its epilogue: h's codes and block scales, which the
      // down projection then reads like activations
      uint8_t* h_q = ws + L.hq;
      float* h_s = reinterpret_cast<float*>(ws + L.hs);
      g.epilogue = MOE_EPI_SWIGLU;
      g.N = 2 * N;
      g.out = h_q;
      g.out_scales = h_s;
      g.k_splits = 1;
      s = run_gemm(&g, ctrl, false, stream, pdl);
      if (s != MOE_OK) return s;
      g.out_scales = nullptr;
      g.gather_rows = 0;
      g.N = K;
      g.K = N;
      g.a = h_q;
      g.a_scales = h_s;
      g.w = f->w2;
      g.w_scales = f->w2_scales;
    } else {
      g.N = N;
    }
    g.epilogue = rows ? MOE_EPI_STORE_BF16 : MOE_EPI_SCATTER;
    g.out = acc;
    g.k_splits = rows ? 1 : f->k_splits;
    s = run_gemm(&g, ctrl, ffn, stream, pdl);
    if (s != MOE_OK) return s;
    if (rows)
      return cuda_status(launch_reduce_rows(acc, slot, wts, M, cols, k, out, device_sms(), stream,
                                            pdl));
    return cuda_status(launch_finalize(acc, out, static_cast<size_t>(M) * cols, device_sms(),
                                       stream, pdl));
  }
  // BF16 gated FFN: (route + rank above) -> gather, placing the routes -> up (SwiGLU)
  // -> down (scatter-add, or bf16 rows) -> finalize (or weighted row reduction)
  void* a = ws + L.a;
  void* h = ws + L.h;
  if (gather)
    e = launch_place_routes(M, k, slot, rows ? nullptr : acc, K, pl, stream, pdl);
  else
    e = launch_gather_rows_bf16(x, M, K, k, slot, a, rows ? nullptr : acc, K, pl, stream, pdl);
  if (e != cudaSuccess) return cuda_status(e);
  moe_gemm_args g;
  std::memset(&g, 0, sizeof(g));
  g.dtype = MOE_DTYPE_BF16;
  g.epilogue = MOE_EPI_SWIGLU;
  g.sched = f->sched;
  g.cta_pairs = f->cta_pairs;
  g.block_m = bm;
  g.E = E;
  g.N = 2 * N;
  g.K = K;
  g.R = R;
  g.M = M;
  g.top_k = k;
  g.a = gather ? x : a;
  g.w = f->w;
  g.offsets = offsets;
  g.tile_offsets = tile_off;
  g.sorted_route_ids = sorted;
  g.out = h;
  g.k_splits = 1;
  g.gather_rows = gather ? 1 : 0;
  moe_status_t s = run_gemm(&g, ctrl, false, stream, pdl);
  if (s != MOE_OK) return s;
  g.gather_rows = 0;
  g.epilogue = rows ? MOE_EPI_STORE_BF16 : MOE_EPI_SCATTER;
  g.N = K;
  g.K = N;
  g.a = h;
  g.w = f->w2;
  g.sorted_route_ids = sorted;
  g.route_weights = wts;
  g.out = acc;
  s = run_gemm(&g, ctrl, true, stream, pdl);
  if (s != MOE_OK) return s;
  if (rows)
    return cuda_status(launch_reduce_rows(acc, slot, wts, M, K, k, out, device_sms(), stream, pdl));
  return cuda_status(launch_finalize(acc, out, static_cast<size_t>(M) * K, device_sms(), stream,
                                     pdl));
}

// ---------------------------------------------------------------------------
// Graph cache: one instantiated graph per (arguments, pointers, stream).
struct GraphEntry {
  moe_forward_args args;
  const float* logits;
  const void* x;
  void* out;
  void* ws;
  int device;
  cudaGraphExec_t exec;
};
constexpr int kGraphCache = 32;
GraphEntry g_graphs[kGraphCache];
int g_graph_count = 0, g_graph_next = 0;
cudaStream_t g_capture_stream[64] = {};
std::mutex g_graph_mu;

bool same_entry(const GraphEntry& g, const moe_forward_args* f, const float* logits, const void* x,
                void* out, void* ws, int dev) {
  return std::memcmp(&g.args, f, sizeof(*f)) == 0 && g.logits == logits && g.x == x &&
         g.out == out && g.ws == ws && g.device == dev;
}

moe_status_t forward_impl(const moe_forward_args* f, const float* logits, const void* x, void* out,
                          void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status_t s = check_forward(f);
  if (s != MOE_OK) return s;
  if (logits == nullptr || x == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(f).total) return MOE_ERR_WORKSPACE;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  moe_status_t cs = cuda_status(cudaStreamIsCapturing(stream, &cap));
  if (cs != MOE_OK) return cs;
  if (!f->use_graph || cap != cudaStreamCaptureStatusNone)
    return enqueue_forward(f, logits, x, out, w8, stream);

  int dev = 0;
  cs = cuda_status(cudaGetDevice(&dev));
  if (cs != MOE_OK) return cs;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_graph_mu);
  for (int i = 0; i < g_graph_count; ++i) {
    if (same_entry(g_graphs[i], f, logits, x, out, ws, dev))
      return cuda_status(cudaGraphLaunch(g_graphs[i].exec, stream));
  }
  // host-side queries the launches make once per device, kept out of the capture
  gemm_cta2_max_clusters();
  // The launch sequence is recorded on a private stream (the caller's may be
  // the legacy default stream, which cannot be captured); the graph itself
  // is then launched on the caller's stream.
  if (g_capture_stream[dev] == nullptr) {
    cs = cuda_status(cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking));
    if (cs != MOE_OK) return cs;
  }
  cudaStream_t cap_stream = g_capture_stream[dev];
  cudaGraph_t graph = nullptr;
  cs = cuda_status(cudaStreamBeginCapture(cap_stream, cudaStreamCaptureModeThreadLocal));
  if (cs != MOE_OK) return cs;
  moe_status_t es = enqueue_forward(f, logits, x, out, w8, cap_stream);
  cudaError_t ce = cudaStreamEndCapture(cap_stream, &graph);
  if (es != MOE_OK) {
    if (graph) cudaGraphDestroy(graph);
    return es;
  }
  cs = cuda_status(ce);
  if (cs != MOE_OK) return cs;
  cudaGraphExec_t exec = nullptr;
  ce = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  cs = cuda_status(ce);
  if (cs != MOE_OK) return cs;
  GraphEntry& slot = g_graphs[g_graph_next];
  if (g_graph_count == kGraphCache) cudaGraphExecDestroy(slot.exec);
  slot.args = *f;
  slot.logits = logits;
  slot.x = x;
  slot.out = out;
  slot.ws = ws;
  slot.device = dev;
  slot.exec = exec;
  g_graph_next = (g_graph_next + 1) % kGraphCache;
  if (g_graph_count < kGraphCache) ++g_graph_count;
  return cuda_status(cudaGraphLaunch(exec, stream));
}

// ---------------------------------------------------------------------------
// Scratch of moe_grouped_gemm_noalloc: the grouped GEMM's control block (tile
// queue counters and status word) in a file-scope device array instead of a
// caller workspace.  Every GPU that loads this library holds these 256 bytes
// until the process exits.  Host code must not pass the symbol itself to a
// kernel (on the host it only stands for the device variable); the device
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];
static_assert(MOE_NOALLOC_SCRATCH_BYTES >= sizeof(Ctrl), "the scratch holds one control block");
void* g_noalloc_addr[64] = {};
std::mutex g_noalloc_mu;

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_DEVICE_FAULT: return "invalid data found on the device";
  }
  return "unknown status";
}

int moe_num_sms(void) {
  gemm_cta2_max_clusters();   // cached per device, outside any capture
  return device_sms();
}

int moe_gemm_cta_pairs(void) { return gemm_cta2_max_clusters(); }

const char* moe_last_cuda_error(void) { return g_last_error; }

moe_status_t moe_route(const float* logits, int M, int E, int top_k, float softcap, int renorm,
                       int32_t* ids, float* weights, void* stream) {
  if (logits == nullptr || ids == nullptr || weights == nullptr) return MOE_ERR_INVALID_ARG;
  if (M <= 0 || E <= 0 || top_k <= 0 || !(softcap >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || top_k > 32 || top_k > E) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_route(logits, M, E, top_k, softcap, renorm, ids, weights,
                                  static_cast<cudaStream_t>(stream), false));
}

moe_status_t moe_layout(const int32_t* ids, int M, int E, int top_k, int block_m, int32_t* counts,
                        int32_t* offsets, int32_t* sorted_route_ids, int32_t* route_slot,
                        int32_t* tile_offsets, void* ws, void* stream) {
  if (ids == nullptr || counts == nullptr || offsets == nullptr || sorted_route_ids == nullptr ||
      route_slot == nullptr || tile_offsets == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (M <= 0 || E <= 0 || top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (block_m < 16 || block_m > 256 || block_m % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(M) * top_k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_layout(ids, M * top_k, E, block_m, counts, offsets, sorted_route_ids,
                                   route_slot, tile_offsets, static_cast<Ctrl*>(ws),
                                   static_cast<cudaStream_t>(stream), false));
}

moe_status_t moe_quant_gather(const void* x, int M, int K, int top_k, const int32_t* route_slot,
                              uint8_t* a_q, float* a_scales, float* zero_acc, int zero_cols,
                              void* stream) {
  if (x == nullptr || route_slot == nullptr || a_q == nullptr || a_scales == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 128 != 0 || K > 16384 || top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(a_q)) return MOE_ERR_INVALID_ARG;
  if (zero_acc != nullptr && (zero_cols <= 0 || zero_cols % 4 != 0 || !aligned16(zero_acc)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant_gather(x, M, K, top_k, const_cast<int32_t*>(route_slot), a_q,
                                         a_scales, zero_acc, zero_cols, Placement(),
                                         static_cast<cudaStream_t>(stream), false));
}

moe_status_t moe_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales,
                              void* stream) {
  if (gu == nullptr || h_q == nullptr || h_scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (R <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(gu) || !aligned16(h_q) || (reinterpret_cast<uintptr_t>(h_scales) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_swiglu_quant(gu, R, I, h_q, h_scales, device_sms(),
                                         static_cast<cudaStream_t>(stream), false));
}

moe_status_t moe_grouped_gemm(const moe_gemm_args* args, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = check_gemm(args);
  if (s != MOE_OK) return s;
  if (ws == nullptr || ws_bytes < MOE_CTRL_BYTES || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  return run_gemm(args, static_cast<Ctrl*>(ws), false, static_cast<cudaStream_t>(stream), false);
}

moe_status_t moe_scatter(const float* rows, const int32_t* route_slot, const float* weights, int M,
                         int N, int top_k, void* out, void* ws, void* stream) {
  if (rows == nullptr || route_slot == nullptr || weights == nullptr || out == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(M) * top_k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_scatter(rows, route_slot, weights, M, N, top_k, out,
                                    static_cast<Ctrl*>(ws), static_cast<cudaStream_t>(stream)));
}

size_t moe_workspace_size(const moe_forward_args* args) {
  if (check_forward(args) != MOE_OK) return 0;
  return ws_layout(args).total;
}

moe_status_t moe_forward_plan(const moe_forward_args* args, int* block_m, int* k_splits) {
  moe_status_t s = check_forward(args);
  if (s != MOE_OK) return s;
  if (block_m == nullptr || k_splits == nullptr) return MOE_ERR_INVALID_ARG;
  const bool fp8 = args->dtype == MOE_DTYPE_FP8_E4M3;
  const int R = args->M * args->top_k;
  *block_m = args->block_m > 0 ? args->block_m : auto_block_m(fp8, R, args->E);
  *k_splits = 1;
  // the scatter-add GEMM (the gated FFN's down projection) may split K; the
  // bf16-rows form uses one split
  if (fp8 && !rows_path(args)) {
    const bool ffn = fp8_ffn(args);
    moe_gemm_args g;
    std::memset(&g, 0, sizeof(g));
    g.dtype = MOE_DTYPE_FP8_E4M3;
    g.epilogue = MOE_EPI_SCATTER;
    g.block_m = *block_m;
    g.E = args->E;
    g.N = ffn ? args->K : args->N;
    g.K = ffn ? args->N : args->K;
    g.R = R;
    g.k_splits = args->k_splits;
    const int sms = device_sms();
    *k_splits = pick_k_splits(&g, sms > 0 ? sms : 148, g.K / 128);
  }
  return MOE_OK;
}

moe_status_t moe_forward_workspace_map(const moe_forward_args* args, moe_workspace_map* map) {
  moe_status_t s = check_forward(args);
  if (s != MOE_OK) return s;
  if (map == nullptr) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(args);
  const bool fp8 = args->dtype == MOE_DTYPE_FP8_E4M3;
  const bool gather = forward_gathers(args);
  const int R = args->M * args->top_k;
  map->ids = L.ids;
  map->weights = L.weights;
  map->counts = L.counts;
  map->offsets = L.offsets;
  map->tile_offsets = L.tile_off;
  map->sorted_route_ids = L.sorted;
  map->route_slot = L.slot;
  map->a = (gather && !fp8) ? MOE_WS_NONE : L.a;
  map->a_scales = fp8 ? L.a_scales : MOE_WS_NONE;
  map->h_q = fp8_ffn(args) ? L.hq : MOE_WS_NONE;
  map->h_scales = fp8_ffn(args) ? L.hs : MOE_WS_NONE;
  map->a_rows = gather ? args->M : R;
  map->block_m = args->block_m > 0 ? args->block_m : auto_block_m(fp8, R, args->E);
  return MOE_OK;
}

moe_status_t moe_forward(const moe_forward_args* args, void* out, void* ws, size_t ws_bytes,
                         void* stream) {
  if (args == nullptr) return MOE_ERR_INVALID_ARG;
  return forward_impl(args, args->logits, args->x, out, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

// Largest input (logits + activations) and output of moe_forward_host that
// its kernels access in host memory directly.
constexpr size_t kDirectHostBytes = 32u << 20;

// The device address of a pinned, device-mapped host buffer; nullptr for any
// other pointer (pageable host memory, device memory, an error).
const void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

moe_status_t moe_forward_host(const moe_forward_args* args, const float* host_logits,
                              const void* host_x, void* host_out, void* ws, size_t ws_bytes,
                              void* stream) {
  moe_status_t s = check_forward(args);
  if (s != MOE_OK) return s;
  if (host_logits == nullptr || host_x == nullptr || host_out == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(args);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const size_t M = args->M;
  const size_t cols = static_cast<size_t>(out_cols(args));
  const size_t logits_bytes = M * args->E * 4, x_bytes = M * args->K * 2;
  const size_t out_bytes = M * cols * 2;
  // Pinned (device-mapped) host buffers of a small forward: its kernels read
  // the logits and activations and write the result over the host link
  // themselves (only plain loads and stores touch them), so the step needs no
  // staging copies and their latency; otherwise copy in and out through the
  // workspace's staging buffers.
  if (args->gather_rows == 0 && logits_bytes + x_bytes <= kDirectHostBytes &&
      out_bytes <= kDirectHostBytes) {
    const void* dl = device_view(host_logits);
    const void* dx = device_view(host_x);
    void* dout = const_cast<void*>(device_view(host_out));
    if (dl != nullptr && dx != nullptr && dout != nullptr)
      return forward_impl(args, static_cast<const float*>(dl), dx, dout, ws, ws_bytes, st);
  }
  if (cudaMemcpyAsync(w8 + L.st_logits, host_logits, logits_bytes, cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(w8 + L.st_x, host_x, M * args->K * 2, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  s = forward_impl(args, reinterpret_cast<const float*>(w8 + L.st_logits), w8 + L.st_x,
                   w8 + L.st_out, ws, ws_bytes, st);
  if (s != MOE_OK) return s;
  return cuda_status(
      cudaMemcpyAsync(host_out, w8 + L.st_out, out_bytes, cudaMemcpyDeviceToHost, st));
}

moe_status_t moe_get_error(void* ws, moe_status_t* status, void* stream) {
  if (ws == nullptr || status == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  Ctrl* c = static_cast<Ctrl*>(ws);
  if (cudaMemcpy(&v, &c->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(&c->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *status = static_cast<moe_status_t>(v);
  return MOE_OK;
}

moe_status_t moe_grouped_gemm_noalloc(const moe_gemm_args* args, void* stream) {
  moe_status_t s = check_gemm(args);
  if (s != MOE_OK) return s;
  int dev = 0;
  s = cuda_status(cudaGetDevice(&dev));
  if (s != MOE_OK) return s;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
      // first call on this device: look up the device address of the array
      s = cuda_status(cudaGetSymbolAddress(&g_noalloc_addr[dev], g_noalloc_scratch));
      if (s != MOE_OK) return s;
    }
    scratch = g_noalloc_addr[dev];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The counters must start at zero; the previous call's contents are still there.
  s = cuda_status(cudaMemsetAsync(scratch, 0, MOE_NOALLOC_SCRATCH_BYTES, st));
  if (s != MOE_OK) return s;
  return run_gemm(args, static_cast<Ctrl*>(scratch), false, st, false);
}

moe_status_t moe_debug_set_pipeline_fault(int drop_producer, uint64_t timeout_ns) {
  g_drop_producer = drop_producer ? 1 : 0;
  g_timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
  return MOE_OK;
}

}  // extern "C"
