/*
 * moe.h — C ABI of the GB300 (sm_103a) fused Mixture-of-Experts forward.
 *
 * The forward routes each token to top_k experts, lays the routed rows out
 * expert by expert, quantises them blockwise to FP8 E4M3 (or keeps them in
 * BF16), multiplies them by the experts' weights in one grouped GEMM and adds
 * the routing-weighted results back into token order.  The steps and their
 * data follow "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)" (section
 * "Pipeline overview" and section "Baseline: 7 kernels", items 1-7); the BF16
 * gated FFN follows the benchmark design (section 3) of "H200 MoE Grouped
 * GEMM: accounting fix, online replay, SM90 tuning"; the persistent tile queue
 * follows section 2.2 of the blog retelling of "Weave".
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, owned by the caller, row-major,
 *    and 16-byte aligned unless stated otherwise ("host" pointers are named so).
 *    The library never allocates device memory in these calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous: they enqueue work and return.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    returned synchronously (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE).  Launch failures return MOE_ERR_CUDA.
 *  - Errors found on the device (an expert id out of range, a pipeline wait
 *    that timed out) are recorded in a status word inside the caller's
 *    workspace (first error wins) and read back with moe_get_error().
 *  - Supported sizes: 1 <= top_k <= min(E, 32); E <= 1024; K % 128 == 0 and
 *    N % 128 == 0 on the FP8 path; K % 64 == 0 and N % 128 == 0 on the BF16
 *    path; M * top_k < 2^31.
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad enum */
  MOE_ERR_UNSUPPORTED = 2,   /* size outside the supported set above */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 5,       /* device: a pipeline wait gave up (no GPU hang) */
  MOE_ERR_DEVICE_FAULT = 6   /* device: invalid data (e.g. expert id >= E) */
} moe_status_t;

typedef enum { MOE_DTYPE_FP8_E4M3 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype_t;

typedef enum {
  MOE_EPI_SCATTER = 0,  /* out f32 [M,N] += route_weight * row   (weighted scatter-add) */
  MOE_EPI_STORE = 1,    /* out f32 [R,N]  = row                   (expert-compact rows) */
  MOE_EPI_SWIGLU = 2,   /* h = silu(gate) * up; weight rows [0,N/2) gate, [N/2,N) up.
                           BF16: out bf16 [R,N/2] = h.  FP8: h in binary32 as moe_swiglu_quant
                           computes it from the fp32 accumulators, re-quantised by the 1x128
                           rule: out u8 [R,N/2] E4M3 codes, out_scales f32 [N/256,R]
                           (N % 256 == 0) */
  MOE_EPI_STORE_BF16 = 3 /* out bf16 [R,N] = bf16(row)            (expert-compact rows; the
                            forward's large-batch path reduces them with the route weights
                            afterwards instead of scatter-adding into an fp32 accumulator) */
} moe_epilogue_t;

typedef enum {
  MOE_SCHED_QUEUE = 0,  /* persistent CTAs pull tiles from one atomic counter */
  MOE_SCHED_STATIC = 1  /* persistent CTAs statically partitioned over experts */
} moe_sched_t;

/* Bytes of the control block (status word and tile-queue counters) that
 * every workspace starts with.  A fresh workspace must have this block
 * zeroed once (cudaMemset) before its first use. */
#define MOE_CTRL_BYTES 256

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t s);

/* Number of streaming multiprocessors of the current device (0 on error). */
int moe_num_sms(void);

/* Clusters of two CTAs that can be resident at once on the current device
 * for the grouped GEMMs whose tiles are each computed by a CTA pair (tcgen05
 * MMAs with M = 256 spanning both SMs): FP8 SCATTER at block_m 128 with N a
 * multiple of 256 (256 weight rows x 128 routed rows per tile), FP8 SWIGLU at
 * block_m 128 (256 routed rows x the gate and up rows of 128 h columns), BF16
 * SCATTER and STORE_BF16 at block_m 256 with N a multiple of 256 (256 weight
 * rows x 256 routed rows), BF16 SWIGLU at block_m 256 (as the FP8 SWIGLU
 * form, accumulated over all of K).  0: that form is unavailable (or on error) and those
 * GEMMs run the single-CTA form.  The grid of such a GEMM is the even number of
 * CTAs min(num_ctas or the SM count, 2 x this). */
int moe_gemm_cta_pairs(void);

/* Name and text of the CUDA error behind the calling thread's most recent
 * MOE_ERR_CUDA ("" if none); a static per-thread buffer. */
const char* moe_last_cuda_error(void);

/* Route — "Fused MoE FP8" section "Baseline: 7 kernels", item 1.
 * For each token t: z_e = softcap * tanh(logits[t,e] / softcap) (softcap == 0:
 * z_e = logits[t,e]); the top_k experts by (z descending, expert id
 * ascending) are written to ids[t, 0..top_k) in that order; weights are
 * renorm = 1: exp(z_j - z_0) / sum over the selected j (sum in selection order),
 * renorm = 0: exp(z_j - z_0) / sum over all E experts (sum in expert-id order).
 * exp and tanh are evaluated by a fixed sequence of IEEE binary32 operations
 * (Cody-Waite exp with a degree-7 Taylor polynomial; tanh by its degree-17
 * Taylor series below |t| = 0.5, else 1 - 2/(exp(2|t|) + 1)), so results are
 * reproducible bit for bit.
 * logits: f32 [M,E]; ids: s32 [M,top_k]; weights: f32 [M,top_k]. */
moe_status_t moe_route(const float* logits, int M, int E, int top_k, float softcap,
                       int renorm, int32_t* ids, float* weights, void* stream);

/* Count + build layout — "Fused MoE FP8" section "Fusion 3" (counts and the
 * exclusive prefix) and section 4.3 of the Weave retelling (per-expert tiles).
 * R = M*top_k routes, route r = t*top_k + j.  Writes
 *   counts[E]            routes per expert,
 *   offsets[E+1]         exclusive prefix of counts (offsets[E] = R),
 *   sorted_route_ids[R]  routes grouped by expert, ascending route id inside
 *                        each expert (a deterministic, stable layout),
 *   route_slot[R]        inverse permutation (slot of each route),
 *   tile_offsets[E+1]    exclusive prefix of ceil(counts[e] / block_m).
 * ids: s32 [M,top_k].  ws: a workspace whose control block receives the
 * status (MOE_ERR_DEVICE_FAULT if an id is outside [0,E)) and whose tile
 * queue counter is reset.  block_m in [16,256], a multiple of 16. */
moe_status_t moe_layout(const int32_t* ids, int M, int E, int top_k, int block_m,
                        int32_t* counts, int32_t* offsets, int32_t* sorted_route_ids,
                        int32_t* route_slot, int32_t* tile_offsets, void* ws, void* stream);

/* Quantise + sort/gather — "Fused MoE FP8" section "Baseline: 7 kernels"
 * item 4 and section "Fusion 2" (QSG).  Per token t and 1x128 block b:
 * amax = max |x|, s = amax / 448, q = E4M3_rne_satfinite(x * (1/s)) (amax = 0:
 * s = 0 and q = 0).  The token's codes go to every slot route_slot[t*top_k+j];
 * a_scales is stored block-major: a_scales[b*R + slot] = s.
 * x: bf16 [M,K]; a_q: u8 [R,K]; a_scales: f32 [K/128, R].
 * zero_acc (optional, may be NULL): f32 [M, zero_cols] set to 0 in the same
 * pass (the fused output memset of section "Fused Memset"). */
moe_status_t moe_quant_gather(const void* x, int M, int K, int top_k,
                              const int32_t* route_slot, uint8_t* a_q, float* a_scales,
                              float* zero_acc, int zero_cols, void* stream);

/* Arguments of one grouped GEMM launch (see moe_grouped_gemm). */
typedef struct {
  moe_dtype_t dtype;          /* FP8_E4M3 (blockwise scales) or BF16 */
  moe_epilogue_t epilogue;    /* SCATTER, STORE, SWIGLU or STORE_BF16 */
  moe_sched_t sched;          /* QUEUE or STATIC (CTA pairs: a fixed round-robin order) */
  int block_m;                /* routed rows per tile: 16..256, multiple of 16
                                 (FP8: at most 128) */
  int E, N, K;                /* weights are [E, N, K] */
  int R;                      /* rows of `a` (M * top_k) */
  int M, top_k;               /* SCATTER only: output rows and routes per token */
  const void* a;              /* [R, K] e4m3 or bf16, expert-compact rows */
  const float* a_scales;      /* FP8: [K/128, R] */
  const void* w;              /* [E, N, K] e4m3 or bf16 */
  const float* w_scales;      /* FP8: [E, N/128, K/128] (one scale per 128x128 block) */
  const int32_t* offsets;     /* [E+1] first slot of each expert */
  const int32_t* tile_offsets;/* [E+1] prefix of ceil(count/block_m), same block_m */
  const int32_t* sorted_route_ids; /* SCATTER: [R] route of each slot */
  const float* route_weights; /* SCATTER: [M*top_k] */
  void* out;                  /* see moe_epilogue_t */
  int k_splits;               /* FP8 SCATTER: K split into this many tiles (0 = auto) */
  int num_ctas;               /* persistent CTAs (0 = one per SM).  With gather_rows 0,
                                 FP8 SCATTER (block_m 128, N a multiple of 256), FP8
                                 SWIGLU (block_m 128), BF16 SWIGLU (block_m 256) and BF16
                                 SCATTER / STORE_BF16 (block_m 256, N a multiple of 256)
                                 run clusters of two
                                 CTAs (moe_gemm_cta_pairs), each pair walking every
                                 (G/2)-th tile in a fixed order: the grid G is then
                                 num_ctas rounded down to even and capped at twice the
                                 resident pairs (num_ctas 1: single CTAs) */
  int gather_rows;            /* 0: `a` holds the expert-compact rows [R, K] (FP8 a_scales
                                 [K/128, R]).  1: `a` is token-major [M, K] and the kernel
                                 gathers compact slot s from row sorted_route_ids[s] / top_k
                                 (FP8 a_scales token-major [K/128, M]); sorted_route_ids, M
                                 and top_k are then required for every epilogue, and an
                                 empty slot (id < 0) reads row 0 (its result is dropped).
                                 Built for FP8 (STORE, STORE_BF16, SCATTER) and the BF16
                                 SWIGLU epilogue; others: MOE_ERR_UNSUPPORTED */
  float* out_scales;          /* FP8 SWIGLU only: f32 [N/256, R] block scales of h (see
                                 moe_epilogue_t); ignored otherwise */
  int cta_pairs;              /* 0: tiles on clusters of two CTAs wherever that form
                                 exists (see num_ctas and moe_gemm_cta_pairs); -1: single
                                 CTAs only.  Other values: MOE_ERR_INVALID_ARG */
} moe_gemm_args;

/* Grouped GEMM — "Fused MoE FP8" section "Baseline: 7 kernels" item 6, with
 * the weighted scatter of item 7 fused into its epilogue (section "Fusion 1").
 * For every slot s of expert e and output column n:
 *   FP8:  Y[s,n] = sum_b a_scales[b,s] * w_scales[e,n/128,b] *
 *                  sum_{k in block b} a[s,k] * w[e,n,k]       (fp32 accumulation)
 *   BF16: Y[s,n] = sum_k a[s,k] * w[e,n,k]
 * and the epilogue stores Y (STORE; STORE_BF16 rounds it to bf16), applies
 * silu(gate)*up (SWIGLU) or adds
 * route_weights[r] * Y[s,:] to out[r / top_k, :] for r = sorted_route_ids[s]
 * (SCATTER; out must be zeroed or hold a partial sum).
 * Runs on tcgen05 tensor cores (TMEM accumulators, TMA-fed shared memory).
 * ws: workspace of at least MOE_CTRL_BYTES (tile-queue counter, status). */
moe_status_t moe_grouped_gemm(const moe_gemm_args* args, void* ws, size_t ws_bytes,
                              void* stream);

/* Standalone weighted scatter (unfused form of "Baseline: 7 kernels" item 7):
 * out[t,n] = bf16( sum_j weights[t*top_k+j] * rows[route_slot[t*top_k+j], n] )
 * with the sum in j order in fp32.  rows: f32 [M*top_k, N]; out: bf16 [M,N].
 * ws: workspace of at least MOE_CTRL_BYTES, 256-byte aligned (else
 * MOE_ERR_WORKSPACE): a route whose slot lies outside [0, M*top_k) adds nothing
 * and records MOE_ERR_DEVICE_FAULT in its status word (read with
 * moe_get_error). */
moe_status_t moe_scatter(const float* rows, const int32_t* route_slot, const float* weights,
                         int M, int N, int top_k, void* out, void* ws, void* stream);

/* SwiGLU + re-quantisation between the projections of the FP8 gated FFN (the
 * two-layer expert MLP — gate+up projection, SiLU, down projection — of "Fused
 * MoE FP8" section "Reference: vLLM full MLP", both projections FP8 as in
 * "Baseline: 7 kernels" item 6).  For every row s of gu (f32 [R, 2I], the up
 * projection's output: gate columns [0,I), up columns [I,2I)):
 *   h[r] = (g / (1 + exp(-g))) * u  with g = gu[s,r], u = gu[s,I+r], in IEEE
 *          binary32 operations (exp by the router's fixed Cody-Waite sequence),
 * then the 1x128 rule of item 4 on h: amax = max |h|, s = amax / 448,
 * h_q = E4M3_rne_satfinite(h * (1/s)) (amax = 0: s = 0, codes 0).
 * h_q: u8 [R, I]; h_scales: f32 [I/128, R] (block-major, the layout the FP8
 * grouped GEMM reads as a_scales).  I a multiple of 128, else
 * MOE_ERR_UNSUPPORTED; gu and h_q 16-byte aligned, h_scales 4-byte aligned, R > 0, else
 * MOE_ERR_INVALID_ARG.  Device pointers, caller-owned; async on `stream`. */
moe_status_t moe_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales,
                              void* stream);

/* Arguments of the fused forward. */
typedef struct {
  moe_dtype_t dtype;      /* FP8_E4M3: one grouped GEMM [E,N,K] with block scales (or,
                             with gated = 1, the FP8 gated FFN);
                             BF16: gated FFN, up [E,2N,K] + SwiGLU, down [E,K,N] */
  int M;                  /* tokens */
  int K;                  /* token feature size (the GEMM's contraction size;
                             for BF16 also the output size) */
  int N;                  /* FP8: output size; gated FFN (BF16, or FP8 with gated = 1):
                             intermediate size I */
  int E, top_k;
  float softcap;          /* 0 = off */
  int renorm;             /* 1 = softmax over the selected top_k (default) */
  const float* logits;    /* [M,E] f32 */
  const void* x;          /* [M,K] bf16 */
  const void* w;          /* FP8: e4m3 [E,N,K]; BF16: bf16 w_up [E,2N,K] (gate rows, then up rows) */
  const float* w_scales;  /* FP8: [E,N/128,K/128] */
  const void* w2;         /* BF16: bf16 w_down [E,K,N] */
  int block_m;            /* rows per tile (0 = chosen from the shape) */
  moe_sched_t sched;      /* tile scheduler of the grouped GEMMs */
  int k_splits;           /* FP8: 0 = auto */
  int use_graph;          /* 1: capture the launch sequence once per argument set and
                             replay it as a CUDA graph; 0: plain launches */
  int gather_rows;        /* large batches (more than 4096 routes, or BF16): 1 = the
                             first grouped GEMM gathers each routed row from the
                             token-major activations (moe_gemm_args.gather_rows) instead
                             of reading an expert-compact copy; the workspace then holds
                             no [R, K] copy (FP8 keeps one token-major [M, K] code matrix).
                             0 (default) = write the compact copy, which is faster on
                             GB300 at the benchmark shapes; same results either way.
                             Ignored by the FP8 gated FFN (its fused SwiGLU up
                             projection reads the compact copy) */
  int gated;              /* FP8_E4M3: 1 = gated FFN in FP8 — w = e4m3 w_up [E,2N,K] (gate
                             rows, then up rows) with w_scales [E,2N/128,K/128]; w2 = e4m3
                             w_down [E,K,N] with w2_scales [E,K/128,N/128]; h =
                             silu(gate)*up re-quantised by the 1x128 rule in the up
                             projection's epilogue (MOE_EPI_SWIGLU, FP8); output [M,K].  0 = the single FP8 GEMM.  BF16:
                             must be 0 or 1 (its forward is always the gated FFN) */
  const float* w2_scales; /* FP8 with gated = 1: [E,K/128,N/128] */
  int cta_pairs;          /* the grouped GEMMs' cta_pairs (see moe_gemm_args): 0 = CTA
                             pairs wherever that form exists, -1 = single CTAs only */
} moe_forward_args;

/* Workspace bytes needed by moe_forward / moe_forward_host for these
 * arguments (0 if the arguments are invalid). */
size_t moe_workspace_size(const moe_forward_args* args);

/* The tile rows (block_m) and FP8 K split that moe_forward uses for these
 * arguments, so a caller can reproduce its grouped GEMM with
 * moe_grouped_gemm (k_splits is 1 on the BF16 path and whenever the forward
 * stores bf16 rows instead of scatter-adding; for the FP8 gated FFN it is the
 * down projection's split, the up projection storing with one split). */
moe_status_t moe_forward_plan(const moe_forward_args* args, int* block_m, int* k_splits);

/* Offset of a buffer that the forward does not keep for these arguments. */
#define MOE_WS_NONE ((size_t)-1)

/* Where moe_forward keeps its intermediates inside the workspace: byte
 * offsets from the workspace's start.  Once a forward has completed on its
 * stream these buffers hold the results of its own steps, each in exactly
 * the form the standalone entry points define (the next forward on the same
 * workspace overwrites them):
 *   ids, weights      s32 / f32 [M, top_k]: moe_route ("Fused MoE FP8",
 *                     section "Baseline: 7 kernels", item 1);
 *   counts [E], offsets [E+1], tile_offsets [E+1] (tiles of block_m rows),
 *   sorted_route_ids [R], route_slot [R]: moe_layout (items 2-3, section
 *                     "Fusion 3"), R = M * top_k;
 *   a, a_scales       FP8: E4M3 codes u8 [a_rows, K] and scales f32
 *                     [K/128, a_rows] of moe_quant_gather (items 4-5): the
 *                     expert-compact rows (a_rows = R, row = slot) or, with
 *                     gather_rows on the large-batch path, each token once
 *                     (a_rows = M, row = token).  BF16: the expert-compact
 *                     bf16 rows [R, K] (row = slot, a copy of x's row
 *                     sorted_route_ids[slot] / top_k), a_scales MOE_WS_NONE;
 *                     a = MOE_WS_NONE when the BF16 up projection gathers
 *                     its rows itself;
 *   h_q, h_scales     FP8 gated FFN only: h's E4M3 codes u8 [R, N] and scales
 *                     f32 [N/128, R] (the moe_swiglu_quant step), else
 *                     MOE_WS_NONE;
 *   block_m           the forward's tile rows (as moe_forward_plan).
 * Host-only query; nothing is enqueued.  MOE_ERR_INVALID_ARG /
 * MOE_ERR_UNSUPPORTED as moe_workspace_size's arguments, or map == NULL. */
typedef struct {
  size_t ids, weights, counts, offsets, tile_offsets, sorted_route_ids, route_slot;
  size_t a, a_scales;
  size_t h_q, h_scales;
  int a_rows;
  int block_m;
} moe_workspace_map;

moe_status_t moe_forward_workspace_map(const moe_forward_args* args, moe_workspace_map* map);

/* Fused forward: route -> layout -> quantise+gather (FP8) or gather (BF16)
 * -> grouped GEMM(s) -> weighted scatter -> bf16 output.  The FP8 gated FFN
 * (gated = 1) runs the up projection with the FP8 SWIGLU epilogue (gate and up
 * tiles of the same 128 h columns; h re-quantised in the epilogue into codes
 * [R, N] and scales [N/128, R]), then the FP8 down projection.  While the fp32
 * output accumulator (M x out x 4 bytes) is at most 112 MiB the weighted
 * scatter is fused into the last GEMM's epilogue (fp32 reductions into the
 * accumulator, then one bf16 rounding); above that the GEMM stores each
 * routed row in bf16 and a reduction kernel sums each token's top_k rows
 * with the route weights in fp32 (in route order) before the bf16 rounding.
 * out: bf16 [M, N] (single FP8 GEMM) or [M, K] (gated FFN).  ws: device workspace of
 * moe_workspace_size() bytes, 256-byte aligned, control block zeroed once.
 * With use_graph = 1 the launch sequence is captured (on a private stream) on
 * first use for this argument set, pointers included, and the graph is
 * replayed on `stream`; when `stream` is already capturing, the kernels are
 * launched directly into the caller's capture.  Cached graphs belong to the
 * device's current context: do not use a forward with use_graph = 1 on a
 * device after cudaDeviceReset. */
moe_status_t moe_forward(const moe_forward_args* args, void* out, void* ws, size_t ws_bytes,
                         void* stream);

/* The same forward for host-resident inputs: `host_logits` (f32 [M,E]) and
 * `host_x` (bf16 [M,K]) go in, the bf16 result goes to `host_out`, all
 * enqueued on `stream`.  When all three are pinned, device-mapped host
 * buffers, the inputs total at most 32 MiB, the output at most 32 MiB and
 * gather_rows is 0, the forward's kernels read the inputs and write the
 * result in host memory directly (over the host link, no staging copies);
 * otherwise the inputs are copied into the workspace and the result out of it
 * (pinned memory makes those copies asynchronous).  args->logits and args->x
 * are ignored; the weights stay device pointers. */
moe_status_t moe_forward_host(const moe_forward_args* args, const float* host_logits,
                              const void* host_x, void* host_out, void* ws, size_t ws_bytes,
                              void* stream);

/* Waits for `stream`, reads the workspace's device status word into *status
 * and clears it. */
moe_status_t moe_get_error(void* ws, moe_status_t* status, void* stream);

/* Bytes of device memory that moe_grouped_gemm_noalloc keeps for its own use. */
#define MOE_NOALLOC_SCRATCH_BYTES 256

/* moe_grouped_gemm without a workspace.  No counterpart on the source pages:
 * this entry point exists for callers that cannot allocate device memory —
 * for example code running under an allocator or runtime that it does not
 * own, or a latency-critical thread that must not call cudaMalloc — and so
 * have no workspace to pass.
 *
 * The arguments, the computation and the output are those of
 * moe_grouped_gemm.  The kernel's scratch (its tile-queue counters and status
 * word, MOE_NOALLOC_SCRATCH_BYTES = 256 bytes) lives in a static device array
 * inside this library instead of a caller workspace; that scratch does not
 * grow with the problem, so every size moe_grouped_gemm accepts is accepted
 * (argument errors are returned exactly as moe_grouped_gemm returns them).
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process: do not call this entry point on a device after cudaDeviceReset
 *   (the reset recreates the array elsewhere).
 * - Each call clears the scratch (cudaMemsetAsync on `stream`) before its
 *   kernel, since the array keeps the previous call's contents.
 * - All calls in the process share the one array per device: calls whose
 *   work overlaps on the GPU (different streams, no ordering between them)
 *   race on the counters and give wrong results.  Order them on one stream.
 * - Device-side errors (a pipeline wait that timed out) are recorded in the
 *   scratch status word, which this entry point does not return; callers who
 *   need them use moe_grouped_gemm with a workspace and moe_get_error. */
moe_status_t moe_grouped_gemm_noalloc(const moe_gemm_args* args, void* stream);

/* Test hook for failure detection: when `drop_producer` is nonzero, the next
 * moe_grouped_gemm launches issue no loads, so every consumer wait runs into
 * its time limit of `timeout_ns` nanoseconds and the kernel exits with
 * MOE_ERR_TIMEOUT in the status word instead of hanging.  timeout_ns = 0
 * restores the default limit (2 s); drop_producer = 0 restores normal runs. */
moe_status_t moe_debug_set_pipeline_fault(int drop_producer, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
