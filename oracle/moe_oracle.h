/*
 * Oracle for the fused MoE forward — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the fused MoE forward
 * computes, written to be checked by eye against the source pages:
 *
 *   [P1] "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)" (Croqtile tutorial):
 *        section "Pipeline overview" (the route -> count/build layout -> QSG ->
 *        grouped GEMM -> scatter graph), section "Baseline: 7 kernels" items 1-7,
 *        section "Fusion 1 / Fusion 2 / Fusion 3" listings (what each stage reads
 *        and writes), and the problem table (FP8 E4M3, 128x128 blocks).
 *   [P2] "H200 MoE Grouped GEMM: accounting fix, online replay, SM90 tuning":
 *        section 4 "Routed-row accounting" (compact rows) and section
 *        "3. Benchmark design" of the config-tuning part (H=3072, I=1536, E=16,
 *        top-8, gated up projection and down projection timed separately).
 *   [P3] Blog retelling of the "Weave" paper: section 4.3 "load-balancing code
 *        and task-queue generation" (histogram -> prefix -> per-expert tiles).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may
 * load this library.  It shares no code with the CUDA path: the router
 * arithmetic, the E4M3 encoder, the layout and the GEMMs are all written out
 * here independently.
 *
 * Every floating-point step that must agree bit-for-bit with the device path
 * (softcap, exp, softmax weights, amax/448 scales, E4M3 codes) is written with
 * single IEEE binary32 operations (+ - * / and fused multiply-add) and built
 * with -ffp-contract=off so the compiler cannot fuse or reorder them.
 * Everything that only has to be close (the GEMM, the SwiGLU, the scatter)
 * is computed in binary64.
 *
 * Thread arguments only split independent output rows across std::threads;
 * the value of every output element is computed by the same sequence of
 * operations regardless of the thread count.
 */
#pragma once
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* --- scalar building blocks (exported so the pins can test them) --- */

/* exp(x) by Cody-Waite reduction x = n*ln2 + r and a degree-7 Taylor
 * polynomial in r evaluated by Horner's rule with fma; result = p * 2^n.
 * x < -87 returns 0, x > 88 returns +inf. */
float oracle_exp_spec(float x);

/* tanh(t): odd Taylor series to degree 17 for |t| < 0.5 (Horner in t^2 with
 * fma, then a + (a*t^2)*q), 1 - 2/(exp_spec(2|t|) + 1) for 0.5 <= |t| < 10,
 * and 1 beyond; the sign of t is restored. */
float oracle_tanh_spec(float t);

/* OCP E4M3 ("E4M3FN": bias 7, max 448, no infinities) encoder with
 * round-to-nearest-even and saturation of finite overflow to +-448. */
uint8_t oracle_e4m3_encode(float v);

/* Exact value of an E4M3 code (NaN codes decode to NaN). */
double oracle_e4m3_decode(uint8_t code);

/* Round a binary64 value to bfloat16 (round to nearest even); returns the bits. */
uint16_t oracle_bf16_round(double v);

/* Element-wise array forms of the three scalar functions above (used by the
 * pins to sweep large input sets). */
void oracle_exp_spec_array(const float* x, int64_t n, float* y);
void oracle_tanh_spec_array(const float* x, int64_t n, float* y);
void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* y);

/* --- pipeline steps --- */

/* Route ([P1] "Baseline: 7 kernels" item 1): z = c*tanh(x/c) (c = 0: z = x),
 * top-k of z ordered by (z descending, expert id ascending), then
 * renorm=1: w_j = exp(z_j - z_max) / sum over the k selected (left fold in
 *           selection order);
 * renorm=0: w_j = exp(z_j - z_max) / sum over all E experts (left fold in
 *           expert-id order).
 * logits [M,E] f32 row-major; ids/weights [M,k]. */
void oracle_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                  int32_t* ids, float* weights);

/* Count + build layout ([P1] "Fusion 3", [P3] section 4.3):
 * counts[E]; offsets[E+1] exclusive prefix; sorted_route_ids[R] stable
 * permutation (routes of expert e in ascending route id t*k+j);
 * route_slot[R] its inverse; tile_offsets[E+1] exclusive prefix of
 * ceil(counts[e]/block_m).  Returns 0, or -1 if an id is out of range. */
int oracle_layout(const int32_t* ids, int M, int E, int k, int block_m,
                  int32_t* counts, int32_t* offsets, int32_t* sorted_route_ids,
                  int32_t* route_slot, int32_t* tile_offsets);

/* Quantise + gather ([P1] "Baseline" item 4 and "Fusion 2"): per token and
 * 1x128 block, amax = max|x|, s = amax/448, q = E4M3(x * (1/s)); amax = 0
 * gives s = 0 and zero codes.  The token's row is written to each of its k
 * slots; a_scales is [K/128, R] (block-major, slots contiguous).
 * x is bf16 bits [M,K]. */
void oracle_quant_gather(const uint16_t* x_bf16, int M, int K, int k,
                         const int32_t* route_slot, uint8_t* a_q, float* a_scales);

/* Blockwise-scaled FP8 grouped GEMM ([P1] "Baseline" item 6) in binary64:
 * Y[s,n] = sum_b sa[b,s] * sb[e,n/128,b] * sum_{k in block b} dq(a[s,k]) dq(w[e,n,k])
 * for every slot s of expert e.  Rows whose row_mask entry is 0 are skipped
 * (row_mask may be NULL = all rows).  Y is [R,N] binary64. */
void oracle_grouped_gemm_fp8(const uint8_t* a_q, const float* a_scales, int R, int K,
                             const uint8_t* w_q, const float* w_scales, int E, int N,
                             const int32_t* offsets, const uint8_t* row_mask,
                             int threads, double* Y);

/* Weighted scatter-add ([P1] "Baseline" item 7):
 * out[t,n] = sum_j w[t,j] * Y[route_slot[t*k+j], n] (binary64, j ascending)
 * for the listed tokens; out is [n_tokens, N]. */
void oracle_scatter(const double* Y, const int32_t* route_slot, const float* weights,
                    int N, int k, const int32_t* tokens, int n_tokens, double* out);

/* Full FP8 forward: route -> layout -> quantise/gather -> grouped GEMM ->
 * scatter, returning the intermediates and binary64 outputs for the listed
 * tokens (tokens = NULL, n_tokens = M for all).  block_m only shapes
 * tile_offsets. */
void oracle_forward_fp8(const float* logits, const uint16_t* x_bf16,
                        const uint8_t* w_q, const float* w_scales,
                        int M, int K, int N, int E, int k, float softcap, int renorm,
                        int block_m, const int32_t* tokens, int n_tokens, int threads,
                        int32_t* ids, float* weights, int32_t* counts, int32_t* offsets,
                        int32_t* sorted_route_ids, int32_t* route_slot,
                        int32_t* tile_offsets, uint8_t* a_q, float* a_scales,
                        double* out);

/* Independent token-major dense check: for each listed token,
 * out[t,n] = sum_j w[t,j] * sum_b sa_t[b] sb[e_j,n/128,b] sum_k dq(q_t[k]) dq(w[e_j,n,k])
 * where (q_t, sa_t) is the token's own quantised row; no layout involved. */
void oracle_dense_fp8(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                      const uint8_t* w_q, const float* w_scales,
                      int M, int K, int N, int E, int k,
                      const int32_t* tokens, int n_tokens, int threads, double* out);

/* BF16 gated FFN ([P2] config-tuning section 3: gated up projection, then down
 * projection).  W_up [E, 2I, H] with rows [0,I) = gate and [I,2I) = up;
 * W_dn [E, H, I].  For each listed token t and each of its k routes:
 *   g = x_t W_gate^T, u = x_t W_up^T (binary64), h = bf16_round(silu(g) * u),
 *   y = h W_dn^T (binary64);  out[t] = sum_j w[t,j] y_j.
 * silu(g) = g / (1 + exp(-g)) in binary64. */
void oracle_ffn_bf16(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                     const uint16_t* w_up, const uint16_t* w_dn,
                     int T, int H, int I, int E, int k,
                     const int32_t* tokens, int n_tokens, int threads, double* out);

/* --- FP8 gated FFN: the two-layer expert MLP (gate+up projection, SiLU,
 * down projection) that "Fused MoE FP8" compares against in its closing
 * section "Reference: vLLM full MLP", in the shape of [P2]'s config-tuning
 * section 3, with both projections in the FP8 format of [P1] "Baseline"
 * item 6.  The pages do not say how h enters an FP8 GEMM; the reading taken
 * is the plainest one the rest supports: h gets the same 1x128 amax/448 rule
 * as the activations (item 4), decided in binary32, the precision the up
 * projection accumulates in. --- */

/* silu(g) * u in binary32 operations: e = exp_spec(-g), d = 1 + e,
 * silu = g / d, result = silu * u. */
float oracle_swiglu_f32(float g, float u);

/* For every row s of gu (f32 [R, 2I]: gate columns [0,I), up columns
 * [I,2I)): h[r] = oracle_swiglu_f32(gu[s,r], gu[s,I+r]), then the 1x128 rule
 * of [P1] item 4 on h: h_q u8 [R, I], h_scales f32 [I/128, R] (block-major,
 * like a_scales).  I a multiple of 128. */
void oracle_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales);

/* Token-major FP8 gated FFN.  x bf16 [T,H] is quantised per token (item 4);
 * for each of the token's routes j (expert e):
 *   gu[r] = binary32( sum_b sa[b] wup_s[e,r/128,b] sum_{c in b} dq(q[c]) dq(wup_q[e,r,c]) ),
 *           r in [0, 2I) (rows [0,I) gate, [I,2I) up; the sum in binary64),
 *   (qh, sh) = oracle_swiglu_quant(gu),
 *   y[n] = sum_b sh[b] wdn_s[e,n/128,b] sum_{c in b} dq(qh[c]) dq(wdn_q[e,n,c])  (binary64),
 * and out[t] = sum_j w[t,j] y_j (binary64, j ascending).
 * wup_q u8 [E,2I,H], wup_s f32 [E,2I/128,H/128]; wdn_q u8 [E,H,I],
 * wdn_s f32 [E,H/128,I/128]; H and I multiples of 128. */
void oracle_ffn_fp8(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                    const uint8_t* wup_q, const float* wup_s, const uint8_t* wdn_q,
                    const float* wdn_s, int T, int H, int I, int E, int k,
                    const int32_t* tokens, int n_tokens, int threads, double* out);

#ifdef __cplusplus
}
#endif
