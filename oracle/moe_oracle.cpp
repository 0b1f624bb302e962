// Oracle for the fused MoE forward — TEST INFRASTRUCTURE ONLY (see moe_oracle.h).
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread
// Parity status of each function is listed in its comment; every function here
// is pinned by a "not gpu" test against brute force, closed forms or libm.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

float bits_to_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t f32_to_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float bf16_to_f32(uint16_t h) { return bits_to_f32(uint32_t(h) << 16); }

// Constants of the router arithmetic: each is the binary32 value nearest the
// stated real number (ln2_lo is the binary32 nearest ln2 - ln2_hi).
const float kLog2e = bits_to_f32(0x3fb8aa3bu);   // 1/ln 2
const float kLn2Hi = bits_to_f32(0x3f317218u);   // ln 2
const float kLn2Lo = bits_to_f32(0xb102e308u);   // ln 2 - kLn2Hi
// Taylor coefficients 1/j! of exp, j = 0..7.
const float kExpC[8] = {bits_to_f32(0x3f800000u), bits_to_f32(0x3f800000u),
                        bits_to_f32(0x3f000000u), bits_to_f32(0x3e2aaaabu),
                        bits_to_f32(0x3d2aaaabu), bits_to_f32(0x3c088889u),
                        bits_to_f32(0x3ab60b61u), bits_to_f32(0x39500d01u)};
// Taylor coefficients of tanh for t^3, t^5, ..., t^17:
// -1/3, 2/15, -17/315, 62/2835, -1382/155925, 21844/6081075,
// -929569/638512875, 6404582/10854718875.
const float kTanhC[8] = {bits_to_f32(0xbeaaaaabu), bits_to_f32(0x3e088889u),
                         bits_to_f32(0xbd5d0dd1u), bits_to_f32(0x3cb327a4u),
                         bits_to_f32(0xbc11371bu), bits_to_f32(0x3b6b69e8u),
                         bits_to_f32(0xbabed1b2u), bits_to_f32(0x3a1aac12u)};

// Run fn(i) for i in [0, n) over `threads` workers (contiguous chunks).
void parallel_for(int n, int threads, const std::function<void(int)>& fn) {
  if (threads <= 1 || n < 2) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  threads = std::min(threads, n);
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    int lo = int((int64_t)n * w / threads), hi = int((int64_t)n * (w + 1) / threads);
    pool.emplace_back([lo, hi, &fn] { for (int i = lo; i < hi; ++i) fn(i); });
  }
  for (auto& t : pool) t.join();
}

}  // namespace

extern "C" {

float oracle_exp_spec(float x) {
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return INFINITY;
  // n = round-half-even(x * log2 e); r = x - n*ln2 in two fma steps.
  float t = x * kLog2e;
  float n = std::nearbyint(t);
  float r = std::fma(-n, kLn2Hi, x);
  r = std::fma(-n, kLn2Lo, r);
  float p = kExpC[7];
  for (int j = 6; j >= 0; --j) p = std::fma(p, r, kExpC[j]);
  int ni = int(n);                                  // in [-126, 127]
  float scale = bits_to_f32(uint32_t(ni + 127) << 23);
  return p * scale;
}

float oracle_tanh_spec(float t) {
  float a = std::fabs(t);
  float y;
  if (a >= 10.0f) {
    y = 1.0f;
  } else if (a < 0.5f) {
    float s = a * a;
    float q = kTanhC[7];
    for (int j = 6; j >= 0; --j) q = std::fma(q, s, kTanhC[j]);
    float as = a * s;
    y = std::fma(as, q, a);
  } else {
    float e = oracle_exp_spec(a + a);
    float d = e + 1.0f;
    float q = 2.0f / d;
    y = 1.0f - q;
  }
  return std::signbit(t) ? -y : y;
}

uint8_t oracle_e4m3_encode(float v) {
  // Written from the format definition: representable magnitudes are
  // m * 2^-9 for m = 0..7 (subnormals) and (8 + m) * 2^(e-10) for exponent
  // field e = 1..15, m = 0..7, except e = 15, m = 7 (NaN).  Largest: 448.
  uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(double(v));
  if (std::isnan(v)) return 0x7f;
  if (a >= 448.0) return sign | 0x7e;              // saturate finite overflow
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);                              // a = f * 2^e2, f in [0.5, 1)
  int ex = e2 - 1;                                 // floor(log2 a)
  double quantum = ex < -6 ? std::ldexp(1.0, -9) : std::ldexp(1.0, ex - 3);
  double q = std::nearbyint(a / quantum);          // a/quantum exact; ties to even
  double val = q * quantum;                        // rounded magnitude, <= 448
  if (val == 0.0) return sign;
  std::frexp(val, &e2);
  ex = e2 - 1;
  if (ex < -6) return sign | uint8_t(val / std::ldexp(1.0, -9));   // subnormal code
  int mant = int(val / std::ldexp(1.0, ex) * 8.0) - 8;
  return sign | uint8_t(((ex + 7) << 3) | mant);
}

double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = e == 0 ? std::ldexp(double(m), -9) : std::ldexp(double(8 + m), e - 10);
  return s ? -mag : mag;
}

uint16_t oracle_bf16_round(double v) {
  // bfloat16: 8 significant bits, binary32 exponent range.  Round |v| on the
  // grid 2^q with q = max(floor(log2|v|), -126) - 7, ties to even.
  if (std::isnan(v)) return 0x7fc0;
  uint16_t sign = std::signbit(v) ? 0x8000 : 0x0000;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);
  int q = std::max(e2 - 1, -126) - 7;
  double val = std::ldexp(std::nearbyint(std::ldexp(a, -q)), q);
  if (val >= std::ldexp(1.0, 128)) return sign | 0x7f80;   // overflow to infinity
  float f = float(val);                                      // exact
  return sign | uint16_t((f32_to_bits(f) >> 16) & 0x7fff);
}

void oracle_exp_spec_array(const float* x, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp_spec(x[i]);
}
void oracle_tanh_spec_array(const float* x, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_tanh_spec(x[i]);
}
void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_e4m3_encode(x[i]);
}

void oracle_route(const float* logits, int M, int E, int k, float softcap, int renorm,
                  int32_t* ids, float* weights) {
  std::vector<float> z(E);
  std::vector<int> order(E);
  for (int t = 0; t < M; ++t) {
    const float* x = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (softcap > 0.0f) {
        float u = x[e] / softcap;
        z[e] = softcap * oracle_tanh_spec(u);
      } else {
        z[e] = x[e];
      }
    }
    // top-k: (z descending, expert id ascending)
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return z[a] > z[b]; });
    float m = z[order[0]];
    float s = 0.0f;
    if (renorm) {
      for (int j = 0; j < k; ++j) s = s + oracle_exp_spec(z[order[j]] - m);
    } else {
      for (int e = 0; e < E; ++e) s = s + oracle_exp_spec(z[e] - m);
    }
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = order[j];
      weights[(size_t)t * k + j] = oracle_exp_spec(z[order[j]] - m) / s;
    }
  }
}

int oracle_layout(const int32_t* ids, int M, int E, int k, int block_m,
                  int32_t* counts, int32_t* offsets, int32_t* sorted_route_ids,
                  int32_t* route_slot, int32_t* tile_offsets) {
  const int R = M * k;
  for (int r = 0; r < R; ++r)
    if (ids[r] < 0 || ids[r] >= E) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int r = 0; r < R; ++r) counts[ids[r]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  tile_offsets[0] = 0;
  for (int e = 0; e < E; ++e)
    tile_offsets[e + 1] = tile_offsets[e] + (counts[e] + block_m - 1) / block_m;
  // Stable fill: visiting routes in ascending id keeps each expert's slots in
  // ascending route order.
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (int r = 0; r < R; ++r) {
    int slot = cursor[ids[r]]++;
    sorted_route_ids[slot] = r;
    route_slot[r] = slot;
  }
  return 0;
}

// The 1x128 block rule of "Baseline: 7 kernels" item 4 on a binary32 row:
// amax = max |v|, s = amax / 448, q = E4M3(v * (1/s)); amax = 0 gives s = 0
// and all-zero codes.
static void quantize_f32_row(const float* v, int K, uint8_t* q, float* scales) {
  for (int b = 0; b < K / 128; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 128; ++i) amax = std::max(amax, std::fabs(v[b * 128 + i]));
    if (amax == 0.0f) {
      scales[b] = 0.0f;
      for (int i = 0; i < 128; ++i) q[b * 128 + i] = 0;
      continue;
    }
    float s = amax / 448.0f;
    float inv = 1.0f / s;
    scales[b] = s;
    for (int i = 0; i < 128; ++i) q[b * 128 + i] = oracle_e4m3_encode(v[b * 128 + i] * inv);
  }
}

// bf16 rows widen to binary32 exactly, then the same rule.
static void quantize_row(const uint16_t* xrow, int K, uint8_t* q, float* scales) {
  std::vector<float> v(K);
  for (int i = 0; i < K; ++i) v[i] = bf16_to_f32(xrow[i]);
  quantize_f32_row(v.data(), K, q, scales);
}

void oracle_quant_gather(const uint16_t* x_bf16, int M, int K, int k,
                         const int32_t* route_slot, uint8_t* a_q, float* a_scales) {
  const int KB = K / 128, R = M * k;
  std::vector<uint8_t> q(K);
  std::vector<float> sc(KB);
  for (int t = 0; t < M; ++t) {
    quantize_row(x_bf16 + (size_t)t * K, K, q.data(), sc.data());
    for (int j = 0; j < k; ++j) {
      int slot = route_slot[t * k + j];
      std::memcpy(a_q + (size_t)slot * K, q.data(), K);
      for (int b = 0; b < KB; ++b) a_scales[(size_t)b * R + slot] = sc[b];
    }
  }
}

void oracle_grouped_gemm_fp8(const uint8_t* a_q, const float* a_scales, int R, int K,
                             const uint8_t* w_q, const float* w_scales, int E, int N,
                             const int32_t* offsets, const uint8_t* row_mask,
                             int threads, double* Y) {
  const int KB = K / 128, NB = N / 128;
  double dq[256];
  for (int c = 0; c < 256; ++c) dq[c] = oracle_e4m3_decode(uint8_t(c));
  std::vector<int> expert_of(R, -1);
  for (int e = 0; e < E; ++e)
    for (int s = offsets[e]; s < offsets[e + 1]; ++s) expert_of[s] = e;
  parallel_for(R, threads, [&](int s) {
    if (row_mask && !row_mask[s]) return;
    int e = expert_of[s];
    const uint8_t* a = a_q + (size_t)s * K;
    for (int n = 0; n < N; ++n) {
      const uint8_t* w = w_q + ((size_t)e * N + n) * K;
      double acc = 0.0;
      for (int b = 0; b < KB; ++b) {
        double blk = 0.0;  // exact: 128 products of E4M3 values
        for (int i = b * 128; i < b * 128 + 128; ++i) blk += dq[a[i]] * dq[w[i]];
        double sa = a_scales[(size_t)b * R + s];
        double sb = w_scales[((size_t)e * NB + n / 128) * KB + b];
        acc += sa * sb * blk;
      }
      Y[(size_t)s * N + n] = acc;
    }
  });
}

// BF16 grouped GEMM ("H200 MoE Grouped GEMM", section 4: compact routed rows;
// the gated up and down projections of its config-tuning benchmark design):
// for every slot s of expert e (offsets[e] <= s < offsets[e+1]) and output n,
// Y[s,n] = sum_k a[s,k] * w[e,n,k], the bf16 values widened exactly and the
// products and sum in binary64.
void oracle_grouped_gemm_bf16(const uint16_t* a_bf16, int R, int K, const uint16_t* w_bf16,
                              int E, int N, const int32_t* offsets, int threads, double* Y) {
  std::vector<int> expert_of(R, -1);
  for (int e = 0; e < E; ++e)
    for (int s = offsets[e]; s < offsets[e + 1]; ++s) expert_of[s] = e;
  parallel_for(R, threads, [&](int s) {
    int e = expert_of[s];
    if (e < 0) return;
    std::vector<double> a(K);
    for (int i = 0; i < K; ++i) a[i] = bf16_to_f32(a_bf16[(size_t)s * K + i]);
    for (int n = 0; n < N; ++n) {
      const uint16_t* w = w_bf16 + ((size_t)e * N + n) * K;
      double acc = 0.0;
      for (int i = 0; i < K; ++i) acc += a[i] * double(bf16_to_f32(w[i]));
      Y[(size_t)s * N + n] = acc;
    }
  });
}

void oracle_scatter(const double* Y, const int32_t* route_slot, const float* weights,
                    int N, int k, const int32_t* tokens, int n_tokens, double* out) {
  for (int i = 0; i < n_tokens; ++i) {
    int t = tokens ? tokens[i] : i;
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += double(weights[t * k + j]) * Y[(size_t)route_slot[t * k + j] * N + n];
      out[(size_t)i * N + n] = acc;
    }
  }
}

void oracle_forward_fp8(const float* logits, const uint16_t* x_bf16,
                        const uint8_t* w_q, const float* w_scales,
                        int M, int K, int N, int E, int k, float softcap, int renorm,
                        int block_m, const int32_t* tokens, int n_tokens, int threads,
                        int32_t* ids, float* weights, int32_t* counts, int32_t* offsets,
                        int32_t* sorted_route_ids, int32_t* route_slot,
                        int32_t* tile_offsets, uint8_t* a_q, float* a_scales,
                        double* out) {
  const int R = M * k;
  oracle_route(logits, M, E, k, softcap, renorm, ids, weights);
  oracle_layout(ids, M, E, k, block_m, counts, offsets, sorted_route_ids, route_slot,
                tile_offsets);
  oracle_quant_gather(x_bf16, M, K, k, route_slot, a_q, a_scales);
  std::vector<uint8_t> mask(R, tokens ? 0 : 1);
  if (tokens)
    for (int i = 0; i < n_tokens; ++i)
      for (int j = 0; j < k; ++j) mask[route_slot[tokens[i] * k + j]] = 1;
  std::vector<double> Y((size_t)R * N, 0.0);
  oracle_grouped_gemm_fp8(a_q, a_scales, R, K, w_q, w_scales, E, N, offsets, mask.data(),
                          threads, Y.data());
  oracle_scatter(Y.data(), route_slot, weights, N, k, tokens, n_tokens, out);
}

void oracle_dense_fp8(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                      const uint8_t* w_q, const float* w_scales,
                      int M, int K, int N, int E, int k,
                      const int32_t* tokens, int n_tokens, int threads, double* out) {
  (void)M; (void)E;
  const int KB = K / 128, NB = N / 128;
  parallel_for(n_tokens, threads, [&](int i) {
    int t = tokens ? tokens[i] : i;
    std::vector<uint8_t> q(K);
    std::vector<float> sa(KB);
    quantize_row(x_bf16 + (size_t)t * K, K, q.data(), sa.data());
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        int e = ids[t * k + j];
        const uint8_t* w = w_q + ((size_t)e * N + n) * K;
        double y = 0.0;
        for (int b = 0; b < KB; ++b) {
          double blk = 0.0;
          for (int c = b * 128; c < b * 128 + 128; ++c)
            blk += oracle_e4m3_decode(q[c]) * oracle_e4m3_decode(w[c]);
          y += double(sa[b]) * double(w_scales[((size_t)e * NB + n / 128) * KB + b]) * blk;
        }
        acc += double(weights[t * k + j]) * y;
      }
      out[(size_t)i * N + n] = acc;
    }
  });
}

void oracle_ffn_bf16(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                     const uint16_t* w_up, const uint16_t* w_dn,
                     int T, int H, int I, int E, int k,
                     const int32_t* tokens, int n_tokens, int threads, double* out) {
  (void)T; (void)E;
  parallel_for(n_tokens, threads, [&](int i) {
    int t = tokens ? tokens[i] : i;
    std::vector<double> x(H), h(I), acc(H, 0.0);
    for (int c = 0; c < H; ++c) x[c] = bf16_to_f32(x_bf16[(size_t)t * H + c]);
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      for (int r = 0; r < I; ++r) {
        const uint16_t* wg = w_up + ((size_t)e * 2 * I + r) * H;
        const uint16_t* wu = w_up + ((size_t)e * 2 * I + I + r) * H;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
          g += x[c] * double(bf16_to_f32(wg[c]));
          u += x[c] * double(bf16_to_f32(wu[c]));
        }
        double silu = g / (1.0 + std::exp(-g));
        h[r] = double(bf16_to_f32(oracle_bf16_round(silu * u)));
      }
      double w = weights[t * k + j];
      for (int n = 0; n < H; ++n) {
        const uint16_t* wd = w_dn + ((size_t)e * H + n) * I;
        double y = 0.0;
        for (int r = 0; r < I; ++r) y += h[r] * double(bf16_to_f32(wd[r]));
        acc[n] += w * y;
      }
    }
    for (int n = 0; n < H; ++n) out[(size_t)i * H + n] = acc[n];
  });
}

float oracle_swiglu_f32(float g, float u) {
  float e = oracle_exp_spec(-g);   // exp(-g): 0 below -87, +inf above 88
  float d = 1.0f + e;
  float sg = g / d;                // silu(g); g / inf = -0 for very negative g
  return sg * u;
}

void oracle_swiglu_quant(const float* gu, int R, int I, uint8_t* h_q, float* h_scales) {
  const int IB = I / 128;
  std::vector<float> h(I), sc(IB);
  for (int s = 0; s < R; ++s) {
    const float* row = gu + (size_t)s * 2 * I;
    for (int r = 0; r < I; ++r) h[r] = oracle_swiglu_f32(row[r], row[I + r]);
    quantize_f32_row(h.data(), I, h_q + (size_t)s * I, sc.data());
    for (int b = 0; b < IB; ++b) h_scales[(size_t)b * R + s] = sc[b];
  }
}

void oracle_ffn_fp8(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                    const uint8_t* wup_q, const float* wup_s, const uint8_t* wdn_q,
                    const float* wdn_s, int T, int H, int I, int E, int k,
                    const int32_t* tokens, int n_tokens, int threads, double* out) {
  (void)T; (void)E;
  const int HB = H / 128, IB = I / 128, UB = 2 * I / 128;
  double dq[256];
  for (int c = 0; c < 256; ++c) dq[c] = oracle_e4m3_decode(uint8_t(c));
  parallel_for(n_tokens, threads, [&](int i) {
    int t = tokens ? tokens[i] : i;
    std::vector<uint8_t> q(H), qh(I);
    std::vector<float> sa(HB), sh(IB), gu(2 * I);
    std::vector<double> acc(H, 0.0);
    quantize_row(x_bf16 + (size_t)t * H, H, q.data(), sa.data());
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      // up projection: gate rows [0, I), up rows [I, 2I); binary64, then
      // rounded to the binary32 the GEMM accumulates in
      for (int r = 0; r < 2 * I; ++r) {
        const uint8_t* w = wup_q + ((size_t)e * 2 * I + r) * H;
        double y = 0.0;
        for (int b = 0; b < HB; ++b) {
          double blk = 0.0;
          for (int c = b * 128; c < b * 128 + 128; ++c) blk += dq[q[c]] * dq[w[c]];
          y += double(sa[b]) * double(wup_s[((size_t)e * UB + r / 128) * HB + b]) * blk;
        }
        gu[r] = float(y);
      }
      // h = silu(gate) * up, re-quantised in 1x128 blocks for the FP8 down projection
      oracle_swiglu_quant(gu.data(), 1, I, qh.data(), sh.data());
      double w = weights[t * k + j];
      for (int n = 0; n < H; ++n) {
        const uint8_t* wd = wdn_q + ((size_t)e * H + n) * I;
        double y = 0.0;
        for (int b = 0; b < IB; ++b) {
          double blk = 0.0;
          for (int c = b * 128; c < b * 128 + 128; ++c) blk += dq[qh[c]] * dq[wd[c]];
          y += double(sh[b]) * double(wdn_s[((size_t)e * HB + n / 128) * IB + b]) * blk;
        }
        acc[n] += w * y;
      }
    }
    for (int n = 0; n < H; ++n) out[(size_t)i * H + n] = acc[n];
  });
}

}  // extern "C"
