// Persistent grouped GEMM on tcgen05 tensor cores (sm_103a).
//
// What it computes: "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)", section
// "Baseline: 7 kernels" item 6 (grouped FP8 GEMM with 128x128 weight blocks
// and 1x128 activation blocks; the blockwise scales are applied per 128-deep
// K block), with item 7 (routing-weighted scatter-add to token order) fused
// into the epilogue as in section "Fusion 1" / "Register-Direct Scatter
// Epilogue".  Scheduling follows section 2.2 of the blog retelling of "Weave":
// a fixed set of persistent CTAs pulls tiles from one global atomic counter;
// the tile order is N-tile-minor so tiles that share a block of routed rows
// run back to back (section "Grid Swap").
//
// How (this design, not the pages'): the MMA is "swap-AB" — the 128 weight
// rows of a tile are the MMA's M side and the routed rows (block_m of them,
// 16..256) are its N side, so a 4-row expert costs a 128x16 MMA instead of a
// padded 128-row one and the kernel streams each touched weight block once.
//   warps 0, 7  TMA producers, taking stages in turn; warp 0 also runs the
//               tile queue.  A stage holds sk K blocks and each of its 3-D
//               boxes (weight and activation tiles, sk K blocks deep) has its
//               own lane.  Gathered rows (kGather): the routed rows come as
//               tile::gather4 copies of four token rows each instead
//   warp 1      one thread issues tcgen05.mma into TMEM, commits to mbarriers;
//               the warp owns the TMEM allocation
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (thread = weight row),
//               FP8: per K block, acc += partial * (a_scale * w_scale) in fp32
//               registers ("promotion"; each K block has its own TMEM buffer;
//               packed f32x2 multiply-adds), then weighted red.global.add into
//               the fp32 output, a plain store, or silu(gate)*up to bf16.
//               More epilogue warps per TMEM lane quadrant, each taking a share
//               of the tile's columns: two (warps 8..11 too) for FP8 tiles of
//               64+ routed rows and BF16 tiles of 128, four (8..19) for BF16
//               tiles of 256
// A stage carries one weight tile, or two (the gate and up rows of the SwiGLU
// up projection; two adjacent weight tiles of a BF16 "wide" tile) that share
// the routed-row operand, so two MMAs per K block come from one stage.
//   warp 6      tile metadata: routed-row tokens, route weights and the FP8
//               scale products of each tile, staged into a shared ring ahead
//               of the epilogue (loads issued in dependency order, about
//               three memory round trips per tile)
// Every wait is bounded (mbar_wait): on a time-out the CTA records
// MOE_ERR_TIMEOUT in the workspace status word, raises a shared abort flag so
// the other roles stop too, waits (bounded) for its own in-flight copies and
// MMAs, frees its TMEM and returns.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "quant_common.cuh"

namespace moe {

namespace {

constexpr int kTileN = 128;           // weight rows per tile (MMA M)
constexpr int kRowBytes = 128;        // bytes per K block row (one swizzle atom row)
constexpr int kATileBytes = kTileN * kRowBytes;
constexpr int kMaxStages = 16;
// Tile descriptors (and metadata slots) in flight: 4, or 2 where a slot of
// FP8 scale products is large (block_m 128) and shared memory is needed for
// deeper stages.
constexpr int kMaxRing = 4;
__host__ __device__ constexpr int ring_slots(bool fp8, int bm) { return fp8 && bm >= 128 ? 2 : 4; }
constexpr int kMetaWarp = 6;
constexpr int kFirstExtraProducer = 7;  // warps 7.. are the extra TMA producers
// Warp roles: 0 producer + tile queue, 1 MMA, 2..5 epilogue (quadrant =
// warp & 3), 6 metadata, 7 .. 7 + kProducers - 2 extra producers, and with a
// second epilogue group the four warps after those (their warp & 3 again
// covers the four quadrants, since the second group starts at warp 8).
constexpr int kMaxE = 1024;

struct TileDesc {
  int e, m0, rows, n_tile, kb0, nkb;
};

// kWide (not SwiGLU): a tile covers two adjacent 128-row weight tiles (256
// output columns) that share its routed-row operand — two MMAs per K block
// from one stage, as the gated up projection has, so a stage carries twice
// the tensor work for 1.5 times the bytes.
//
// FP8 pair tiles (FP8 with two weight tiles per stage: kWide, or the gated up
// projection's gate + up tiles) keep one K block's two partial products per
// TMEM buffer (2 * BM columns), promote them into two register accumulators
// per epilogue thread, and run one TMA producer warp so that four epilogue
// warps per TMEM lane quadrant fit the register file at 128 routed rows.
//
// CTA pairs (kCta2): a cluster of two CTAs on two SMs shares each MMA
// (tcgen05.mma.cta_group::2, M = 256).  The even CTA issues every MMA; its
// mbarriers count both CTAs' copies and both CTAs' epilogue releases.
//   FP8 scatter at block_m 128: a tile of 256 weight rows x 128 routed rows;
//     each CTA stages its own 128 weight rows and half of the routed rows (64)
//     and holds its weight rows' 128 x 128 accumulator in its own TMEM, so a
//     K block's buffer is 128 columns (four in TMEM) and a stage 24 KB per K
//     block.
//   BF16 scatter / bf16 rows at block_m 256: a tile of 256 weight rows x 256
//     routed rows; each CTA stages its 128 weight rows and half of the routed
//     rows and holds its weight rows' 128 x 256 accumulator, so TMEM takes two
//     tiles (the single-CTA 256 x 256 tile fills it) and a tile's reductions or
//     stores overlap the next tile's MMAs.
//   SwiGLU (token-major; FP8 at block_m 128, BF16 at block_m 256): a tile of
//     256 routed rows x the gate and up rows of 128 h columns; each CTA stages
//     128 routed rows and one weight tile (the even CTA the gate rows, the odd
//     one the up rows) and its TMEM holds gate and up (256 columns) for its
//     own routed rows, so the SwiGLU (and the FP8 1x128 re-quantisation) stay
//     within the CTA.  FP8: 32 KB per K block against 48 KB for the
//     single-CTA tile; BF16: two accumulators in TMEM where the single-CTA
//     gate + up tile fills it.
template <int BM, bool kFP8, int kEpi, bool kWide = false, bool kCta2 = false>
struct Cfg {
  static constexpr bool kSwiglu = kEpi == MOE_EPI_SWIGLU;
  static constexpr bool kPair = kSwiglu || kWide;          // two weight tiles per stage
  static constexpr bool kFP8Pair = kFP8 && kPair;
  // FP8 pair tiles of 128 routed rows that store their results run
  // token-major: the routed rows are the MMA's M side (TMEM lanes) and both
  // weight tiles, contiguous in the stage, its N = 256 side, so each
  // instruction carries twice the work, each epilogue thread owns one routed
  // row (one scale per weight tile and K block) and its outputs leave as
  // 16-byte vectors.  The scatter keeps weight rows on the lanes: a warp's
  // reduction then covers 32 consecutive columns of one token (4 sectors)
  // instead of 16 bytes of 32 tokens (32 sectors), which measured faster.
  static constexpr bool kTok = kFP8Pair && BM == 128 && kEpi != MOE_EPI_SCATTER;
  static constexpr int kAccCols = kPair ? 2 * BM : BM;
  // FP8: one buffer per K block, up to all 512 columns, so the MMA can run a
  // whole tile or more ahead of the epilogue; BF16: double-buffered tiles.
  static constexpr int kNumAcc = kFP8 ? (512 / kAccCols < 32 ? 512 / kAccCols : 32)
                                      : (512 / kAccCols >= 2 ? 2 : 1);
  static constexpr int kTmemNeed = kNumAcc * kAccCols;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64
                                 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  // weight tiles a CTA stages per K block (CTA pairs: one each, gate or up)
  static constexpr int kATiles = (kPair && !kCta2) ? 2 : 1;
  static constexpr int kRing = ring_slots(kFP8, BM);
  // TMA producer warps (warp 0 plus warps 7..): two measured best (four were
  // no faster on any workload and slower on the BF16 FFN); FP8 pair tiles and
  // CTA pairs: one
  static constexpr int kProducers = (kFP8Pair || kCta2) ? 1 : 2;
  // FP8 with block_m >= 64 and BF16 with block_m >= 128: two epilogue warps per
  // TMEM lane quadrant, each taking half of the tile's columns (routed rows),
  // so two warps on every scheduler share the per-K-block promotion (FP8) or
  // the per-tile stores and reductions (BF16); otherwise one per quadrant
  // (BF16 with block_m 256: four, since its SwiGLU accumulator fills TMEM, so
  // the tile's epilogue is not overlapped with the next tile's MMAs).  FP8
  // pair tiles: one warp per quadrant for every 32 routed rows; CTA pairs:
  // four per quadrant.
  static constexpr int kEpiGroups = kFP8Pair ? (BM >= 32 ? BM / 32 : 1)
                                  : kCta2 ? 4
                                  : (!kFP8 && BM >= 256) ? 4
                                  : (kFP8 && BM >= 64) || (!kFP8 && BM >= 128) ? 2 : 1;
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  static constexpr int kEpiCols = BM / kEpiGroups;  // columns promoted by one epilogue warp
  // first warp of the second epilogue group (after the extra producers)
  static constexpr int kGroup1Warp = kFirstExtraProducer + kProducers - 1;
  static constexpr int kWarps = kGroup1Warp + 4 * (kEpiGroups - 1);
  static constexpr int kThreads = 32 * kWarps;
  // routed rows of a stage (CTA-pair scatter: this CTA's half of the tile's)
  static constexpr int kBRows = (kCta2 && !kSwiglu) ? BM / 2 : BM;
  // routed rows of one tile (CTA-pair SwiGLU: BM per CTA, so 2 * BM per pair)
  static constexpr int kTileRows = (kCta2 && kSwiglu) ? 2 * BM : BM;
  // bytes of one K block of a stage; a stage holds p.sk K blocks laid out as
  // [kATiles][sk] weight tiles, then [sk] activation tiles
  static constexpr int kStageBytes = kATiles * kATileBytes + kBRows * kRowBytes;
  // FP8 epilogue: K blocks whose partials are loaded before one wait (<= 64 columns)
  static constexpr int kKbGroup = BM <= 64 ? 64 / BM : 1;
  static constexpr int kLdCols = BM <= 64 ? BM : 64;   // columns per load wave
  static_assert(BM % 16 == 0 && BM >= 16 && BM <= 256, "block_m");
  static_assert(!kFP8 || BM <= 128, "FP8 block_m <= 128");
  static_assert(kTmemNeed <= 512, "TMEM");
  static_assert(!kCta2 || (BM == 128 && !kWide && kSwiglu) ||
                    (kFP8 && BM == 128 && !kPair && kEpi == MOE_EPI_SCATTER) ||
                    (!kFP8 && BM == 256 && !kPair &&
                     (kEpi == MOE_EPI_SCATTER || kEpi == MOE_EPI_STORE_BF16)),
                "CTA pairs");
};

// Bytes of one metadata slot.  FP8 single tiles: [kb_per_split][BM] scale
// products a_scale * w_scale; FP8 pair tiles: [kb_per_split][BM] activation
// scales, then the two weight tiles' scales [2][kb_per_split].  Then BM token
// ids and BM route weights.
// Floats of the pair tiles' weight-scale vectors, padded so the token ids
// that follow stay 16-byte aligned (they are read as 4-int vectors).
__host__ __device__ inline int pair_sw_floats(int kb_per_split) {
  return (2 * kb_per_split + 3) & ~3;
}

__host__ __device__ inline int meta_slot_bytes(bool fp8, int bm, int kb_per_split,
                                               bool pair = false) {
  const int n = (fp8 ? kb_per_split * bm + (pair ? pair_sw_floats(kb_per_split) : 0) : 0) + 2 * bm;
  return (n * 4 + 15) & ~15;
}

// Shared memory of the FP8 SwiGLU epilogue's block amax exchange: per epilogue
// group, two tile buffers of [4 quadrants][32 routed rows] floats.
__host__ __device__ constexpr int swiglu_red_bytes(int groups) { return groups * 2 * 4 * 32 * 4; }

// Output tiles handed out as tail_parts K parts each (halves or quarters) at
// the end of the work list, one K split only: p.tail_tiles of them for the
// queue (one per CTA: the last wave), or, for the fixed round-robin order of
// G = -p.tail_tiles CTA pairs, the remainder of an even split plus one round
// (every tile when T < 2G), so that every pair gets the same number of whole
// tiles and the parts spread the rest.
__device__ __forceinline__ int tail_count(const GemmParams& p, int T) {
  if (p.tail_tiles >= 0) return min(p.tail_tiles, T);
  const int G = -p.tail_tiles;
  return T >= 2 * G ? T % G + G : T;
}

// Work items: whole tiles, then the split tail's parts.
__device__ __forceinline__ int work_items(const GemmParams& p, const int* s_tile_off) {
  const int T = s_tile_off[p.E] * p.n_tiles * p.k_splits;
  return T + tail_count(p, T) * (p.tail_parts - 1);
}

__device__ __forceinline__ void decode_tile(int t, const GemmParams& p, const int* s_tile_off,
                                            const int* s_off, int BM, TileDesc& d) {
  int part = -1;  // >= 0: K part of a split tail tile
  if (p.tail_tiles != 0) {
    const int T = s_tile_off[p.E] * p.n_tiles;
    const int F = T - tail_count(p, T);
    if (t >= F) {
      part = (t - F) % p.tail_parts;
      t = F + (t - F) / p.tail_parts;
    }
  }
  const int per_m = p.n_tiles * p.k_splits;
  const int mt = t / per_m;
  const int r = t - mt * per_m;
  // expert: last e with tile_off[e] <= mt (tile_off[E] > mt).  The whole warp
  // searches: each lane tests one entry of a stride-spaced sample, then one
  // entry of the chosen stride (two ballots instead of log2(E) dependent
  // loads); the caller's 32 lanes are converged.
  const int lane = threadIdx.x & 31;
  const int stride = (p.E + 32) / 32;  // ceil((E + 1) / 32)
  int e;
  if (stride <= 32) {
    unsigned m = __ballot_sync(0xffffffffu, s_tile_off[min(p.E, lane * stride)] <= mt);
    const int base = (31 - __clz(m)) * stride;
    m = __ballot_sync(0xffffffffu, lane < stride && s_tile_off[min(p.E, base + lane)] <= mt);
    e = base + 31 - __clz(m);
  } else {
    int lo = 0, hi = p.E;  // invariant: tile_off[lo] <= mt < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_off[mid] <= mt) lo = mid; else hi = mid;
    }
    e = lo;
  }
  const int seg_begin = s_off[e], seg_end = s_off[e + 1];
  d.e = e;
  d.m0 = seg_begin + (mt - s_tile_off[e]) * BM;
  d.rows = min(BM, seg_end - d.m0);
  d.n_tile = r / p.k_splits;
  const int ks = r - d.n_tile * p.k_splits;
  d.kb0 = ks * p.kb_per_split;
  d.nkb = min(p.kb_per_split, p.KB - d.kb0);
  if (part >= 0) {  // split points on stage boundaries (tail_partkb is a multiple of sk)
    d.kb0 = part * p.tail_partkb;
    d.nkb = part == p.tail_parts - 1 ? p.KB - d.kb0 : p.tail_partkb;
  }
}

// One tile's metadata, filled by the 32 lanes of the metadata warp: FP8
// scale products sc[kb][row] = a_scale * w_scale, and for the scatter the
// row's token tok[row] and route weight wt[row].  Loads are issued in
// dependency order across the whole tile — every route id, then every scale,
// then every route weight (which needs its route id) — so a tile costs about
// three memory round trips.  kGather: the route ids come from the tile's
// ring slot (rr) and the activation scales are token-major ([KB, M]);
// otherwise the ids are loaded from sorted_route_ids and the scales are
// compact ([KB, R]), their addresses independent of the ids.
// FP8 pair tiles (kPair): sc holds the activation scales alone and the two
// weight tiles' scales follow as sw[2][kb_per_split] (the epilogue forms the
// products), so the slot stays the size of a single tile's.
template <int BM, bool kFP8, int kEpi, bool kGather, bool kPair = false, bool kWide = false>
__device__ __forceinline__ void meta_fill(const GemmParams& p, const TileDesc& d, int lane,
                                          const int* rr, float* sc, int* tok, float* wt) {
  constexpr int kRows = (BM + 31) / 32;  // rows of the tile per lane
  const int NB = p.N / kTileN;
  int rid[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const int s = lane + 32 * j;
    if constexpr (kGather)
      rid[j] = s < BM ? rr[s] : -1;
    else
      rid[j] = (kEpi == MOE_EPI_SCATTER && s < d.rows) ? __ldg(p.sorted_route_ids + d.m0 + s) : -1;
  }
  if constexpr (kFP8 && kPair) {
    // the two weight tiles' 128-row blocks: adjacent (wide) or gate and up
    const int nb0 = kWide ? 2 * d.n_tile : d.n_tile;
    const int nb1 = kWide ? 2 * d.n_tile + 1 : d.n_tile + NB / 2;
    float* sw = sc + p.kb_per_split * BM;
    for (int kb = lane; kb < d.nkb; kb += 32) {
      sw[kb] = __ldg(p.w_scales + (static_cast<size_t>(d.e) * NB + nb0) * p.KB + d.kb0 + kb);
      sw[p.kb_per_split + kb] =
          __ldg(p.w_scales + (static_cast<size_t>(d.e) * NB + nb1) * p.KB + d.kb0 + kb);
    }
  }
  if constexpr (kFP8) {
    // scale products for up to 16 K blocks at a time, all loads in flight together
    // (pair tiles: the activation scales alone, vb = 1)
    const float* wsc = p.w_scales + (static_cast<size_t>(d.e) * NB + d.n_tile) * p.KB + d.kb0;
    const size_t a_ld = kGather ? static_cast<size_t>(p.M) : static_cast<size_t>(p.R);
    const float* asc = p.a_scales + static_cast<size_t>(d.kb0) * a_ld + (kGather ? 0 : d.m0);
    int arow[kRows];  // column of each row in the scale matrix
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      if constexpr (kGather)
        arow[j] = rid[j] >= 0 ? rid[j] / p.top_k : -1;
      else
        arow[j] = lane + 32 * j;
    }
    for (int kb0 = 0; kb0 < d.nkb; kb0 += 16) {
      float va[16][kRows];
      float vb[16];
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) {
        if constexpr (kPair)
          vb[kb] = 1.0f;
        else
          vb[kb] = kb0 + kb < d.nkb ? __ldg(wsc + kb0 + kb) : 0.0f;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int s = lane + 32 * j;
          va[kb][j] = (kb0 + kb < d.nkb && s < d.rows && arow[j] >= 0)
                          ? __ldg(asc + static_cast<size_t>(kb0 + kb) * a_ld + arow[j])
                          : 0.0f;
        }
      }
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) {
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int s = lane + 32 * j;
          if (kb0 + kb < d.nkb && s < BM) sc[(kb0 + kb) * BM + s] = va[kb][j] * vb[kb];
        }
      }
    }
  }
  if constexpr (kEpi == MOE_EPI_SCATTER) {
    float w[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) w[j] = rid[j] >= 0 ? __ldg(p.route_weights + rid[j]) : 0.0f;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int s = lane + 32 * j;
      if (s < BM) {
        tok[s] = rid[j] >= 0 ? rid[j] / p.top_k : 0;
        wt[s] = w[j];
      }
    }
  }
}

template <int BM, bool kFP8, int kEpi, bool kGather, bool kWide, bool kCta2>
__global__ void __launch_bounds__(Cfg<BM, kFP8, kEpi, kWide, kCta2>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_a, const GemmParams p) {
  using C = Cfg<BM, kFP8, kEpi, kWide, kCta2>;
  static_assert(!(kCta2 && kGather), "CTA pairs read compact rows");
  static_assert(!(kWide && (C::kSwiglu || kGather)), "wide tiles: store / scatter, compact rows");
  static_assert(!(C::kFP8Pair && kGather), "FP8 pair tiles read compact rows");
  // weight rows of a tile (two weight tiles when wide or split over a CTA pair)
  constexpr int kWRows = (kWide || (kCta2 && !C::kSwiglu)) ? 2 * kTileN : kTileN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_tfull[C::kNumAcc], bar_tempty[C::kNumAcc];
  __shared__ __align__(8) uint64_t bar_dfull[kMaxRing], bar_dempty[kMaxRing], bar_mfull[kMaxRing];
  __shared__ __align__(8) uint64_t bar_drain;
  // FP8 SwiGLU: per epilogue group, the four quadrant warps' block-amax exchange
  __shared__ __align__(8) uint64_t bar_red[4];
  __shared__ TileDesc s_desc[kMaxRing];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs: 0 for the CTA that issues the MMAs, 1 for its peer
  const uint32_t rank = kCta2 ? cluster_ctarank() : 0u;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const int NST = p.num_stages;
  const int SK = p.sk;                                  // K blocks per stage
  const int stage_bytes = SK * C::kStageBytes;
  const int meta_bytes = meta_slot_bytes(kFP8, BM, p.kb_per_split, C::kFP8Pair);
  // first int of a metadata slot's token ids (after the FP8 scales)
  const int tok_off =
      kFP8 ? p.kb_per_split * BM + (C::kFP8Pair ? pair_sw_floats(p.kb_per_split) : 0) : 0;
  uint8_t* s_meta = smem_gen + NST * stage_bytes;       // C::kRing slots of meta_bytes
  // tile offsets and row offsets of the experts ([E + 1] each) after the ring
  int* s_tile_off = reinterpret_cast<int*>(s_meta + C::kRing * meta_bytes);
  int* s_off = s_tile_off + (p.E + 1);
  // gathered-rows mode: route id of every routed row of each ring slot's tile
  // ([kRing][BM], -1 past the tile's rows), after the tables; the FP8 SwiGLU
  // epilogue's block-amax exchange sits in the same place (neither mode has
  // the other)
  int* s_rows = s_tile_off + ((2 * (p.E + 1) + 3) & ~3);
  float* s_red = reinterpret_cast<float*>(s_rows);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    for (int i = 0; i < C::kNumAcc; ++i) {
      mbar_init(smem_u32(&bar_tfull[i]), 1);
      mbar_init(smem_u32(&bar_tempty[i]), kCta2 ? 2 * C::kEpiWarps : C::kEpiWarps);
    }
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(smem_u32(&bar_dfull[i]), 1);
      // MMA, the epilogue warps, the extra producers
      mbar_init(smem_u32(&bar_dempty[i]), 1 + C::kEpiWarps + C::kProducers - 1);
      mbar_init(smem_u32(&bar_mfull[i]), 1);
    }
    mbar_init(smem_u32(&bar_drain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bar_red[i]), 4);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    if constexpr (kCta2) {
      // one warp of each CTA of the pair: the same columns in both TMEMs
      tmem_alloc_pair(smem_u32(&s_tmem), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
      tmem_relinquish();
    }
  }
  if (!kCta2 && p.warm_first > 0 && warp == 0) {
    // The queue hands CTA c tile c first and tiles c + G, c + 2G ... mostly
    // next (G CTAs).  When every expert has a single row tile (small batches),
    // tile t is expert t / (n_tiles * k_splits); its weight rows do not depend
    // on the routing, so the first warm_first waves' weights are prefetched
    // into L2 while the router and layout still run (HBM is otherwise idle).
    const int per_e = p.n_tiles * p.k_splits;
    for (int w = 0; w < p.warm_first; ++w) {
      const int t = blockIdx.x + w * gridDim.x;
      const int e = t / per_e, r = t - e * per_e;
      const int nt = r / p.k_splits, ks = r - nt * p.k_splits;
      const int kb0 = ks * p.kb_per_split, kb1 = min(p.KB, kb0 + p.kb_per_split);
      if (e < p.E)
        for (int kb = kb0 + lane * p.sk; kb < kb1; kb += 32 * p.sk)
          tma_prefetch_l2_3d(&tmap_w, 0, e * p.N + nt * (kWide ? 2 * kTileN : kTileN), kb);
    }
  }
  // Everything above is independent of the preceding kernel's results.
  pdl_wait();
  for (int i = threadIdx.x; i <= p.E; i += C::kThreads) {  // all copies in flight, one wait
    cp_async4(smem_u32(&s_tile_off[i]), p.tile_offsets + i);
    cp_async4(smem_u32(&s_off[i]), p.offsets + i);
  }
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if constexpr (C::kTileRows != BM) {
    // CTA-pair SwiGLU: tiles of 2 * BM routed rows, so the tile offsets are
    // the prefix of ceil(count / (2 * BM)) over the experts, from the row
    // offsets (one warp: a run of experts per lane, then a warp scan)
    if (warp == 0) {
      const int per = (p.E + 31) / 32;
      const int e0 = min(p.E, lane * per), e1 = min(p.E, e0 + per);
      int local = 0;
      for (int e = e0; e < e1; ++e)
        local += (s_off[e + 1] - s_off[e] + C::kTileRows - 1) / C::kTileRows;
      int inc = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      int run = inc - local;
      for (int e = e0; e < e1; ++e) {
        s_tile_off[e] = run;
        run += (s_off[e + 1] - s_off[e] + C::kTileRows - 1) / C::kTileRows;
      }
      if (lane == 31) s_tile_off[p.E] = inc;
    }
    __syncthreads();
  }
  // CTA pairs: both CTAs' mbarriers are initialised (and their TMEM
  // allocated) before either CTA signals the other's
  if constexpr (kCta2) cluster_sync();
  tc_fence_after();
  // The dependent kernel (the forward's finalize) may become resident now;
  // its griddepcontrol.wait still waits for this grid to complete.
  pdl_launch_dependents();
  const uint32_t tmem_base = s_tmem;
  const int total_tiles = work_items(p, s_tile_off);
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0 || (warp >= kFirstExtraProducer && warp < kFirstExtraProducer + C::kProducers - 1)) {
    // ------------------------------------------------------------ producers
    // A warp's bulk-tensor copy instructions are served one after another, at
    // a bounded rate of instructions rather than bytes.  So kProducers warps
    // fill the ring in turn (global stage q goes to producer q % kProducers),
    // and within an instruction every box of the stage goes out from its own
    // lane: lane a < kATiles loads weight
    // tile a, lane kATiles the activation tile, each box SK K blocks deep.
    // Warp 0 also runs the tile queue and publishes each tile's descriptor.
    const int pw = warp == 0 ? 0 : warp - kFirstExtraProducer + 1;
    // weights: evict-first when each expert's tile is read once (small
    // batches stream every touched expert once), evict-last when several row
    // tiles of an expert reuse it; routed rows: evict-last (every N tile of a
    // row tile reads them)
    const uint64_t pol_w = p.w_reuse ? policy_evict_last() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0, ds = 0, q = 0;   // q: global stage number (every producer counts all stages)
    // Producers in use: at most one per stage.  A producer waits on a slot's
    // "empty" barrier by phase parity, which is only unambiguous while the
    // slot's previous fill (issued by another producer) cannot lag by a whole
    // ring; with nprod <= NST it cannot.
    const int nprod = min(C::kProducers, NST);
    int q_own = -1;                 // last global stage this warp filled
    uint32_t phase = 0, dphase = 0;
    bool ok = true;
    // static schedule state: experts handled by this CTA
    const int G = gridDim.x, c = blockIdx.x;
    int st_e = G >= p.E ? c % p.E : c;
    const int st_idx = G >= p.E ? c / p.E : 0;
    const int st_stride = G >= p.E ? (G - (c % p.E) + p.E - 1) / p.E : 1;
    int st_lt = st_idx;
    // queue: CTA c starts with tile c; later tiles come from the counter
    // (offset by the grid size), claimed one tile ahead — after the current
    // tile's first stage has been issued, so the atomic's round trip overlaps
    // that tile's loads instead of delaying them
    int queued = p.sched == MOE_SCHED_QUEUE ? c : -1;
    // CTA pairs: both CTAs walk the same list, tiles c/2, c/2 + G/2, ...
    int rr_i = 0;
    bool claim = false;             // lane 0 of warp 0: the next tile is still to be claimed
    // Gathered rows: warp 0 loads each tile's route ids (kRpl per lane) and
    // puts them in the tile's ring slot with its descriptor.  The queue's next
    // tile is decoded and its ids loaded halfway through the current tile
    // ("pre"), so the loads' round trip overlaps the current tile's copies.
    constexpr int kRpl = (BM + 31) / 32;
    int nr[kRpl];
    TileDesc dn;
    bool pre = false;
    for (;;) {
      TileDesc d;
      bool got = true;
      if (pw == 0) {
        if (pre) {
          d = dn;
          pre = false;
          if (lane == 0) claim = true;
        } else {
          int t = -1;
          if (lane == 0) {
            if (kCta2) {
              const int t2 = (c >> 1) + rr_i * (G >> 1);
              ++rr_i;
              t = t2 < total_tiles ? t2 : -1;
            } else if (p.sched == MOE_SCHED_QUEUE) {
              t = queued < total_tiles ? queued : -1;
              claim = t >= 0;
            } else {
              while (st_e < p.E) {
                const int per_e = (s_tile_off[st_e + 1] - s_tile_off[st_e]) * p.n_tiles * p.k_splits;
                if (st_lt < per_e) {
                  t = s_tile_off[st_e] * p.n_tiles * p.k_splits + st_lt;
                  st_lt += st_stride;
                  break;
                }
                if (G >= p.E) { st_e = p.E; break; }
                st_e += G;
                st_lt = 0;
              }
            }
          }
          t = __shfl_sync(0xffffffffu, t, 0);
          if (t >= 0) {
            decode_tile(t, p, s_tile_off, s_off, C::kTileRows, d);
            if (d.rows <= 0 || d.nkb <= 0) {
              if (lane == 0 && claim) {
                queued = G + static_cast<int>(atomicAdd(p.queue_ctr, 1u));
                claim = false;
              }
              continue;
            }
            if constexpr (kGather) {
#pragma unroll
              for (int j = 0; j < kRpl; ++j) {
                const int s = lane + 32 * j;
                nr[j] = s < d.rows ? __ldg(p.sorted_route_ids + d.m0 + s) : -1;
              }
            }
          } else {
            d.nkb = -1;
          }
        }
        if (lane == 0) got = mbar_wait(smem_u32(&bar_dempty[ds]), dphase ^ 1u, &s_abort, tmo);
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
        if (kGather && d.nkb >= 0) {
#pragma unroll
          for (int j = 0; j < kRpl; ++j) {
            const int s = lane + 32 * j;
            if (s < BM) s_rows[ds * BM + s] = nr[j];
          }
        }
        __syncwarp();
        if (lane == 0) {
          s_desc[ds] = d;
          mbar_arrive(smem_u32(&bar_dfull[ds]));
        }
      } else {
        if (lane == 0) got = mbar_wait(smem_u32(&bar_dfull[ds]), dphase, &s_abort, tmo);
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
        __syncwarp();
        d = s_desc[ds];
        __syncwarp();
        // (the slot's route ids stay valid until the epilogue has finished
        // this tile, long after its last copy is issued)
        if (lane == 0) mbar_arrive(smem_u32(&bar_dempty[ds]));
      }
      const int* rr = s_rows + ds * BM;   // this tile's route ids (gathered rows)
      if (++ds == C::kRing) { ds = 0; dphase ^= 1u; }
      if (d.nkb < 0) break;
      // CTA pairs: the odd CTA's weight tile is the scatter tile's second
      // 128 rows, or the SwiGLU tile's up rows (N / 2 on)
      const int w_row = d.e * p.N + d.n_tile * kWRows +
                        (kCta2 ? static_cast<int>(rank) * (C::kSwiglu ? p.N / 2 : kTileN) : 0);
      const int w_pair = C::kSwiglu ? p.N / 2 : kTileN;  // row offset of the second weight tile
      for (int i = 0; i < d.nkb; i += SK) {
        if (q % nprod == pw) {
          const uint32_t full = smem_u32(&bar_full[stage]);
          if (lane == 0) {
            got = mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, &s_abort, tmo);
            // CTA pairs: the even CTA's barrier counts both CTAs' bytes
            if (got && !p.drop_producer && rank == 0)
              mbar_arrive_expect_tx(full, kCta2 ? 2 * stage_bytes : stage_bytes);
          }
          if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
          q_own = q;
          if (!p.drop_producer) {
            // one box per lane: weight tile(s), then the activation tile; each
            // box spans SK K blocks (a box running past K reads the fill value)
            const uint32_t sa = smem_base + stage * stage_bytes;
            const int kb = d.kb0 + i;
            if constexpr (kCta2) {
              // this CTA's weight rows and its half of the routed rows, both
              // counted on the even CTA's barrier
              const uint32_t full0 = mapa_shared(full, 0);
              if (lane == 0)
                tma_load_3d_pair(sa, &tmap_w, full0, 0, w_row, kb, pol_w);
              else if (lane == 1)
                tma_load_3d_pair(sa + SK * kATileBytes, &tmap_a, full0, 0,
                                 d.m0 + static_cast<int>(rank) * C::kBRows, kb, pol_a);
            } else if constexpr (!kGather) {
              // one if / else-if chain: the boxes go out from their lanes as one instruction
              if (lane < C::kATiles)
                tma_load_3d(sa + lane * SK * kATileBytes, &tmap_w, full, 0, w_row + lane * w_pair,
                            kb, pol_w);
              else if (lane == C::kATiles)
                tma_load_3d(sa + C::kATiles * SK * kATileBytes, &tmap_a, full, 0, d.m0, kb, pol_a);
            } else {
              if (lane < C::kATiles)
                tma_load_3d(sa + lane * SK * kATileBytes, &tmap_w, full, 0, w_row + lane * w_pair,
                            kb, pol_w);
              // the routed rows, four per copy (SK * BM / 4 copies over the
              // warp's lanes); a K block past the tile's end reloads its last
              // one, which the MMA does not read; an empty row reads token 0
              const int nk = min(SK, d.nkb - i);
              constexpr int kG = BM / 4;
              for (int g = lane; g < SK * kG; g += 32) {
                const int kbl = g / kG, g4 = g - kbl * kG;
                const int4 r4 = *reinterpret_cast<const int4*>(rr + 4 * g4);
                const int kc = (kb + min(kbl, nk - 1)) * (kFP8 ? 128 : 64);
                tma_gather4(sa + C::kATiles * SK * kATileBytes + kbl * (BM * kRowBytes) + g4 * 512,
                            &tmap_a, full, kc, max(r4.x, 0) / p.top_k, max(r4.y, 0) / p.top_k,
                            max(r4.z, 0) / p.top_k, max(r4.w, 0) / p.top_k);
              }
            }
          }
          __syncwarp();
        }
        if (pw == 0 && lane == 0 && claim) {  // the next tile, now that this one is under way
          queued = G + static_cast<int>(atomicAdd(p.queue_ctr, 1u));
          claim = false;
        }
        if (kGather && pw == 0 && i > 0 && i == ((d.nkb / SK) / 2) * SK &&
            p.sched == MOE_SCHED_QUEUE) {
          // halfway through the tile the claim has returned: decode the claimed
          // tile and start its id loads (reading the claim any earlier would
          // stall this warp on the atomic's round trip)
          const int nt = __shfl_sync(0xffffffffu, queued, 0);
          if (nt < total_tiles) {
            decode_tile(nt, p, s_tile_off, s_off, C::kTileRows, dn);
            if (dn.rows > 0 && dn.nkb > 0) {
              {
#pragma unroll
                for (int j = 0; j < kRpl; ++j) {
                  const int s = lane + 32 * j;
                  nr[j] = s < dn.rows ? __ldg(p.sorted_route_ids + dn.m0 + s) : -1;
                }
              }
              pre = true;
            }
          }
        }
        ++q;
        if (++stage == NST) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    if (lane == 0) {
      if (!ok) {
        set_error(p.ctrl, MOE_ERR_TIMEOUT, 1);
        s_abort = 1;
      }
      // Each producer waits (bounded by time, also after an abort) until the
      // loads it issued into the ring's last pass (global stages after
      // q - NST, whose slots are not refilled) have landed, so no copy is
      // still writing shared memory when the CTA exits.
      // CTA pairs: a copy counts on the even CTA's barrier, so each CTA waits
      // instead until the MMAs that read the stage have completed
      if (!p.drop_producer) {
        for (int qq = q_own; qq >= 0 && qq > q - NST; qq -= nprod)
          mbar_wait_drain(smem_u32(kCta2 ? &bar_empty[qq % NST] : &bar_full[qq % NST]),
                          static_cast<uint32_t>(qq / NST) & 1u, tmo);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (kCta2 && rank != 0 && lane == 0) {
      // the peer of a CTA pair issues nothing: it only retires the descriptors
      int ds = 0;
      uint32_t dphase = 0;
      for (;;) {
        if (!mbar_wait(smem_u32(&bar_dfull[ds]), dphase, &s_abort, tmo)) {
          set_error(p.ctrl, MOE_ERR_TIMEOUT, 2);
          s_abort = 1;
          break;
        }
        const int nkb = s_desc[ds].nkb;
        mbar_arrive(smem_u32(&bar_dempty[ds]));
        if (++ds == C::kRing) { ds = 0; dphase ^= 1u; }
        if (nkb < 0) break;
      }
    } else if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kFP8 ? 0u : 1u, 128u, static_cast<uint32_t>(BM));
      int stage = 0, ds = 0, acc_n = 0;
      uint32_t phase = 0, dphase = 0;
      bool ok = true;
      for (;;) {
        if (!mbar_wait(smem_u32(&bar_dfull[ds]), dphase, &s_abort, tmo)) { ok = false; break; }
        const TileDesc d = s_desc[ds];
        mbar_arrive(smem_u32(&bar_dempty[ds]));
        if (++ds == C::kRing) { ds = 0; dphase ^= 1u; }
        if (d.nkb < 0) break;
        int buf = 0;
        for (int i = 0; i < d.nkb; i += SK) {
          const int nk = min(SK, d.nkb - i);
          if (!kFP8 && i == 0) {
            buf = acc_n % C::kNumAcc;
            const uint32_t use = static_cast<uint32_t>(acc_n / C::kNumAcc);
            if (!mbar_wait(smem_u32(&bar_tempty[buf]), (use & 1u) ^ 1u, &s_abort, tmo)) { ok = false; break; }
            tc_fence_after();
          }
          if (!mbar_wait(smem_u32(&bar_full[stage]), phase, &s_abort, tmo)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sbase = smem_base + stage * stage_bytes;
          for (int kb = 0; kb < nk; ++kb) {
            if constexpr (kFP8) {
              buf = acc_n % C::kNumAcc;
              const uint32_t use = static_cast<uint32_t>(acc_n / C::kNumAcc);
              if (!mbar_wait(smem_u32(&bar_tempty[buf]), (use & 1u) ^ 1u, &s_abort, tmo)) { ok = false; break; }
              tc_fence_after();
            }
            const uint32_t a_addr = sbase + kb * kATileBytes;
            const uint32_t b_addr =
                sbase + C::kATiles * SK * kATileBytes + kb * (C::kBRows * kRowBytes);
            const uint32_t d_tmem = tmem_base + buf * C::kAccCols;
            // descriptor low words of this K block's operands (a K step adds 2)
            const uint32_t alo = smem_desc_lo(a_addr), blo = smem_desc_lo(b_addr);
            if constexpr (kCta2 && C::kSwiglu) {
              // M = 256 routed rows (128 per CTA), N = the gate rows (even CTA)
              // and the up rows (odd CTA) of 128 h columns (FP8: one K block
              // per buffer; BF16: accumulated over all of K)
              constexpr uint32_t idesc_p = make_idesc(kFP8 ? 0u : 1u, 256u, 256u);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_lo<kFP8, true>(d_tmem, blo + 2 * kk, alo + 2 * kk, idesc_p,
                                    (kFP8 ? kk > 0 : (i > 0 || kb > 0 || kk > 0)) ? 1u : 0u);
            } else if constexpr (kCta2 && !kFP8) {
              // BF16: M = 256 weight rows (128 per CTA), N = 256 routed rows (128
              // per CTA), accumulated over all of K
              constexpr uint32_t idesc_p = make_idesc(1u, 256u, static_cast<uint32_t>(BM));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_lo<false, true>(d_tmem, alo + 2 * kk, blo + 2 * kk, idesc_p,
                                     (i > 0 || kb > 0 || kk > 0) ? 1u : 0u);
            } else if constexpr (kCta2) {
              // M = 256 weight rows (128 per CTA), N = 128 routed rows (64 per CTA)
              constexpr uint32_t idesc_p = make_idesc(0u, 256u, 128u);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_lo<true, true>(d_tmem, alo + 2 * kk, blo + 2 * kk, idesc_p, kk > 0 ? 1u : 0u);
            } else if constexpr (C::kTok) {
              // M = the 128 routed rows, N = both weight tiles (256 rows,
              // contiguous because a stage holds one K block)
              constexpr uint32_t idesc_t = make_idesc(0u, 128u, 256u);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_lo<true>(d_tmem, blo + 2 * kk, alo + 2 * kk, idesc_t, kk > 0 ? 1u : 0u);
            } else {
              const uint32_t alo2 = smem_desc_lo(a_addr + SK * kATileBytes);  // second weight tile
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = kFP8 ? (kk > 0) : (i > 0 || kb > 0 || kk > 0);
                umma_lo<kFP8>(d_tmem, alo + 2 * kk, blo + 2 * kk, idesc, acc);
                if constexpr (C::kPair)
                  umma_lo<kFP8>(d_tmem + BM, alo2 + 2 * kk, blo + 2 * kk, idesc, acc);
              }
            }
            if constexpr (kFP8) {
              if constexpr (kCta2) umma_commit_pair(smem_u32(&bar_tfull[buf]), 3);
              else umma_commit(smem_u32(&bar_tfull[buf]));
              ++acc_n;
            }
          }
          if (!ok) break;
          if constexpr (kCta2) umma_commit_pair(smem_u32(&bar_empty[stage]), 3);
          else umma_commit(smem_u32(&bar_empty[stage]));
          if constexpr (!kFP8) {
            if (i + nk >= d.nkb) {
              if constexpr (kCta2) umma_commit_pair(smem_u32(&bar_tfull[buf]), 3);
              else umma_commit(smem_u32(&bar_tfull[buf]));
              ++acc_n;
            }
          }
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (!ok) {
        set_error(p.ctrl, MOE_ERR_TIMEOUT, 2);
        s_abort = 1;
      }
      // drain: every MMA issued above has completed before TMEM is freed
      if constexpr (kCta2) umma_commit_pair(smem_u32(&bar_drain), 1);
      else umma_commit(smem_u32(&bar_drain));
      mbar_wait(smem_u32(&bar_drain), 0u, &s_abort, tmo);
    }
  } else if (warp == kMetaWarp) {
    // ------------------------------------------------------------ tile metadata
    int ds = 0;
    uint32_t dphase = 0;
    for (;;) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_dfull[ds]), dphase, &s_abort, tmo))) {
        set_error(p.ctrl, MOE_ERR_TIMEOUT, 4);
        s_abort = 1;
        break;
      }
      const TileDesc d = s_desc[ds];
      if (d.nkb >= 0) {
        float* sc = reinterpret_cast<float*>(s_meta + ds * meta_bytes);
        int* tok = reinterpret_cast<int*>(sc + tok_off);
        float* wt = reinterpret_cast<float*>(tok + BM);
        // CTA pairs: this CTA's 128-row weight block of the 256-row tile
        TileDesc dm = d;
        if constexpr (kCta2 && !C::kSwiglu) dm.n_tile = 2 * d.n_tile + static_cast<int>(rank);
        if constexpr (kCta2 && C::kSwiglu) {   // this CTA's routed rows of the pair tile
          dm.m0 = d.m0 + static_cast<int>(rank) * BM;
          dm.rows = max(0, min(BM, d.rows - static_cast<int>(rank) * BM));
        }
        meta_fill<BM, kFP8, kEpi, kGather, C::kPair, kWide>(p, dm, lane, s_rows + ds * BM, sc, tok,
                                                            wt);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_mfull[ds]));
      if (++ds == C::kRing) { ds = 0; dphase ^= 1u; }
      if (d.nkb < 0) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                     // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;              // weight row within the tile
    // epilogue group of this warp (four consecutive warps, one per quadrant):
    // warps 2..5, then from kGroup1Warp (7 or 8) on, four at a time
    const int grp = warp < C::kGroup1Warp ? 0 : 1 + (warp - C::kGroup1Warp) / 4;
    // first column (routed row) of this warp's share of the tile
    const int c_lo = grp * C::kEpiCols;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + c_lo;
    int ds = 0, acc_n = 0;
    int ntile = 0;   // tiles finished by this warp (FP8 pair tiles)
    uint32_t dphase = 0;
    bool ok = true;
    for (;;) {
      // every lane waits; the warp proceeds only if all lanes saw the phase
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_mfull[ds]), dphase, &s_abort, tmo))) {
        ok = false;
        break;
      }
      TileDesc d = s_desc[ds];
      if (d.nkb < 0) break;
      if constexpr (kCta2 && C::kSwiglu) {   // this CTA's routed rows of the pair tile
        d.m0 += static_cast<int>(rank) * BM;
        d.rows = max(0, min(BM, d.rows - static_cast<int>(rank) * BM));
      }
      const float* sc = reinterpret_cast<const float*>(s_meta + ds * meta_bytes);
      const int* tok = reinterpret_cast<const int*>(sc + tok_off);
      const float* wt = reinterpret_cast<const float*>(tok + BM);
      // output column (of the first weight tile; CTA pairs: of this CTA's half)
      const int col =
          d.n_tile * kWRows + ((kCta2 && !C::kSwiglu) ? static_cast<int>(rank) * kTileN : 0) + row;

      if constexpr (kCta2 && C::kSwiglu && !kFP8) {
        // Token-major BF16 SwiGLU pair tile: TMEM lane = routed row s of this
        // CTA's half, columns [0, 128) the gate rows and [128, 256) the up rows
        // of h columns n_tile * 128 + [0, 128), accumulated over all of K.  This
        // warp: h columns [32 grp, +32) of its quadrant's 32 rows.
        const int s = row;
        const int buf = acc_n % C::kNumAcc;
        const uint32_t use = static_cast<uint32_t>(acc_n / C::kNumAcc);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bar_tfull[buf]), use & 1u, &s_abort, tmo))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                              buf * C::kAccCols + 32 * grp;
        float g[32], u[32];
        tmem_ld16(base, *reinterpret_cast<float(*)[16]>(&g[0]));
        tmem_ld16(base + 16, *reinterpret_cast<float(*)[16]>(&g[16]));
        tmem_ld16(base + kTileN, *reinterpret_cast<float(*)[16]>(&u[0]));
        tmem_ld16(base + kTileN + 16, *reinterpret_cast<float(*)[16]>(&u[16]));
        tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&g[0]));
        tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&g[16]));
        tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&u[0]));
        tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&u[16]));
        tc_fence_before();                             // the tile is in registers: release it
        __syncwarp();                                  // to the even CTA
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bar_tempty[buf]), 0));
        ++acc_n;
        if (s < d.rows) {
          // silu(g) * u with the fast exponential and division, as the
          // single-CTA BF16 SwiGLU epilogue; 32 bf16 = four 16-byte stores
          const int I = p.N / 2;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float h0 = __fdividef(g[j], 1.0f + __expf(-g[j])) * u[j];
            const float h1 = __fdividef(g[j + 1], 1.0f + __expf(-g[j + 1])) * u[j + 1];
            const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
            w[j / 2] = *reinterpret_cast<const uint32_t*>(&b);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                static_cast<size_t>(d.m0 + s) * I +
                                                d.n_tile * kTileN + 32 * grp);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      } else if constexpr (C::kTok) {
        // Token-major pair tile: TMEM lane = routed row s of the tile, 256
        // accumulator columns = the two weight tiles' rows.  This warp's 64
        // columns: store / scatter [64 grp, +64) of tile grp / 2; SwiGLU the
        // gate columns [32 grp, +32) and the matching up columns [128 + 32 grp,
        // +32), i.e. h columns n_tile * 128 + 32 grp + j.
        const int s = row;
        const uint32_t lrow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        const float* sw = sc + p.kb_per_split * BM;    // weight scales [2][kb_per_split]
        float acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
        for (int i = 0; i < d.nkb && ok; ++i) {
          const int a = acc_n;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bar_tfull[a % C::kNumAcc]),
                                    static_cast<uint32_t>(a / C::kNumAcc) & 1u, &s_abort, tmo))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = lrow + (a % C::kNumAcc) * C::kAccCols;
          const float sa = sc[i * BM + s];             // this row's activation scale
          const float fa = __fmul_rn(sa, sw[i]);       // a_scale * w_scale, rounded once
          const float fb = __fmul_rn(sa, sw[p.kb_per_split + i]);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c0 = C::kSwiglu ? (u < 2 ? 32 * grp + 16 * u : 128 + 32 * grp + 16 * (u - 2))
                                      : 64 * grp + 16 * u;
            const float f = C::kSwiglu ? (u < 2 ? fa : fb) : (grp < 2 ? fa : fb);
            float v[16];
            tmem_ld16(base + c0, v);
            tmem_ld_wait(v);
            if (u == 3) {                              // the K block is in registers: release it
              tc_fence_before();                       // (CTA pairs: to the even CTA)
              __syncwarp();
              if (lane == 0) {
                if constexpr (kCta2)
                  mbar_arrive_cluster(mapa_shared(smem_u32(&bar_tempty[a % C::kNumAcc]), 0));
                else
                  mbar_arrive(smem_u32(&bar_tempty[a % C::kNumAcc]));
              }
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2)
              fma2(acc[16 * u + j], acc[16 * u + j + 1], v[j], v[j + 1], f, f);
          }
          ++acc_n;
        }
        if (!ok) break;
        const bool live = s < d.rows;
        if constexpr (C::kSwiglu) {
          // h = silu(gate) * up in binary32 with the fast exponential and
          // division (each within a few ulp; the tile end is on the MMA's
          // critical path, since TMEM holds only two K blocks of the next
          // tile), into acc[0, 32)
          const int I = p.N / 2;
          float mx = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float e = __expf(-acc[j]);           // +inf for very negative g: h = -0
            acc[j] = __fmul_rn(__fdividef(acc[j], __fadd_rn(1.0f, e)), acc[32 + j]);
            mx = fmaxf(mx, fabsf(acc[j]));
          }
          // the row's 1x128 block = its 32 h columns in each of the quadrant's
          // four group warps: one exchange through shared memory (double-
          // buffered by tile) under a bounded mbarrier wait
          float* red = s_red + ((ntile & 1) * 4 + quad) * 128;   // [4 groups][32 lanes]
          red[grp * 32 + lane] = mx;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_red[quad]));
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_red[quad]),
                                                 static_cast<uint32_t>(ntile) & 1u, &s_abort,
                                                 tmo))) {
            ok = false;
            break;
          }
          const float amax =
              fmaxf(fmaxf(red[lane], red[32 + lane]), fmaxf(red[64 + lane], red[96 + lane]));
          uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          float scale = 0.0f;
          if (amax > 0.0f) {
            scale = __fdiv_rn(amax, 448.0f);
            const float inv = __fdiv_rn(1.0f, scale);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t c01 = cvt_e4m3x2(__fmul_rn(acc[4 * q], inv), __fmul_rn(acc[4 * q + 1], inv));
              const uint32_t c23 =
                  cvt_e4m3x2(__fmul_rn(acc[4 * q + 2], inv), __fmul_rn(acc[4 * q + 3], inv));
              w[q] = c01 | (c23 << 16);
            }
          }
          if (live) {
            if (grp == 0) p.out_scales[static_cast<size_t>(d.n_tile) * p.R + d.m0 + s] = scale;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                  static_cast<size_t>(d.m0 + s) * I +
                                                  d.n_tile * kTileN + 32 * grp);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        } else if (live) {
          const int c_out = d.n_tile * 2 * kTileN + 64 * grp;   // first output column
          if constexpr (kEpi == MOE_EPI_SCATTER) {
            const float wv = wt[s];
            float* o = static_cast<float*>(p.out) + static_cast<size_t>(tok[s]) * p.N + c_out;
#pragma unroll
            for (int j = 0; j < 64; j += 4)
              red_add_v4_f32(o + j, wv * acc[j], wv * acc[j + 1], wv * acc[j + 2], wv * acc[j + 3]);
          } else if constexpr (kEpi == MOE_EPI_STORE_BF16) {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                static_cast<size_t>(d.m0 + s) * p.N + c_out);
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
              __nv_bfloat162 b[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) b[q] = __floats2bfloat162_rn(acc[j + 2 * q], acc[j + 2 * q + 1]);
              o[j / 8] = *reinterpret_cast<const uint4*>(b);
            }
          } else {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) +
                                                  static_cast<size_t>(d.m0 + s) * p.N + c_out);
#pragma unroll
            for (int j = 0; j < 64; j += 4) o[j / 4] = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
          }
        }
        ++ntile;
      } else if constexpr (C::kFP8Pair) {
        // Two weight tiles per K block (adjacent tiles, or gate and up): each
        // thread promotes its weight row of both for its CW routed rows, in
        // chunks of 8 columns per tile (the accumulators fill the register
        // budget of 16 epilogue warps).
        constexpr int CW = C::kEpiCols;
        static_assert(CW == 16 || CW == 32, "pair-tile columns per warp");
        float acc_a[CW], acc_b[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          acc_a[j] = 0.0f;
          acc_b[j] = 0.0f;
        }
        const float* sw = sc + p.kb_per_split * BM;   // weight scales [2][kb_per_split]
        for (int i = 0; i < d.nkb && ok; ++i) {
          const int a = acc_n;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bar_tfull[a % C::kNumAcc]),
                                    static_cast<uint32_t>(a / C::kNumAcc) & 1u, &s_abort, tmo))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = lane_addr + (a % C::kNumAcc) * C::kAccCols;
          const float swa = sw[i], swb = sw[p.kb_per_split + i];
          const float* sav = sc + i * BM + c_lo;     // activation scales of this warp's rows
          // 8 columns of one tile at a time: [tile][chunk] in order, each load
          // waited for before its multiply-adds
#pragma unroll
          for (int u = 0; u < 2 * (CW / 8); ++u) {
            const int t = u & 1, c0 = (u >> 1) * 8;
            float v[8];
            tmem_ld8(base + t * BM + c0, v);
            tmem_ld_wait(v);
            if (u == 2 * (CW / 8) - 1) {             // the K block is in registers: release it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&bar_tempty[a % C::kNumAcc]));
            }
            float* acc = t ? acc_b : acc_a;
            const float wsc = t ? swb : swa;
#pragma unroll
            for (int q = 0; q < 8; q += 4) {
              const float4 s4 = *reinterpret_cast<const float4*>(sav + c0 + q);
              float f0, f1, f2, f3;                  // a_scale * w_scale, rounded once
              mul2(f0, f1, s4.x, s4.y, wsc, wsc);
              mul2(f2, f3, s4.z, s4.w, wsc, wsc);
              fma2(acc[c0 + q], acc[c0 + q + 1], v[q], v[q + 1], f0, f1);
              fma2(acc[c0 + q + 2], acc[c0 + q + 3], v[q + 2], v[q + 3], f2, f3);
            }
          }
          ++acc_n;
        }
        if (!ok) break;
        if constexpr (C::kSwiglu) {
          // h = silu(gate) * up = (g / (1 + exp(-g))) * u in binary32 for this
          // thread's h column n_tile * 128 + row and routed rows c_lo + j (the
          // fast exponential and division, each within a few ulp; the IEEE
          // division's slow path would push the 64 accumulators out of
          // registers); then the 1x128 rule over the tile's 128 h columns,
          // which are the 128 TMEM lanes of the group's four quadrant warps
          const int I = p.N / 2;
          float* h = acc_a;                          // h overwrites the gate accumulator
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const float e = __expf(-acc_a[j]);       // +inf for very negative g: h = -0
            h[j] = __fmul_rn(__fdividef(acc_a[j], __fadd_rn(1.0f, e)), acc_b[j]);
          }
          // reduce-scatter of the maxima over the warp: lane l ends with the
          // maximum over its quadrant's 32 h columns of routed row c_lo + l % CW
          // (the first step, over lane bit 4, reads |h| directly)
          float m[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if constexpr (CW == 16) {
              m[j] = fmaxf(fabsf(h[j]), __shfl_xor_sync(0xffffffffu, fabsf(h[j]), 16));
            } else {
              const bool hi = (lane & 16) != 0;
              const float send = fabsf(hi ? h[j] : h[j + 16]);
              const float keep = fabsf(hi ? h[j + 16] : h[j]);
              m[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
            }
          }
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < o; ++j) {
              const float send = hi ? m[j] : m[j + o];
              const float keep = hi ? m[j + o] : m[j];
              m[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
            }
          }
          // ... then over the four quadrant warps (double-buffered by tile)
          float* red = s_red + (grp * 2 + (ntile & 1)) * 128;   // [4 quadrants][32]
          if (lane < CW) red[quad * 32 + lane] = m[0];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_red[grp]));
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_red[grp]),
                                                 static_cast<uint32_t>(ntile) & 1u, &s_abort,
                                                 tmo))) {
            ok = false;
            break;
          }
          const int cl = lane % CW;
          const float amax = fmaxf(fmaxf(red[cl], red[32 + cl]), fmaxf(red[64 + cl], red[96 + cl]));
          float scale = 0.0f, inv = 0.0f;
          if (amax > 0.0f) {
            scale = __fdiv_rn(amax, 448.0f);
            inv = __fdiv_rn(1.0f, scale);
          }
          // block scales [I/128, R] (the quadrant-0 warp writes its group's rows)
          if (quad == 0 && lane < CW && c_lo + lane < d.rows)
            p.out_scales[static_cast<size_t>(d.n_tile) * p.R + d.m0 + c_lo + lane] = scale;
          // codes [R, I]: routed row c_lo + j, h column n_tile * 128 + row
          uint8_t* hq = static_cast<uint8_t*>(p.out) + static_cast<size_t>(d.m0 + c_lo) * I + col;
#pragma unroll
          for (int j = 0; j < CW; j += 2) {
            const float i0 = __shfl_sync(0xffffffffu, inv, j);
            const float i1 = __shfl_sync(0xffffffffu, inv, j + 1);
            const uint16_t q2 = cvt_e4m3x2(__fmul_rn(h[j], i0), __fmul_rn(h[j + 1], i1));
            // a block whose amax is 0 has all-zero codes
            if (c_lo + j < d.rows) hq[static_cast<size_t>(j) * I] = i0 > 0.0f ? (q2 & 0xff) : 0;
            if (c_lo + j + 1 < d.rows)
              hq[static_cast<size_t>(j + 1) * I] = i1 > 0.0f ? (q2 >> 8) : 0;
          }
        } else if constexpr (kEpi == MOE_EPI_SCATTER) {
          // both weight tiles' outputs of each routed row (columns col and col + 128)
          float* out = static_cast<float*>(p.out) + col;
#pragma unroll
          for (int s0 = 0; s0 < CW; s0 += 4) {
            if (c_lo + s0 < d.rows) {
              const int4 t4 = *reinterpret_cast<const int4*>(tok + c_lo + s0);
              const float4 w4 = *reinterpret_cast<const float4*>(wt + c_lo + s0);
              const int tk[4] = {t4.x, t4.y, t4.z, t4.w};
              const float ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (c_lo + s0 + j < d.rows) {
                  float* o = out + static_cast<size_t>(tk[j]) * p.N;
                  red_add_f32(o, ww[j] * acc_a[s0 + j]);
                  red_add_f32(o + kTileN, ww[j] * acc_b[s0 + j]);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            if (c_lo + j < d.rows) {
              const size_t o = static_cast<size_t>(d.m0 + c_lo + j) * p.N + col;
              if constexpr (kEpi == MOE_EPI_STORE_BF16) {
                static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(acc_a[j]);
                static_cast<__nv_bfloat16*>(p.out)[o + kTileN] = __float2bfloat16_rn(acc_b[j]);
              } else {
                static_cast<float*>(p.out)[o] = acc_a[j];
                static_cast<float*>(p.out)[o + kTileN] = acc_b[j];
              }
            }
          }
        }
        ++ntile;
      } else if constexpr (kFP8) {
        constexpr int CW = C::kEpiCols;
        float acc[CW];
#pragma unroll
        for (int s = 0; s < CW; ++s) acc[s] = 0.0f;
        if constexpr (C::kKbGroup == 1 && BM >= 64) {
          // One K block per TMEM buffer; this warp's columns are read in
          // 32-column chunks with two register buffers: the next chunk's load
          // is in flight while this chunk is folded in, and the buffer is
          // released as soon as the last chunk has arrived (before that
          // chunk's multiply-adds).  Two columns per packed multiply-add.
          constexpr int kCh = 32, kNCh = CW / kCh;
          static_assert(CW % kCh == 0, "chunks");
          for (int i = 0; i < d.nkb && ok; ++i) {
            const int a = acc_n;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&bar_tfull[a % C::kNumAcc]),
                                      static_cast<uint32_t>(a / C::kNumAcc) & 1u, &s_abort, tmo))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t base = lane_addr + (a % C::kNumAcc) * C::kAccCols;
            const float4* scb = reinterpret_cast<const float4*>(sc + i * BM + c_lo);
            float va[kCh], vb[kCh];
            tmem_ld16(base, *reinterpret_cast<float(*)[16]>(&va[0]));
            tmem_ld16(base + 16, *reinterpret_cast<float(*)[16]>(&va[16]));
            tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&va[0]));
            tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&va[16]));
#pragma unroll
            for (int ch = 0; ch < kNCh; ++ch) {
              float* cur = (ch & 1) ? vb : va;
              float* nxt = (ch & 1) ? va : vb;
              if (ch + 1 < kNCh) {
                tmem_ld16(base + (ch + 1) * kCh, *reinterpret_cast<float(*)[16]>(nxt));
                tmem_ld16(base + (ch + 1) * kCh + 16, *reinterpret_cast<float(*)[16]>(nxt + 16));
              } else {
                // every chunk of this K block is in registers: hand the buffer back
                // (CTA pairs: to the even CTA, which issues the MMAs)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                  if constexpr (kCta2)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&bar_tempty[a % C::kNumAcc]), 0));
                  else
                    mbar_arrive(smem_u32(&bar_tempty[a % C::kNumAcc]));
                }
              }
#pragma unroll
              for (int j = 0; j < kCh; j += 4) {
                const float4 f = scb[(ch * kCh + j) / 4];
                fma2(acc[ch * kCh + j], acc[ch * kCh + j + 1], cur[j], cur[j + 1], f.x, f.y);
                fma2(acc[ch * kCh + j + 2], acc[ch * kCh + j + 3], cur[j + 2], cur[j + 3], f.z, f.w);
              }
              if (ch + 1 < kNCh) {
                tmem_ld_wait(*reinterpret_cast<float(*)[16]>(nxt));
                tmem_ld_wait(*reinterpret_cast<float(*)[16]>(nxt + 16));
              }
            }
            ++acc_n;
          }
        } else {
          for (int i = 0; i < d.nkb && ok; i += C::kKbGroup) {
            const int ng = min(C::kKbGroup, d.nkb - i);
            // wait for the partials of K blocks i .. i+ng-1
            bool got = true;
            for (int g = 0; g < ng; ++g) {
              const int a = acc_n + g;
              got = got && mbar_wait(smem_u32(&bar_tfull[a % C::kNumAcc]),
                                     static_cast<uint32_t>(a / C::kNumAcc) & 1u, &s_abort, tmo);
            }
            if (!__all_sync(0xffffffffu, got)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < BM; c0 += C::kLdCols) {
              float v[C::kKbGroup][C::kLdCols];
#pragma unroll
              for (int g = 0; g < C::kKbGroup; ++g) {
                if (g < ng) {
                  const uint32_t base = lane_addr + ((acc_n + g) % C::kNumAcc) * C::kAccCols + c0;
#pragma unroll
                  for (int j = 0; j < C::kLdCols; j += 16)
                    tmem_ld16(base + j, *reinterpret_cast<float(*)[16]>(&v[g][j]));
                }
              }
#pragma unroll
              for (int g = 0; g < C::kKbGroup; ++g) {
                if (g < ng) {
#pragma unroll
                  for (int j = 0; j < C::kLdCols; j += 16)
                    tmem_ld_wait(*reinterpret_cast<float(*)[16]>(&v[g][j]));
                }
              }
#pragma unroll
              for (int g = 0; g < C::kKbGroup; ++g) {
                if (g < ng) {
                  // scale products of this K block (16-byte aligned, broadcast reads)
                  const float4* scg = reinterpret_cast<const float4*>(sc + (i + g) * BM + c0);
#pragma unroll
                  for (int j = 0; j < C::kLdCols; j += 4) {
                    const float4 f = scg[j / 4];
                    acc[c0 + j] = fmaf(v[g][j], f.x, acc[c0 + j]);
                    acc[c0 + j + 1] = fmaf(v[g][j + 1], f.y, acc[c0 + j + 1]);
                    acc[c0 + j + 2] = fmaf(v[g][j + 2], f.z, acc[c0 + j + 2]);
                    acc[c0 + j + 3] = fmaf(v[g][j + 3], f.w, acc[c0 + j + 3]);
                  }
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
              for (int g = 0; g < ng; ++g) mbar_arrive(smem_u32(&bar_tempty[(acc_n + g) % C::kNumAcc]));
            acc_n += ng;
          }
        }
        if (!ok) break;
        if constexpr (kEpi == MOE_EPI_SCATTER) {
          // tokens and route weights 8 rows at a time (vector loads), then
          // the 8 row reductions back to back
          float* out = static_cast<float*>(p.out) + col;
#pragma unroll
          for (int s0 = 0; s0 < CW; s0 += 8) {
            if (c_lo + s0 < d.rows) {
              const int4 t0 = *reinterpret_cast<const int4*>(tok + c_lo + s0);
              const int4 t1 = *reinterpret_cast<const int4*>(tok + c_lo + s0 + 4);
              const float4 w0 = *reinterpret_cast<const float4*>(wt + c_lo + s0);
              const float4 w1 = *reinterpret_cast<const float4*>(wt + c_lo + s0 + 4);
              const int tk[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
              const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (c_lo + s0 + j < d.rows)
                  red_add_f32(out + static_cast<size_t>(tk[j]) * p.N, ww[j] * acc[s0 + j]);
            }
          }
        } else if constexpr (kEpi == MOE_EPI_STORE_BF16) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int s = 0; s < CW; ++s) {
            if (c_lo + s < d.rows)
              out[static_cast<size_t>(d.m0 + c_lo + s) * p.N + col] = __float2bfloat16_rn(acc[s]);
          }
        } else {
          float* out = static_cast<float*>(p.out);
#pragma unroll
          for (int s = 0; s < CW; ++s) {
            if (c_lo + s < d.rows) out[static_cast<size_t>(d.m0 + c_lo + s) * p.N + col] = acc[s];
          }
        }
      } else {
        const int buf = acc_n % C::kNumAcc;
        const uint32_t use = static_cast<uint32_t>(acc_n / C::kNumAcc);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bar_tfull[buf]), use & 1u, &s_abort, tmo))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this warp's columns: [c_lo, c_lo + kEpiCols) (lane_addr includes c_lo)
        for (int c0 = 0; c0 < C::kEpiCols && c_lo + c0 < d.rows; c0 += 16) {
          float v[16];
          tmem_ld16(lane_addr + buf * C::kAccCols + c0, v);
          const int s0 = c_lo + c0;  // routed row of v[0]
          if constexpr (C::kSwiglu) {
            float u[16];
            tmem_ld16(lane_addr + buf * C::kAccCols + BM + c0, u);
            tmem_ld_wait(v);
            tmem_ld_wait(u);
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
            const int I = p.N / 2;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (s0 + j < d.rows) {
                // silu(g) * u with the fast exponential and division (relative
                // error ~1e-6, far inside the bf16 rounding of h); for very
                // negative g the denominator overflows and silu -> 0
                const float g = v[j];
                const float h = __fdividef(g, 1.0f + __expf(-g)) * u[j];
                out[static_cast<size_t>(d.m0 + s0 + j) * I + col] = __float2bfloat16_rn(h);
              }
            }
          } else {
            // wide tiles: the second weight tile's accumulator is BM columns on,
            // its output columns 128 on
            float v2[16];
            if constexpr (kWide) tmem_ld16(lane_addr + buf * C::kAccCols + BM + c0, v2);
            tmem_ld_wait(v);
            if constexpr (kWide) tmem_ld_wait(v2);
#pragma unroll
            for (int h = 0; h < (kWide ? 2 : 1); ++h) {
              const float* vh = h ? v2 : v;
              const int colh = col + h * kTileN;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (s0 + j < d.rows) {
                  const size_t r = static_cast<size_t>(d.m0 + s0 + j);
                  if constexpr (kEpi == MOE_EPI_SCATTER)
                    red_add_f32(static_cast<float*>(p.out) + static_cast<size_t>(tok[s0 + j]) * p.N + colh,
                                wt[s0 + j] * vh[j]);
                  else if constexpr (kEpi == MOE_EPI_STORE_BF16)
                    static_cast<__nv_bfloat16*>(p.out)[r * p.N + colh] = __float2bfloat16_rn(vh[j]);
                  else
                    static_cast<float*>(p.out)[r * p.N + colh] = vh[j];
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {   // (CTA pairs: to the even CTA)
          if constexpr (kCta2) mbar_arrive_cluster(mapa_shared(smem_u32(&bar_tempty[buf]), 0));
          else mbar_arrive(smem_u32(&bar_tempty[buf]));
        }
        ++acc_n;
      }
      // this tile's descriptor and metadata slot may now be reused
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_dempty[ds]));
      if (++ds == C::kRing) { ds = 0; dphase ^= 1u; }
    }
    if (!ok) {
      set_error(p.ctrl, MOE_ERR_TIMEOUT, 3);
      s_abort = 1;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  // CTA pairs: neither CTA frees its TMEM or leaves (its shared memory and
  // mbarriers) until the other is done with them
  if constexpr (kCta2) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kCta2) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.done_ctr, 1u);
    if (prev == gridDim.x - 1) {  // last CTA: leave the counters zeroed for the next launch
      atomicExch(p.queue_ctr, 0u);
      atomicExch(p.done_ctr, 0u);
      __threadfence();
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side: instantiations, launch.

struct GemmVariant {
  const void* fn;
  int stage_bytes;
  int threads;
};

template <int BM, bool kFP8, int kEpi, bool kGather, bool kWide = false, bool kCta2 = false>
GemmVariant variant() {
  using C = Cfg<BM, kFP8, kEpi, kWide, kCta2>;
  return GemmVariant{
      reinterpret_cast<const void*>(&grouped_gemm_kernel<BM, kFP8, kEpi, kGather, kWide, kCta2>),
      C::kStageBytes, C::kThreads};
}

// Wide tiles: store / scatter epilogues; BF16 at block_m 128 or 256, FP8 at 128.
template <int kEpi>
bool pick_wide(bool fp8, int bm, GemmVariant& v) {
  if (fp8) {
    if (bm == 128) { v = variant<128, true, kEpi, false, true>(); return true; }
    return false;
  }
  if (bm == 128) { v = variant<128, false, kEpi, false, true>(); return true; }
  if (bm == 256) { v = variant<256, false, kEpi, false, true>(); return true; }
  return false;
}

template <bool kFP8, int kEpi, bool kGather>
bool pick_bm(int bm, GemmVariant& v) {
  switch (bm) {
    case 16: v = variant<16, kFP8, kEpi, kGather>(); return true;
    case 32: v = variant<32, kFP8, kEpi, kGather>(); return true;
    case 64: v = variant<64, kFP8, kEpi, kGather>(); return true;
    case 128: v = variant<128, kFP8, kEpi, kGather>(); return true;
    default: break;
  }
  if constexpr (!kFP8) {
    if (bm == 256) { v = variant<256, kFP8, kEpi, kGather>(); return true; }
  }
  return false;
}

// Gathered rows are built for the FP8 GEMM (every epilogue) and the BF16
// gated up projection (the first GEMM of the BF16 forward).
bool select_gemm_variant(bool fp8, int epi, int bm, bool gather, bool wide, bool cta2,
                         GemmVariant& v) {
  if (cta2) {
    if (!gemm_cta2_supported(fp8, epi, bm) || gather || wide) return false;
    if (!fp8 && epi == MOE_EPI_SWIGLU)   // 128 routed rows per CTA: block_m 256 per pair
      v = variant<128, false, MOE_EPI_SWIGLU, false, false, true>();
    else if (!fp8)
      v = epi == MOE_EPI_SCATTER ? variant<256, false, MOE_EPI_SCATTER, false, false, true>()
                                 : variant<256, false, MOE_EPI_STORE_BF16, false, false, true>();
    else if (epi == MOE_EPI_SWIGLU)
      v = variant<128, true, MOE_EPI_SWIGLU, false, false, true>();
    else
      v = variant<128, true, MOE_EPI_SCATTER, false, false, true>();
    return true;
  }
  if (wide) {
    if (gather) return false;
    if (epi == MOE_EPI_SCATTER) return pick_wide<MOE_EPI_SCATTER>(fp8, bm, v);
    if (epi == MOE_EPI_STORE) return pick_wide<MOE_EPI_STORE>(fp8, bm, v);
    if (epi == MOE_EPI_STORE_BF16) return pick_wide<MOE_EPI_STORE_BF16>(fp8, bm, v);
    return false;
  }
  if (fp8 && epi == MOE_EPI_SWIGLU) {
    // gate + up pair tiles with the SwiGLU + 1x128 re-quantisation epilogue
    if (gather) return false;
    switch (bm) {
      case 16: v = variant<16, true, MOE_EPI_SWIGLU, false>(); return true;
      case 32: v = variant<32, true, MOE_EPI_SWIGLU, false>(); return true;
      case 64: v = variant<64, true, MOE_EPI_SWIGLU, false>(); return true;
      case 128: v = variant<128, true, MOE_EPI_SWIGLU, false>(); return true;
      default: return false;
    }
  }
  if (fp8) {
    if (epi == MOE_EPI_SCATTER)
      return gather ? pick_bm<true, MOE_EPI_SCATTER, true>(bm, v)
                    : pick_bm<true, MOE_EPI_SCATTER, false>(bm, v);
    if (epi == MOE_EPI_STORE)
      return gather ? pick_bm<true, MOE_EPI_STORE, true>(bm, v)
                    : pick_bm<true, MOE_EPI_STORE, false>(bm, v);
    if (epi == MOE_EPI_STORE_BF16)
      return gather ? pick_bm<true, MOE_EPI_STORE_BF16, true>(bm, v)
                    : pick_bm<true, MOE_EPI_STORE_BF16, false>(bm, v);
    return false;
  }
  if (epi == MOE_EPI_SWIGLU)
    return gather ? pick_bm<false, MOE_EPI_SWIGLU, true>(bm, v)
                  : pick_bm<false, MOE_EPI_SWIGLU, false>(bm, v);
  if (gather) return false;
  if (epi == MOE_EPI_SCATTER) return pick_bm<false, MOE_EPI_SCATTER, false>(bm, v);
  if (epi == MOE_EPI_STORE) return pick_bm<false, MOE_EPI_STORE, false>(bm, v);
  if (epi == MOE_EPI_STORE_BF16) return pick_bm<false, MOE_EPI_STORE_BF16, false>(bm, v);
  return false;
}

bool gemm_gather_supported(bool fp8, int epi) { return fp8 || epi == MOE_EPI_SWIGLU; }

bool gemm_wide_supported(bool fp8, int epi, int bm) {
  return epi != MOE_EPI_SWIGLU && (fp8 ? bm == 128 : (bm == 128 || bm == 256));
}

bool gemm_cta2_supported(bool fp8, int epi, int bm) {
  if (fp8) return bm == 128 && (epi == MOE_EPI_SCATTER || epi == MOE_EPI_SWIGLU);
  return bm == 256 && (epi == MOE_EPI_SCATTER || epi == MOE_EPI_STORE_BF16 ||
                       epi == MOE_EPI_SWIGLU);
}

int gemm_stage_bytes(bool fp8, int epi, int bm, bool wide, bool cta2) {
  GemmVariant v;
  if (!select_gemm_variant(fp8, epi, bm, false, wide, cta2, v)) return 0;
  return v.stage_bytes;
}

// Clusters of two CTAs of the CTA-pair kernels (one CTA per SM, at most 608
// threads) that can be resident at once; 0 if unknown.  Cached per device: the
// first call sets the kernel's shared-memory limit and asks the occupancy
// calculator — unless `query` is false (a caller inside a stream capture),
// which then gets 0 and the single-CTA form.
int gemm_cta2_max_clusters(bool query) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0 || !query) return cached[dev];
  const GemmVariant v = variant<128, true, MOE_EPI_SCATTER, false, false, true>();
  // more than half of an SM's shared memory (one CTA per SM), leaving the
  // per-block limit room for the kernel's static shared memory
  constexpr int kSmem = 160 * 1024;
  if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(v.threads);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, v.fn, &cfg) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

int gemm_table_bytes(int E) { return (2 * (E + 1) * 4 + 15) & ~15; }

int gemm_rows_bytes(bool fp8, int bm) { return ring_slots(fp8, bm) * bm * 4; }

int gemm_meta_bytes(bool fp8, int bm, int kb_per_split, bool pair) {
  return ring_slots(fp8, bm) * meta_slot_bytes(fp8, bm, kb_per_split, pair);
}

int gemm_extra_bytes(bool fp8, int epi, int bm, bool gather) {
  if (gather) return gemm_rows_bytes(fp8, bm);
  if (fp8 && epi == MOE_EPI_SWIGLU) return swiglu_red_bytes(bm >= 32 ? bm / 32 : 1);
  return 0;
}

cudaError_t launch_grouped_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_a,
                                const GemmParams& p, bool fp8, int epi, int bm, int num_ctas,
                                cudaStream_t stream, bool pdl) {
  GemmVariant v;
  if (!select_gemm_variant(fp8, epi, bm, p.gather != 0, p.wide != 0, p.cta2 != 0, v))
    return cudaErrorInvalidValue;
  if (p.cta2 && (num_ctas < 2 || num_ctas % 2 != 0)) return cudaErrorInvalidValue;
  if (p.sk != 1 && p.sk != 2 && p.sk != 4) return cudaErrorInvalidValue;
  const bool pair = fp8 && (p.wide != 0 || epi == MOE_EPI_SWIGLU);
  const size_t smem = 1024 + static_cast<size_t>(p.num_stages) * p.sk * v.stage_bytes +
                      gemm_meta_bytes(fp8, bm, p.kb_per_split, pair) + gemm_table_bytes(p.E) +
                      gemm_extra_bytes(fp8, epi, bm, p.gather != 0);
  cudaError_t err = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(v.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(v.threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.cta2) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  void* args[] = {const_cast<CUtensorMap*>(&tmap_w), const_cast<CUtensorMap*>(&tmap_a),
                  const_cast<GemmParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, v.fn, args);
}

}  // namespace moe
