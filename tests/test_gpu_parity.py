"""GPU parity: every step of the path through the C ABI against the oracle.

Bit-exact: routing ids and weights, counts, offsets, tile offsets, the stable
permutation and its inverse, E4M3 codes and scales.  Within tolerance
(rel-L2 <= 5e-3, max-abs <= 1e-2 max|ref| against the oracle's binary64 sum
over the same quantised values): the grouped GEMM and the fused forward."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (THREADS, assert_close, bits, ensure_built, fp8_device_inputs, np_,
                         run_forward_bf16, run_forward_fp8, sample_tokens)
from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


# ------------------------------------------------------------------ route
@pytest.mark.parametrize("M,E,k,softcap,renorm,scale", [
    (16, 8, 2, 0.0, 1, 1.0), (16, 8, 2, 30.0, 1, 1.0), (128, 256, 8, 30.0, 1, 1.0),
    (333, 33, 5, 30.0, 1, 20.0), (64, 1024, 32, 0.0, 1, 1.0), (7, 4, 4, 0.0, 0, 1.0),
    (100, 256, 8, 30.0, 0, 5.0), (1, 1, 1, 0.0, 1, 1.0), (50, 64, 1, 7.5, 1, 3.0)])
def test_route_bit_exact(M, E, k, softcap, renorm, scale):
    g = torch.Generator().manual_seed(M * 7 + E)
    logits = (torch.randn(M, E, generator=g) * scale).float()
    ids, w = L.route(logits.cuda(), k, softcap=softcap, renorm=renorm)
    rid, rw = oracle.route(logits.numpy(), k, softcap=softcap, renorm=renorm)
    assert np.array_equal(np_(ids), rid)
    assert np.array_equal(np_(w).view(np.uint32), rw.view(np.uint32))


def test_route_ties_and_large_values():
    logits = torch.zeros(4, 40)
    logits[0, [3, 9, 17, 33]] = 2.0           # four-way tie for top-4
    logits[1] = 1.0                           # all equal
    logits[2] = torch.arange(40).float() * 1e3  # large values, softcap saturates
    logits[3, ::2] = -50.0
    for c in (0.0, 30.0):
        ids, w = L.route(logits.cuda(), 4, softcap=c)
        rid, rw = oracle.route(logits.numpy(), 4, softcap=c)
        assert np.array_equal(np_(ids), rid)
        assert np.array_equal(np_(w).view(np.uint32), rw.view(np.uint32))


@pytest.mark.parametrize("name", ["qwen_small_batch_fp8", "skewed_large_batch_fp8"])
def test_route_configs(name):
    d = inputs.make_fp8_inputs(dict(inputs.FP8_CONFIGS[name], E=inputs.FP8_CONFIGS[name]["E"],
                                    N=128, K=128))  # weights are not used here
    ids, w = L.route(d["logits"].cuda(), d["cfg"]["k"], softcap=d["cfg"]["softcap"])
    rid, rw = oracle.route(d["logits"].numpy(), d["cfg"]["k"], softcap=d["cfg"]["softcap"])
    assert np.array_equal(np_(ids), rid)
    assert np.array_equal(np_(w).view(np.uint32), rw.view(np.uint32))


# ------------------------------------------------------------------ layout
def _layout_case(ids_np, E, bm):
    ws = L.new_workspace(L.CTRL_BYTES)
    got = L.layout(torch.from_numpy(ids_np).cuda(), E, bm, ws)
    torch.cuda.synchronize()
    ref = oracle.layout(ids_np, E, block_m=bm)
    for key in ("counts", "offsets", "sorted_route_ids", "route_slot", "tile_offsets"):
        assert np.array_equal(np_(got[key]), ref[key]), key
    assert L.get_error(ws) == L.MOE_OK


@pytest.mark.parametrize("M,E,k,bm", [(16, 8, 2, 16), (128, 256, 8, 16), (4096, 256, 8, 128),
                                      (8192, 16, 8, 256), (16384, 8, 2, 64), (1, 1024, 7, 32),
                                      (999, 1024, 32, 16), (3, 5, 5, 256)])
def test_layout_bit_exact(M, E, k, bm):
    g = torch.Generator().manual_seed(M + E + k)
    ids = torch.rand(M, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32).numpy()
    _layout_case(ids, E, bm)


def test_layout_skewed_empty_and_single_expert():
    ids = np.zeros((5000, 2), np.int32)
    ids[:, 1] = 7
    ids[17, 0] = 3
    _layout_case(ids, 9, 16)
    _layout_case(np.zeros((300, 1), np.int32), 1, 128)


def test_layout_reports_bad_ids():
    ids = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    ws = L.new_workspace(L.CTRL_BYTES)
    got = L.layout(ids, 4, 16, ws)
    assert L.get_error(ws) == L.MOE_ERR_DEVICE_FAULT
    assert np_(got["route_slot"])[3] == -1
    assert L.get_error(ws) == L.MOE_OK           # reading clears the status


# ------------------------------------------------------------------ quantise + gather
@pytest.mark.parametrize("M,K,k", [(16, 256, 2), (128, 2048, 8), (37, 384, 3), (5, 8192, 1),
                                   (64, 16384, 2), (333, 128, 4), (4096, 2048, 8), (5000, 1024, 6),
                                   (100, 128, 32), (77, 256, 20)])
def test_quant_gather_bit_exact(M, K, k):
    """Includes batches large enough for 32 elements per thread (one wave),
    and more routes per token than the token has threads (K/16 < top_k)."""
    g = torch.Generator().manual_seed(M + K)
    x = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g) * 4)).to(torch.bfloat16)
    x[0, :128] = 0.0                                   # an all-zero block
    x[-1, -128:] = -0.0
    E = max(8, k)
    ids = torch.rand(M, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32).numpy()
    lay = oracle.layout(ids, E)
    slot = torch.from_numpy(lay["route_slot"]).cuda()
    acc = torch.full((M, 256), 7.0, device="cuda")
    a_q, a_s = L.quant_gather(x.cuda(), k, slot, zero_acc=acc)
    rq, rs = oracle.quant_gather(bits(x), k, lay["route_slot"])
    assert np.array_equal(np_(a_q), rq)
    assert np.array_equal(np_(a_s).view(np.uint32), rs.view(np.uint32))
    assert torch.count_nonzero(acc).item() == 0


# ------------------------------------------------------------------ grouped GEMM
def _fp8_gemm_case(M, K, N, E, k, bm, epilogue, sched=L.SCHED_QUEUE, k_splits=0, seed=0,
                   skew=0.0, num_ctas=0, cta_pairs=0):
    d = inputs.make_fp8_inputs(dict(M=M, K=K, N=N, E=E, k=k, softcap=0.0, zipf_bias=skew),
                               seed=seed)
    rid, rw = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])
    Y = oracle.grouped_gemm_fp8(a_q, a_s, d["w_q"].numpy(), d["w_scales"].numpy(),
                                lay["offsets"], threads=THREADS)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = L.new_workspace(L.CTRL_BYTES)
    R = M * k
    if epilogue == L.EPI_STORE_BF16:
        out = torch.zeros(R, N, dtype=torch.bfloat16, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_STORE_BF16, a=cu(a_q), a_scales=cu(a_s),
                       w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                       tile_offsets=cu(lay["tile_offsets"]), out=out, ws=ws, block_m=bm,
                       sched=sched, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert L.get_error(ws) == L.MOE_OK
        assert_close(out, Y, "fp8 store bf16")
    elif epilogue == L.EPI_STORE:
        out = torch.zeros(R, N, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_STORE, a=cu(a_q), a_scales=cu(a_s),
                       w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                       tile_offsets=cu(lay["tile_offsets"]), out=out, ws=ws, block_m=bm,
                       sched=sched, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert L.get_error(ws) == L.MOE_OK
        assert_close(out, Y, "fp8 store")
    else:
        out = torch.zeros(M, N, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER, a=cu(a_q), a_scales=cu(a_s),
                       w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                       tile_offsets=cu(lay["tile_offsets"]), out=out, ws=ws, block_m=bm,
                       sorted_route_ids=cu(lay["sorted_route_ids"]), route_weights=cu(rw),
                       M=M, top_k=k, sched=sched, k_splits=k_splits, num_ctas=num_ctas,
                       cta_pairs=cta_pairs)
        torch.cuda.synchronize()
        assert L.get_error(ws) == L.MOE_OK
        ref = oracle.scatter(Y, lay["route_slot"], rw)
        assert_close(out, ref, "fp8 scatter")


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_gemm_fp8_store_tiles_and_ragged_tail(bm):
    _fp8_gemm_case(M=300, K=512, N=256, E=16, k=4, bm=bm, epilogue=L.EPI_STORE)


@pytest.mark.parametrize("bm", [16, 128])
def test_gemm_fp8_store_bf16_rows(bm):
    """Expert-compact rows rounded to bf16 (the large-batch forward's epilogue)."""
    _fp8_gemm_case(M=300, K=1024, N=256, E=16, k=4, bm=bm, epilogue=L.EPI_STORE_BF16, skew=1.0)


@pytest.mark.parametrize("bm,sched,ks", [(16, L.SCHED_QUEUE, 1), (64, L.SCHED_STATIC, 1),
                                         (32, L.SCHED_QUEUE, 4), (128, L.SCHED_QUEUE, 0)])
def test_gemm_fp8_scatter(bm, sched, ks):
    _fp8_gemm_case(M=257, K=1024, N=384, E=8, k=2, bm=bm, epilogue=L.EPI_SCATTER, sched=sched,
                   k_splits=ks, skew=1.5)


def test_gemm_fp8_few_ctas_many_tiles():
    """Eight persistent CTAs loop over many tiles (the smem ring wraps many times)."""
    _fp8_gemm_case(M=512, K=2048, N=512, E=4, k=2, bm=64, epilogue=L.EPI_SCATTER, num_ctas=8)


@pytest.mark.parametrize("epi,sched,ks,ctas", [
    (L.EPI_SCATTER, L.SCHED_QUEUE, 1, 0), (L.EPI_SCATTER, L.SCHED_STATIC, 1, 0),
    (L.EPI_SCATTER, L.SCHED_QUEUE, 2, 0), (L.EPI_SCATTER, L.SCHED_QUEUE, 0, 8),
    (L.EPI_STORE, L.SCHED_QUEUE, 0, 0), (L.EPI_STORE_BF16, L.SCHED_QUEUE, 0, 5)])
def test_gemm_fp8_wide_tiles(epi, sched, ks, ctas):
    """128 routed rows against two adjacent 128-row weight tiles per tile (N a
    multiple of 256): one TMEM buffer per K block holds both tiles' partial
    products, four epilogue warps per lane quadrant promote them; ragged
    expert tiles, K splits, few CTAs looping over many tiles."""
    _fp8_gemm_case(M=700, K=1024, N=512, E=8, k=3, bm=128, epilogue=epi, sched=sched,
                   k_splits=ks, skew=1.5, num_ctas=ctas)


@pytest.mark.parametrize("M,E,k,N,ctas,skew", [
    (2000, 4, 2, 1024, 4, 1.0),   # two pairs loop over many tiles; the last tiles in K halves
    (3, 8, 2, 512, 0, 0.0),       # fewer tiles than pairs, most experts empty
    (700, 8, 3, 512, 3, 1.5),     # an odd grid: one pair
    (700, 8, 3, 512, 1, 1.5),     # one CTA: the single-CTA form of the 256-row tile
])
def test_gemm_fp8_scatter_cta_pairs(M, E, k, N, ctas, skew):
    """FP8 scatter at 128 routed rows with N a multiple of 256: a cluster of two
    CTAs computes each 256-row weight tile (one M = 256 MMA per K step, each
    CTA holding its 128 weight rows, half of the routed rows and its own
    accumulator); checked element by element against the oracle."""
    assert L.gemm_cta_pairs() > 0, "the CTA-pair form is not in use on this device"
    _fp8_gemm_case(M=M, K=2048, N=N, E=E, k=k, bm=128, epilogue=L.EPI_SCATTER, skew=skew,
                   num_ctas=ctas)


@pytest.mark.parametrize("case", ["fp8_scatter_one_weight_tile", "fp8_scatter_one_expert",
                                  "fp8_swiglu_one_h_tile", "bf16_scatter_one_k_block",
                                  "bf16_swiglu_exact_tile"])
def test_gemm_cta_pairs_edges(case):
    """CTA pairs at the edges of their tilings: a single 256-row weight tile
    (N = 256), every route on one expert, a single 128-column h tile, a single
    64-deep BF16 K block, and a pair tile filled exactly (256 routed rows)."""
    assert L.gemm_cta_pairs() > 0, "the CTA-pair form is not in use on this device"
    if case == "fp8_scatter_one_weight_tile":
        _fp8_gemm_case(M=300, K=512, N=256, E=8, k=2, bm=128, epilogue=L.EPI_SCATTER, skew=1.0)
    elif case == "fp8_scatter_one_expert":
        _fp8_gemm_case(M=400, K=384, N=512, E=1, k=1, bm=128, epilogue=L.EPI_SCATTER)
    elif case == "fp8_swiglu_one_h_tile":
        _fp8_swiglu_case(M=300, K=512, I=128, E=4, k=2, bm=128, skew=1.0)
    elif case == "bf16_scatter_one_k_block":
        _bf16_gemm_case(R_tokens=300, K=64, N=512, E=4, k=2, bm=256, epilogue=L.EPI_SCATTER)
    else:
        _bf16_gemm_case(R_tokens=128, K=256, N=256, E=1, k=2, bm=256, epilogue=L.EPI_SWIGLU)


@pytest.mark.parametrize("form", ["fp8_scatter", "fp8_swiglu", "bf16_scatter", "bf16_swiglu"])
def test_gemm_cta_pairs_off(form):
    """cta_pairs = -1: shapes that have a CTA-pair form run single CTAs."""
    if form == "fp8_scatter":
        _fp8_gemm_case(M=700, K=1024, N=512, E=8, k=3, bm=128, epilogue=L.EPI_SCATTER, skew=1.5,
                       cta_pairs=-1)
    elif form == "fp8_swiglu":
        _fp8_swiglu_case(M=700, K=1024, I=256, E=8, k=3, bm=128, skew=1.5, cta_pairs=-1)
    else:
        _bf16_gemm_case(R_tokens=600, K=512, N=512, E=8, k=2, bm=256,
                        epilogue=L.EPI_SCATTER if form == "bf16_scatter" else L.EPI_SWIGLU,
                        cta_pairs=-1)


def _e4m3_order(c: np.ndarray) -> np.ndarray:
    """Signed position of an E4M3 code on the number line; 0x00 and 0x80 both 0."""
    c = c.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _fp8_swiglu_case(M, K, I, E, k, bm, sched=L.SCHED_QUEUE, num_ctas=0, skew=1.0, seed=0,
                     cta_pairs=0):
    """The FP8 SWIGLU epilogue (gate rows [0, I), up rows [I, 2I) of [E, 2I, K])
    against the oracle's pipeline: binary64 up projection of the same codes
    rounded to binary32, then its SwiGLU + 1x128 rule.  The device accumulates
    in fp32 in another order, so an h on an E4M3 rounding boundary may take the
    neighbouring code: codes equal or one step apart (at most 0.2 %), block
    scales within 3e-5 relative, dequantised h within the output tolerance."""
    d = inputs.make_fp8_inputs(dict(M=M, K=K, N=2 * I, E=E, k=k, softcap=0.0, zipf_bias=skew),
                               seed=seed)
    rid, _ = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])
    gu = oracle.grouped_gemm_fp8(a_q, a_s, d["w_q"].numpy(), d["w_scales"].numpy(),
                                 lay["offsets"], threads=THREADS).astype(np.float32)
    hq_ref, hs_ref = oracle.swiglu_quant(gu)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    R = M * k
    h_q = torch.full((R, I), 0x7F, dtype=torch.uint8, device="cuda")
    h_s = torch.full((I // 128, R), -1.0, device="cuda")
    ws = L.new_workspace(L.CTRL_BYTES)
    L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SWIGLU, a=cu(a_q), a_scales=cu(a_s),
                   w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                   tile_offsets=cu(lay["tile_offsets"]), out=h_q, out_scales=h_s, ws=ws,
                   block_m=bm, sched=sched, num_ctas=num_ctas, cta_pairs=cta_pairs)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    hq, hs = np_(h_q), np_(h_s)
    assert np.all(np.abs(hs - hs_ref) <= 3e-5 * np.abs(hs_ref)), "h block scales"
    step = np.abs(_e4m3_order(hq) - _e4m3_order(hq_ref))
    assert step.max() <= 1, f"h codes off by {step.max()} steps"
    assert (step > 0).mean() <= 2e-3, f"{(step > 0).mean():.2e} of h codes on the other side"
    dq = oracle.e4m3_decode_table()
    h_got = dq[hq].astype(np.float64) * np.repeat(hs.T, 128, axis=1)
    h_ref = dq[hq_ref].astype(np.float64) * np.repeat(hs_ref.T, 128, axis=1)
    assert_close(torch.from_numpy(h_got), h_ref, f"fp8 swiglu bm={bm}")


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_gemm_fp8_swiglu_epilogue(bm):
    _fp8_swiglu_case(M=300, K=512, I=384, E=16, k=4, bm=bm)


@pytest.mark.parametrize("sched,ctas", [(L.SCHED_STATIC, 0), (L.SCHED_QUEUE, 6)])
def test_gemm_fp8_swiglu_schedules(sched, ctas):
    """Static partition, and six CTAs looping over many tiles (at 128 routed
    rows both run CTA pairs, which walk a fixed round-robin order)."""
    _fp8_swiglu_case(M=900, K=1024, I=256, E=6, k=2, bm=128, sched=sched, num_ctas=ctas, skew=2.0)


@pytest.mark.parametrize("M,E,k,I,ctas,skew", [
    (1500, 4, 2, 512, 4, 1.0),    # two pairs loop over many 256-row tiles
    (200, 16, 3, 256, 0, 2.0),    # experts of 1..255 rows: half-empty and odd-CTA-empty tiles
    (700, 8, 3, 256, 5, 1.5),     # an odd grid: two pairs
    (700, 8, 3, 256, 1, 1.5),     # one CTA: the single-CTA token-major tile
])
def test_gemm_fp8_swiglu_cta_pairs(M, E, k, I, ctas, skew):
    """FP8 SWIGLU at 128 routed rows: a cluster of two CTAs computes tiles of
    256 routed rows (128 per CTA, the M = 256 side of each MMA) against the gate
    rows (even CTA) and up rows (odd CTA) of 128 h columns; each CTA applies
    the SwiGLU and the 1x128 re-quantisation to its own rows.  Tile offsets of
    the 256-row tiles come from the row offsets inside the kernel."""
    assert L.gemm_cta_pairs() > 0, "the CTA-pair form is not in use on this device"
    _fp8_swiglu_case(M=M, K=1024, I=I, E=E, k=k, bm=128, num_ctas=ctas, skew=skew)


def _bf16_gemm_case(R_tokens, K, N, E, k, bm, epilogue, sched=L.SCHED_QUEUE, seed=0, num_ctas=0,
                    cta_pairs=0):
    g = torch.Generator().manual_seed(seed)
    M = R_tokens
    logits = torch.randn(M, E, generator=g)
    rid, rw = oracle.route(logits.numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    a = x[torch.from_numpy(lay["sorted_route_ids"] // k).long()]  # expert-compact rows
    Y = oracle.grouped_gemm_bf16(bits(a), bits(w), lay["offsets"], threads=THREADS)
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    ws = L.new_workspace(L.CTRL_BYTES)
    if epilogue == L.EPI_SWIGLU:
        out = torch.zeros(M * k, N // 2, dtype=torch.bfloat16, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_BF16, epilogue=epilogue, a=a.cuda(), w=w.cuda(),
                       offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), out=out,
                       ws=ws, block_m=bm, sched=sched, num_ctas=num_ctas,
                       cta_pairs=cta_pairs)
        torch.cuda.synchronize()
        gate, up = Y[:, :N // 2], Y[:, N // 2:]
        ref = gate / (1.0 + np.exp(-gate)) * up
        assert_close(out, ref, "bf16 swiglu")
    elif epilogue == L.EPI_SCATTER:
        out = torch.zeros(M, N, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_BF16, epilogue=epilogue, a=a.cuda(), w=w.cuda(),
                       offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), out=out,
                       ws=ws, block_m=bm, sorted_route_ids=cu(lay["sorted_route_ids"]),
                       route_weights=cu(rw), M=M, top_k=k, sched=sched, num_ctas=num_ctas,
                       cta_pairs=cta_pairs)
        torch.cuda.synchronize()
        assert_close(out, oracle.scatter(Y, lay["route_slot"], rw), "bf16 scatter")
    else:
        dt = torch.bfloat16 if epilogue == L.EPI_STORE_BF16 else torch.float32
        out = torch.zeros(M * k, N, dtype=dt, device="cuda")
        L.grouped_gemm(dtype=L.DTYPE_BF16, epilogue=epilogue, a=a.cuda(), w=w.cuda(),
                       offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), out=out,
                       ws=ws, block_m=bm, sched=sched, num_ctas=num_ctas,
                       cta_pairs=cta_pairs)
        torch.cuda.synchronize()
        assert_close(out, Y, "bf16 store")
    assert L.get_error(ws) == L.MOE_OK


@pytest.mark.parametrize("R,K,N,E,k,epi,ctas", [
    (1200, 1024, 1024, 4, 2, L.EPI_SCATTER, 4),      # two pairs loop over many tiles
    (1200, 1024, 1024, 4, 2, L.EPI_STORE_BF16, 5),   # an odd grid: two pairs
    (90, 640, 512, 16, 3, L.EPI_SCATTER, 0),         # tiles of 1..127 rows: the odd CTA's half empty
    (600, 512, 512, 8, 2, L.EPI_STORE_BF16, 1),      # one CTA: the single-CTA 256-row tile
    (1200, 1024, 1024, 4, 2, L.EPI_SWIGLU, 4),       # SwiGLU: two pairs, many tiles
    (90, 640, 512, 16, 3, L.EPI_SWIGLU, 0),          # SwiGLU: the odd CTA's 128 rows empty
    (700, 512, 512, 8, 3, L.EPI_SWIGLU, 3),          # SwiGLU: an odd grid
    (600, 512, 512, 8, 2, L.EPI_SWIGLU, 1),          # SwiGLU: one CTA
])
def test_gemm_bf16_cta_pairs(R, K, N, E, k, epi, ctas):
    """BF16 at block_m 256 on CTA pairs, each CTA's accumulator double-buffered
    in TMEM.  Scatter / bf16-rows store (N a multiple of 256): each 256 x 256
    tile has M = 256 weight rows and N = 256 routed rows, 128 of each staged per
    CTA.  SwiGLU: token-major, M = 256 routed rows (128 per CTA) and N = the
    gate rows (even CTA) and up rows (odd CTA) of 128 h columns."""
    assert L.gemm_cta_pairs() > 0, "the CTA-pair form is not in use on this device"
    _bf16_gemm_case(R_tokens=R, K=K, N=N, E=E, k=k, bm=256, epilogue=epi, num_ctas=ctas)


@pytest.mark.parametrize("bm", [16, 64, 128, 256])
@pytest.mark.parametrize("epi", [L.EPI_STORE, L.EPI_SWIGLU, L.EPI_SCATTER, L.EPI_STORE_BF16])
def test_gemm_bf16(bm, epi):
    _bf16_gemm_case(R_tokens=200, K=320, N=256, E=8, k=2, bm=bm, epilogue=epi)


@pytest.mark.parametrize("bm", [64, 256])
def test_gemm_bf16_static_schedule(bm):
    """Static per-expert partition; block_m 256 with N % 256 == 0 runs wide tiles."""
    _bf16_gemm_case(R_tokens=300, K=256, N=512, E=3, k=2, bm=bm, epilogue=L.EPI_SCATTER,
                    sched=L.SCHED_STATIC)


@pytest.mark.parametrize("bm", [128, 256])
@pytest.mark.parametrize("epi", [L.EPI_SCATTER, L.EPI_STORE_BF16])
def test_gemm_bf16_narrow_tiles_when_n_is_odd_multiple_of_128(bm, epi):
    """N = 384 is not a multiple of 256: one weight tile per tile (no wide tiles)."""
    _bf16_gemm_case(R_tokens=180, K=192, N=384, E=4, k=2, bm=bm, epilogue=epi)


def _gather_gemm_fp8_case(M, K, N, E, k, bm, epilogue, sched=L.SCHED_QUEUE, k_splits=0, seed=0,
                          skew=0.0, num_ctas=0):
    """gather_rows=1: the GEMM reads each routed row from the token-major
    codes (row sorted_route_ids[s] // k) and its scales from [K/128, M]."""
    d = inputs.make_fp8_inputs(dict(M=M, K=K, N=N, E=E, k=k, softcap=0.0, zipf_bias=skew),
                               seed=seed)
    rid, rw = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])       # compact (reference)
    a_tok, s_tok = oracle.quant_gather(bits(d["x"]), 1, np.arange(M, dtype=np.int32))  # token-major
    Y = oracle.grouped_gemm_fp8(a_q, a_s, d["w_q"].numpy(), d["w_scales"].numpy(),
                                lay["offsets"], threads=THREADS)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = L.new_workspace(L.CTRL_BYTES)
    common = dict(dtype=L.DTYPE_FP8, a=cu(a_tok), a_scales=cu(s_tok), w=d["w_q"].cuda(),
                  w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                  tile_offsets=cu(lay["tile_offsets"]), ws=ws, block_m=bm, sched=sched,
                  num_ctas=num_ctas, sorted_route_ids=cu(lay["sorted_route_ids"]), M=M, top_k=k,
                  gather_rows=1)
    if epilogue == L.EPI_SCATTER:
        out = torch.zeros(M, N, device="cuda")
        L.grouped_gemm(epilogue=epilogue, out=out, route_weights=cu(rw), k_splits=k_splits,
                       **common)
        ref = oracle.scatter(Y, lay["route_slot"], rw)
    else:
        out = torch.zeros(M * k, N, device="cuda")
        L.grouped_gemm(epilogue=epilogue, out=out, **common)
        ref = Y
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    assert_close(out, ref, "fp8 gathered rows")


@pytest.mark.parametrize("bm,epi,sched,ks", [
    (16, L.EPI_SCATTER, L.SCHED_QUEUE, 1), (64, L.EPI_SCATTER, L.SCHED_STATIC, 1),
    (128, L.EPI_SCATTER, L.SCHED_QUEUE, 0), (32, L.EPI_SCATTER, L.SCHED_QUEUE, 4),
    (128, L.EPI_STORE, L.SCHED_QUEUE, 1), (64, L.EPI_STORE, L.SCHED_STATIC, 1)])
def test_gemm_fp8_gathered_rows(bm, epi, sched, ks):
    """Ragged tails, empty experts (skewed loads), K splits and both schedulers."""
    _gather_gemm_fp8_case(M=300, K=1024, N=384, E=16, k=4, bm=bm, epilogue=epi, sched=sched,
                          k_splits=ks, skew=1.5)


def test_gemm_fp8_gathered_rows_few_ctas():
    """Eight CTAs loop over many tiles: the route-id ring wraps many times."""
    _gather_gemm_fp8_case(M=700, K=2048, N=512, E=4, k=2, bm=128, epilogue=L.EPI_SCATTER,
                          num_ctas=8)


@pytest.mark.parametrize("bm,epi", [(16, L.EPI_SWIGLU), (64, L.EPI_SWIGLU), (256, L.EPI_SWIGLU),
                                    (128, L.EPI_SCATTER)])
def test_gemm_bf16_gathered_rows(bm, epi):
    """The gated up projection gathers x's rows; other BF16 epilogues do not
    gather (MOE_ERR_UNSUPPORTED)."""
    g = torch.Generator().manual_seed(3)
    M, K, N, E, k = 230, 320, 256, 8, 2
    rid, rw = oracle.route(torch.randn(M, E, generator=g).numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    A = x[torch.from_numpy(lay["sorted_route_ids"] // k).long()].double().numpy()
    W = w.double().numpy()
    Y = np.zeros((M * k, N))
    for e in range(E):
        s0, s1 = lay["offsets"][e], lay["offsets"][e + 1]
        Y[s0:s1] = A[s0:s1] @ W[e].T
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    ws = L.new_workspace(L.CTRL_BYTES)
    common = dict(dtype=L.DTYPE_BF16, epilogue=epi, a=x.cuda(), w=w.cuda(),
                  offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), ws=ws,
                  block_m=bm, sorted_route_ids=cu(lay["sorted_route_ids"]), M=M, top_k=k,
                  gather_rows=1)
    if epi == L.EPI_SWIGLU:
        out = torch.zeros(M * k, N // 2, dtype=torch.bfloat16, device="cuda")
        L.grouped_gemm(out=out, **common)
        gate, up = Y[:, :N // 2], Y[:, N // 2:]
        ref = gate / (1.0 + np.exp(-gate)) * up
    else:
        out = torch.zeros(M, N, device="cuda")
        with pytest.raises(L.MoeError) as err:
            L.grouped_gemm(out=out, route_weights=cu(rw), **common)
        assert err.value.code == L.MOE_ERR_UNSUPPORTED
        return
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    assert_close(out, ref, "bf16 gathered rows")


# ------------------------------------------------------------------ fused forward
@pytest.mark.parametrize("softcap", [0.0, 30.0])
@pytest.mark.parametrize("use_graph", [0, 1])
def test_forward_tiny_fp8(softcap, use_graph):
    d = inputs.make_fp8_inputs("tiny_fp8", seed=0)
    dev = fp8_device_inputs(d)
    out, _, _ = run_forward_fp8(dev, d["cfg"], softcap=softcap, use_graph=use_graph)
    r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=2, softcap=softcap)
    assert_close(out, r["out"], "tiny")


def test_forward_medium_fp8_all_rows():
    cfg = dict(M=300, K=1024, N=384, E=32, k=4, softcap=30.0, zipf_bias=1.0)
    d = inputs.make_fp8_inputs(cfg, seed=4)
    dev = fp8_device_inputs(d)
    for bm in (16, 64):
        out, _, _ = run_forward_fp8(dev, d["cfg"], block_m=bm)
        r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                               d["w_scales"].numpy(), k=4, softcap=30.0, threads=THREADS)
        assert_close(out, r["out"], f"medium bm={bm}")


def test_forward_qwen_small_batch_fp8_full():
    """The 128-token / 256-expert workload at full size, every output row."""
    d = inputs.make_fp8_inputs("qwen_small_batch_fp8", seed=0)
    dev = fp8_device_inputs(d)
    out, _, _ = run_forward_fp8(dev, d["cfg"])
    r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=8, softcap=30.0, threads=THREADS)
    assert_close(out, r["out"], "qwen")
    # the same call replayed from the graph cache gives the same bits
    out2, _, _ = run_forward_fp8(dev, d["cfg"])
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) or \
        (out.float() - out2.float()).abs().max().item() <= 1e-2 * out.float().abs().max().item()


def test_forward_skewed_large_batch_fp8_load_skew():
    """The skewed workload's expert loads differ by more than 10x (its every
    output row and every intermediate are checked in test_gpu_forward_steps)."""
    d = inputs.make_fp8_inputs("skewed_large_batch_fp8", seed=0)
    ids, _ = oracle.route(d["logits"].numpy(), 8, softcap=30.0)
    counts = np.bincount(ids.reshape(-1), minlength=256)
    assert counts.max() >= 10 * max(1, counts[counts > 0].min())


def test_forward_fp8_bf16_rows_path_sampled():
    """An FP8 forward whose fp32 output accumulator (8192 x 4096 x 4 B) is too
    large to keep on chip: the GEMM stores bf16 rows and a reduction kernel
    applies the route weights."""
    cfg = dict(M=8192, K=256, N=4096, E=8, k=2, softcap=30.0, zipf_bias=0.5)
    d = inputs.make_fp8_inputs(cfg, seed=5)
    dev = fp8_device_inputs(d)
    out, _, _ = run_forward_fp8(dev, d["cfg"])
    tok = sample_tokens(cfg["M"], 1024)
    r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=2, softcap=30.0, tokens=tok, threads=THREADS)
    assert_close(out[torch.from_numpy(tok).long().cuda()], r["out"], "fp8 bf16-rows path")


def _bf16_forward_case(cfg_name, routing, rho=1.0, n_tok=1024, variants=None, overrides=None):
    """One BF16 gated-FFN workload through moe_forward under each of
    ``variants`` (dicts of block_m / sched / gather_rows), checked against one
    oracle evaluation of ``n_tok`` seeded tokens (all tokens when n_tok >= T)."""
    d = inputs.make_bf16_inputs(cfg_name, routing=routing, rho=rho, seed=0, **(overrides or {}))
    dev = dict(logits=d["logits"].cuda(), x=d["x"].cuda(), w_up=d["w_up"].cuda(),
               w_dn=d["w_dn"].cuda())
    k = d["cfg"]["k"]
    ids, w = oracle.route(d["logits"].numpy(), k)
    assert np.array_equal(np.sort(ids, axis=1), np.sort(d["chosen"].numpy(), axis=1))
    tok = sample_tokens(d["cfg"]["T"], n_tok)
    ref = oracle.ffn_bf16(bits(d["x"]), ids, w, bits(d["w_up"]), bits(d["w_dn"]), tokens=tok,
                          threads=THREADS)
    sel = torch.from_numpy(tok).long().cuda()
    for v in (variants or [{}]):
        out, _, _ = run_forward_bf16(dev, d["cfg"], **v)
        assert_close(out[sel], ref, f"{cfg_name}/{routing}/rho={rho:g} {v}")


def test_forward_bf16_small_all_rows():
    _bf16_forward_case("bf16_ffn", "uniform", n_tok=10**9,
                       overrides=dict(T=200, H=256, I=256, E=8, k=3))


@pytest.mark.parametrize("bm", [64, 256])
def test_forward_bf16_gathered_rows_all_rows(bm):
    """gather_rows=1: the up projection reads x's rows by route id (no copy)."""
    _bf16_forward_case("bf16_ffn", "uniform", n_tok=10**9,
                       variants=[dict(block_m=bm, gather_rows=1)],
                       overrides=dict(T=300, H=256, I=256, E=8, k=3))


@pytest.mark.parametrize("bm", [64, 128])
def test_forward_fp8_gathered_rows_all_rows(bm):
    """gather_rows=1 on the large-batch FP8 path (more than 4096 routes): codes
    and scales token-major, rows gathered in the GEMM; every output row."""
    cfg = dict(M=1100, K=1024, N=384, E=32, k=4, softcap=30.0, zipf_bias=1.0)
    d = inputs.make_fp8_inputs(cfg, seed=5)
    dev = fp8_device_inputs(d)
    out, args, _ = run_forward_fp8(dev, d["cfg"], block_m=bm, gather_rows=1)
    assert L.workspace_size(args) < L.workspace_size(L.forward_args(
        dtype=L.DTYPE_FP8, M=1100, K=1024, N=384, E=32, top_k=4, w=dev["w_q"],
        w_scales=dev["w_scales"], gather_rows=0))
    r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=4, softcap=30.0, threads=THREADS)
    assert_close(out, r["out"], f"fp8 gathered rows bm={bm}")


@pytest.mark.parametrize("routing", ["balanced", "uniform", "zipf1.2"])
def test_forward_bf16_ffn_full(routing):
    """The 8192-token gated FFN, 1024 seeded tokens checked, under the
    forward's own tile choice."""
    _bf16_forward_case("bf16_ffn", routing, n_tok=1024)


@pytest.mark.parametrize("rho", [1.0, 4.0, 16.0, 40.0])
def test_forward_imbalance_bf16(rho):
    """The 16384-token load-imbalance sweep, 1024 seeded tokens checked, under
    the atomic queue and the static partition at several tile heights."""
    _bf16_forward_case("imbalance_bf16", "loads", rho=rho, n_tok=1024,
                       variants=[dict(block_m=128, sched=L.SCHED_QUEUE),
                                 dict(block_m=64, sched=L.SCHED_STATIC),
                                 dict(block_m=256, sched=L.SCHED_QUEUE),
                                 dict(block_m=256, sched=L.SCHED_STATIC)])


def test_forward_host_matches_device():
    d = inputs.make_fp8_inputs("tiny_fp8", seed=2)
    dev = fp8_device_inputs(d)
    out, args, ws = run_forward_fp8(dev, d["cfg"])
    h_logits = d["logits"].pin_memory()
    h_x = d["x"].pin_memory()
    h_out = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    L.forward_host(args, h_logits, h_x, h_out, ws)
    torch.cuda.synchronize()
    assert torch.equal(h_out.view(torch.int16), out.cpu().view(torch.int16)) or \
        (h_out.float() - out.cpu().float()).abs().max() <= 1e-2 * out.float().abs().max().item()


@pytest.mark.parametrize("name", ["tiny_fp8", "qwen_small_batch_fp8"])
def test_forward_host_pinned_and_pageable(name):
    """Pinned host buffers are read and written by the kernels directly,
    pageable ones go through the staging copies; both match the device path."""
    d = inputs.make_fp8_inputs(name, seed=3)
    dev = fp8_device_inputs(d)
    out, args, ws = run_forward_fp8(dev, d["cfg"])
    ref = out.cpu()
    for pinned in (True, False):
        h_logits = d["logits"].contiguous()
        h_x = d["x"].contiguous()
        h_out = torch.empty(out.shape, dtype=torch.bfloat16)
        if pinned:
            h_logits, h_x, h_out = h_logits.pin_memory(), h_x.pin_memory(), h_out.pin_memory()
        for _ in range(2):  # the second call replays the cached graph
            h_out.zero_()
            L.forward_host(args, h_logits, h_x, h_out, ws)
            torch.cuda.synchronize()
            assert L.get_error(ws) == L.MOE_OK
            diff = (h_out.float() - ref.float()).abs().max().item()
            assert diff <= 1e-2 * ref.float().abs().max().item(), (pinned, diff)


def test_scatter_standalone():
    g = torch.Generator().manual_seed(3)
    M, N, k = 70, 384, 3
    rows = torch.randn(M * k, N, generator=g)
    w = torch.rand(M, k, generator=g)
    slot = torch.randperm(M * k, generator=g).to(torch.int32)
    ws = L.new_workspace(L.CTRL_BYTES)
    out = L.scatter(rows.cuda(), slot.cuda(), w.cuda(), ws)
    ref = oracle.scatter(rows.double().numpy(), slot.numpy(), w.numpy())
    assert_close(out, ref, "scatter")
    assert L.get_error(ws) == L.MOE_OK


def test_scatter_reports_bad_slots():
    """A route whose slot is outside [0, M*top_k) adds nothing and records
    MOE_ERR_DEVICE_FAULT; reading the status clears it."""
    g = torch.Generator().manual_seed(4)
    M, N, k = 9, 256, 2
    rows = torch.randn(M * k, N, generator=g)
    w = torch.rand(M, k, generator=g)
    slot = torch.randperm(M * k, generator=g).to(torch.int32)
    ws = L.new_workspace(L.CTRL_BYTES)
    bad = slot.clone()
    bad[5] = M * k                       # token 2, route 1
    bad[8] = -3                          # token 4, route 0
    out = L.scatter(rows.cuda(), bad.cuda(), w.cuda(), ws)
    assert L.get_error(ws) == L.MOE_ERR_DEVICE_FAULT
    w0 = w.clone()
    w0[2, 1] = 0.0
    w0[4, 0] = 0.0
    ref = oracle.scatter(rows.double().numpy(), slot.numpy(), w0.numpy())
    assert_close(out, ref, "scatter without the bad routes")
    assert L.get_error(ws) == L.MOE_OK


# ------------------------------------------------------------------ failure detection
def test_pipeline_timeout_reports_status_and_recovers():
    """A producer that issues nothing: every consumer wait runs into its time
    limit, the kernel exits with MOE_ERR_TIMEOUT, and the next call works."""
    d = inputs.make_fp8_inputs("tiny_fp8", seed=0)
    dev = fp8_device_inputs(d)
    try:
        L.debug_set_pipeline_fault(True, 20_000_000)   # 20 ms
        args = L.forward_args(dtype=L.DTYPE_FP8, M=16, K=256, N=128, E=8, top_k=2,
                              logits=dev["logits"], x=dev["x"], w=dev["w_q"],
                              w_scales=dev["w_scales"], use_graph=0)
        ws = L.new_workspace(L.workspace_size(args))
        out = torch.empty(16, 128, dtype=torch.bfloat16, device="cuda")
        L.forward(args, out, ws)
        assert L.get_error(ws) == L.MOE_ERR_TIMEOUT
    finally:
        L.debug_set_pipeline_fault(False, 0)
    out, _, _ = run_forward_fp8(dev, d["cfg"], use_graph=0)
    r = oracle.forward_fp8(d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=2)
    assert_close(out, r["out"], "after timeout")


@pytest.mark.parametrize("form", ["fp8_scatter", "fp8_swiglu", "bf16_scatter"])
def test_cta_pair_timeout_reports_status_and_recovers(form):
    """The same fault on the CTA-pair kernels: neither CTA of a pair receives
    any copy, the even CTA's MMA thread and both CTAs' other roles run into
    their time limits, both CTAs still meet at the closing cluster barrier,
    the launch ends with MOE_ERR_TIMEOUT, and the next call is correct."""
    assert L.gemm_cta_pairs() > 0, "the CTA-pair form is not in use on this device"
    M, k, E, K = 256, 2, 4, 256
    ids = np.stack([np.arange(M) % E, (np.arange(M) + 1) % E], axis=1).astype(np.int32)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    fp8 = form != "bf16_scatter"
    bm = 128 if fp8 else 256
    lay = oracle.layout(ids, E, block_m=bm)
    R = M * k
    ws = L.new_workspace(L.CTRL_BYTES)
    common = dict(offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), ws=ws,
                  block_m=bm, M=M, top_k=k)
    try:
        L.debug_set_pipeline_fault(True, 20_000_000)   # 20 ms
        if form == "fp8_scatter":
            L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER,
                           a=torch.zeros(R, K, dtype=torch.uint8, device="cuda"),
                           a_scales=torch.zeros(K // 128, R, device="cuda"),
                           w=torch.zeros(E, 512, K, dtype=torch.uint8, device="cuda"),
                           w_scales=torch.zeros(E, 4, K // 128, device="cuda"),
                           out=torch.zeros(M, 512, device="cuda"),
                           sorted_route_ids=cu(lay["sorted_route_ids"]),
                           route_weights=torch.ones(M, k, device="cuda"), **common)
        elif form == "fp8_swiglu":
            L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SWIGLU,
                           a=torch.zeros(R, K, dtype=torch.uint8, device="cuda"),
                           a_scales=torch.zeros(K // 128, R, device="cuda"),
                           w=torch.zeros(E, 512, K, dtype=torch.uint8, device="cuda"),
                           w_scales=torch.zeros(E, 4, K // 128, device="cuda"),
                           out=torch.zeros(R, 256, dtype=torch.uint8, device="cuda"),
                           out_scales=torch.zeros(2, R, device="cuda"), **common)
        else:
            L.grouped_gemm(dtype=L.DTYPE_BF16, epilogue=L.EPI_SCATTER,
                           a=torch.zeros(R, K, dtype=torch.bfloat16, device="cuda"),
                           w=torch.zeros(E, 512, K, dtype=torch.bfloat16, device="cuda"),
                           out=torch.zeros(M, 512, device="cuda"),
                           sorted_route_ids=cu(lay["sorted_route_ids"]),
                           route_weights=torch.ones(M, k, device="cuda"), **common)
        torch.cuda.synchronize()
        assert L.get_error(ws) == L.MOE_ERR_TIMEOUT
    finally:
        L.debug_set_pipeline_fault(False, 0)
    if form == "fp8_scatter":
        _fp8_gemm_case(M=700, K=1024, N=512, E=8, k=3, bm=128, epilogue=L.EPI_SCATTER, skew=1.5)
    elif form == "fp8_swiglu":
        _fp8_swiglu_case(M=700, K=1024, I=256, E=8, k=3, bm=128, skew=1.5)
    else:
        _bf16_gemm_case(R_tokens=600, K=512, N=512, E=8, k=2, bm=256, epilogue=L.EPI_SCATTER)
