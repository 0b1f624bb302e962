"""Bit-exact GPU parity of the fused forward's OWN intermediate steps.

moe_forward does not call the standalone step kernels: small FP8 batches
route and then quantise + lay out in one kernel; large batches rank routes per
CTA while routing and place them while quantising (or, with gathered rows,
write each token's codes once); the BF16 forward places routes while copying
rows.  moe_forward_workspace_map says where each of those steps leaves its
result in the workspace, and this file compares every one of them with the
oracle bit for bit after a real forward:

* route ("Fused MoE FP8", section "Baseline: 7 kernels", item 1): expert ids
  and the route weights' bits;
* count + layout (items 2-3, section "Fusion 3"): counts, offsets, tile
  offsets at the forward's block_m, the stable permutation and its inverse;
* quantise + gather (items 4-5): E4M3 codes and the scales' bits, expert-
  compact or token-major; the BF16 path's copied rows;
* the FP8 gated FFN's re-quantised h, against the oracle's binary64 up
  projection rounded to binary32: the same code except where the device's
  fp32 accumulation puts h on the other side of an E4M3 rounding boundary
  (then the neighbouring code), block scales within fp32 accumulation error.

The outputs of the same forwards are compared with the oracle's binary64
result on every row (FP8 workloads) or on 1024 seeded tokens (the gated FFNs)
within rel-L2 5e-3 and max-abs 1e-2 max|ref|."""
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


def _view(ws, m, name, dtype, shape) -> np.ndarray:
    assert m[name] is not None, name
    return np_(L.ws_view(ws, m[name], dtype, shape))


def _eq(got: np.ndarray, ref: np.ndarray, what: str):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = np.flatnonzero(got.reshape(-1) != ref.reshape(-1))
    assert bad.size == 0, f"{what}: {bad.size} of {got.size} differ, first at {bad[:5]}"


def _f32_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _check_route_layout(ws, m, M, E, k, ref):
    """ref: dict with ids, weights, counts, offsets, tile_offsets,
    sorted_route_ids, route_slot (the oracle's)."""
    R = M * k
    _eq(_view(ws, m, "ids", torch.int32, (M, k)), ref["ids"], "ids")
    _eq(_f32_bits(_view(ws, m, "weights", torch.float32, (M, k))), _f32_bits(ref["weights"]),
        "route weights (bits)")
    _eq(_view(ws, m, "counts", torch.int32, (E,)), ref["counts"], "counts")
    _eq(_view(ws, m, "offsets", torch.int32, (E + 1,)), ref["offsets"], "offsets")
    _eq(_view(ws, m, "tile_offsets", torch.int32, (E + 1,)), ref["tile_offsets"], "tile offsets")
    _eq(_view(ws, m, "sorted_route_ids", torch.int32, (R,)), ref["sorted_route_ids"],
        "sorted route ids")
    _eq(_view(ws, m, "route_slot", torch.int32, (R,)), ref["route_slot"], "route slot")


_ORACLE_CACHE = {}


def _oracle_fp8(name, d, cfg, bm):
    key = (name, bm)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.forward_fp8(
            d["logits"].numpy(), bits(d["x"]), d["w_q"].numpy(), d["w_scales"].numpy(),
            k=cfg["k"], softcap=cfg["softcap"], block_m=bm, threads=THREADS)
    return _ORACLE_CACHE[key]


FP8_CASES = {
    # (workload or shape, forward options): the path each one takes
    "qwen_small": ("qwen_small_batch_fp8", {}),                       # fused quantise + layout
    "skewed_large": ("skewed_large_batch_fp8", {}),                   # route + rank, placement
    "skewed_large_gathered": ("skewed_large_batch_fp8", dict(gather_rows=1)),  # token-major
    "edge_4096_routes": (dict(M=512, K=512, N=256, E=64, k=8, softcap=30.0, zipf_bias=1.0), {}),
    "edge_4104_routes": (dict(M=513, K=512, N=256, E=64, k=8, softcap=30.0, zipf_bias=1.0), {}),
    "tiny": ("tiny_fp8", {}),
    # top_k above K/16 (more routes per token than the quantiser has threads)
    "many_experts": (dict(M=300, K=256, N=128, E=1024, k=32, softcap=0.0, zipf_bias=0.0), {}),
    "many_experts_gathered": (dict(M=300, K=256, N=128, E=1024, k=32, softcap=0.0,
                                   zipf_bias=0.0), dict(gather_rows=1)),
    "large_bm64_static": (dict(M=1500, K=1024, N=384, E=48, k=6, softcap=30.0, zipf_bias=2.0),
                          dict(block_m=64, sched=L.SCHED_STATIC)),
}


@pytest.mark.parametrize("case", list(FP8_CASES))
def test_fp8_forward_steps_bit_exact(case):
    name_or_cfg, opts = FP8_CASES[case]
    d = inputs.make_fp8_inputs(name_or_cfg, seed=0)
    cfg = d["cfg"]
    M, K, E, k = cfg["M"], cfg["K"], cfg["E"], cfg["k"]
    R = M * k
    out, args, ws = run_forward_fp8(fp8_device_inputs(d), cfg, **opts)
    m = L.workspace_map(args)
    key = name_or_cfg if isinstance(name_or_cfg, str) else case
    r = _oracle_fp8(key, d, cfg, m["block_m"])
    _check_route_layout(ws, m, M, E, k, r)
    if m["a_rows"] == R:
        _eq(_view(ws, m, "a", torch.uint8, (R, K)), r["a_q"], "compact E4M3 codes")
        _eq(_f32_bits(_view(ws, m, "a_scales", torch.float32, (K // 128, R))),
            _f32_bits(r["a_scales"]), "compact scales (bits)")
    else:
        # gathered rows: each token's codes once, token-major
        assert m["a_rows"] == M and opts.get("gather_rows") == 1
        tq, ts = oracle.quant_gather(bits(d["x"]), 1, np.arange(M, dtype=np.int32))
        _eq(_view(ws, m, "a", torch.uint8, (M, K)), tq, "token-major E4M3 codes")
        _eq(_f32_bits(_view(ws, m, "a_scales", torch.float32, (K // 128, M))), _f32_bits(ts),
            "token-major scales (bits)")
    assert_close(out, r["out"], f"{case}: every output row")


BF16_CASES = {
    "ffn_uniform": ("bf16_ffn", "uniform", 1.0, {}),
    "imbalance_rho40_static": ("imbalance_bf16", "loads", 40.0,
                               dict(block_m=64, sched=L.SCHED_STATIC)),
    "ffn_zipf_gathered": ("bf16_ffn", "zipf1.2", 1.0, dict(gather_rows=1)),
}


@pytest.mark.parametrize("case", list(BF16_CASES))
def test_bf16_forward_steps_bit_exact(case):
    name, routing, rho, opts = BF16_CASES[case]
    d = inputs.make_bf16_inputs(name, routing=routing, rho=rho, seed=0)
    cfg = d["cfg"]
    T, H, E, k = cfg["T"], cfg["H"], cfg["E"], cfg["k"]
    R = T * k
    dev = dict(logits=d["logits"].cuda(), x=d["x"].cuda(), w_up=d["w_up"].cuda(),
               w_dn=d["w_dn"].cuda())
    out, args, ws = run_forward_bf16(dev, cfg, **opts)
    m = L.workspace_map(args)
    ids, w = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(ids, E, block_m=m["block_m"])
    _check_route_layout(ws, m, T, E, k, dict(ids=ids, weights=w, **lay))
    if opts.get("gather_rows") == 1:
        assert m["a"] is None                      # the up projection reads x's rows itself
    else:
        xb = bits(d["x"])
        rows = _view(ws, m, "a", torch.int16, (R, H)).view(np.uint16)
        _eq(rows, xb[lay["sorted_route_ids"] // k], "expert-compact bf16 rows")
    tok = sample_tokens(T, 1024)
    ref = oracle.ffn_bf16(bits(d["x"]), ids, w, bits(d["w_up"]), bits(d["w_dn"]), tokens=tok,
                          threads=THREADS)
    assert_close(out[torch.from_numpy(tok).long().cuda()], ref, f"{case}: 1024 tokens")


def _e4m3_order(c: np.ndarray) -> np.ndarray:
    """Signed position of an E4M3 code on the number line (codes of equal
    sign are ordered by their low 7 bits); 0x00 and 0x80 both map to 0."""
    c = c.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


FFN_FP8_CASES = {
    "small_batch": (dict(T=200, H=256, I=256, E=8, k=3), "uniform", {}),
    "large_batch": (dict(T=1500, H=512, I=384, E=16, k=4), "zipf1.2", dict(block_m=64)),
    "large_bm128": (dict(T=1500, H=512, I=384, E=16, k=4), "zipf1.2", dict(block_m=128)),
    "gather_flag_ignored": (dict(T=1500, H=512, I=384, E=16, k=4), "uniform",
                            dict(gather_rows=1)),
}


@pytest.mark.parametrize("case", list(FFN_FP8_CASES))
def test_ffn_fp8_forward_steps(case):
    """The FP8 gated FFN's route, layout and first quantisation bit-exact;
    its re-quantised h against the oracle's pipeline (binary64 up projection
    of the same codes, rounded to binary32, then the SwiGLU + 1x128 rule)."""
    shape, routing, opts = FFN_FP8_CASES[case]
    d = inputs.make_fp8_ffn_inputs("ffn_fp8", routing=routing, seed=4, **shape)
    c = d["cfg"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    R = T * k
    dev = {n: d[n].cuda() for n in ("logits", "x", "wup_q", "wup_s", "wdn_q", "wdn_s")}
    args = L.forward_args(dtype=L.DTYPE_FP8, gated=1, M=T, K=H, N=I, E=E, top_k=k, softcap=0.0,
                          logits=dev["logits"], x=dev["x"], w=dev["wup_q"], w_scales=dev["wup_s"],
                          w2=dev["wdn_q"], w2_scales=dev["wdn_s"], use_graph=1, **opts)
    ws = L.new_workspace(L.workspace_size(args))
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    L.forward(args, out, ws)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    m = L.workspace_map(args)
    ids, w = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(ids, E, block_m=m["block_m"])
    _check_route_layout(ws, m, T, E, k, dict(ids=ids, weights=w, **lay))
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])
    # the fused SwiGLU up projection reads the expert-compact copy (gathered
    # rows are not used by the FP8 gated FFN)
    assert m["a_rows"] == R
    _eq(_view(ws, m, "a", torch.uint8, (R, H)), a_q, "compact E4M3 codes")
    _eq(_f32_bits(_view(ws, m, "a_scales", torch.float32, (H // 128, R))), _f32_bits(a_s),
        "compact scales (bits)")
    # h: the oracle's up projection of the same codes (binary64, then binary32)
    gu = oracle.grouped_gemm_fp8(a_q, a_s, d["wup_q"].numpy(), d["wup_s"].numpy(),
                                 lay["offsets"], threads=THREADS).astype(np.float32)
    hq_ref, hs_ref = oracle.swiglu_quant(gu)
    hq = _view(ws, m, "h_q", torch.uint8, (R, I))
    hs = _view(ws, m, "h_scales", torch.float32, (I // 128, R))
    assert np.all(np.abs(hs - hs_ref) <= 3e-5 * np.abs(hs_ref)), "h block scales"
    step = np.abs(_e4m3_order(hq) - _e4m3_order(hq_ref))
    assert step.max() <= 1, f"h codes off by {step.max()} steps"
    assert (step > 0).mean() <= 2e-3, f"{(step > 0).mean():.2e} of h codes on the other side"
    ref = oracle.ffn_fp8(bits(d["x"]), ids, w, d["wup_q"].numpy(), d["wup_s"].numpy(),
                         d["wdn_q"].numpy(), d["wdn_s"].numpy(), threads=THREADS)
    assert_close(out, ref, f"ffn fp8 {case}: every output row")
