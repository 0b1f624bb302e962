"""moe_grouped_gemm_noalloc — the grouped GEMM for callers that cannot
allocate device memory (no workspace argument; the kernel's 256-byte control
block lives in a static array inside the library).

Its output must match moe_grouped_gemm's, and the oracle's (FP8 scatter) or a
binary64 numpy SwiGLU (BF16), within the tolerance the parity tests use, on two
calls in a row (the second call finds the previous call's scratch contents),
and a call that follows one whose pipeline waits timed out must be correct
(the per-call clear of the shared scratch).  This file is collected last."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, ensure_built
from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import inputs

pytestmark = pytest.mark.gpu


def _close(got: torch.Tensor, ref, what: str):
    r = ref if isinstance(ref, np.ndarray) else ref.float().cpu().numpy()
    assert_close(got, np.asarray(r, np.float64), what)


def _fp8_case():
    M, K, N, E, k, bm = 200, 1024, 384, 16, 4, 32
    d = inputs.make_fp8_inputs(dict(M=M, K=K, N=N, E=E, k=k, softcap=0.0, zipf_bias=1.0), seed=7)
    rid, rw = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    common = dict(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER, a=cu(a_q), a_scales=cu(a_s),
                  w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                  tile_offsets=cu(lay["tile_offsets"]), block_m=bm,
                  sorted_route_ids=cu(lay["sorted_route_ids"]), route_weights=cu(rw), M=M,
                  top_k=k)
    Y = oracle.grouped_gemm_fp8(a_q, a_s, d["w_q"].numpy(), d["w_scales"].numpy(), lay["offsets"])
    ref = oracle.scatter(Y, lay["route_slot"], rw)
    return common, (M, N), ref


def test_noalloc_fp8_scatter_matches_workspace_entry_point_and_oracle():
    ensure_built()
    common, shape, ref_oracle = _fp8_case()
    ws = L.new_workspace(L.CTRL_BYTES)
    ref = torch.zeros(*shape, device="cuda")
    L.grouped_gemm(out=ref, ws=ws, **common)
    torch.cuda.synchronize()
    _close(ref, ref_oracle, "workspace entry point vs oracle")
    for call in range(2):
        out = torch.zeros(*shape, device="cuda")
        L.grouped_gemm_noalloc(out=out, **common)
        torch.cuda.synchronize()
        _close(out, ref, f"fp8 scatter, call {call}, vs moe_grouped_gemm")
        _close(out, ref_oracle, f"fp8 scatter, call {call}, vs oracle")


def test_noalloc_bf16_swiglu_matches_workspace_entry_point_and_numpy():
    ensure_built()
    g = torch.Generator().manual_seed(11)
    M, K, N, E, k, bm = 150, 256, 512, 6, 2, 64
    ids, _ = oracle.route(torch.randn(M, E, generator=g).numpy(), k)
    lay = oracle.layout(ids, E, block_m=bm)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    a_cpu = x[torch.from_numpy(lay["sorted_route_ids"] // k).long()]
    w_cpu = (torch.randn(E, N, K, generator=g) / 16).to(torch.bfloat16)
    # binary64 SwiGLU of the expert-compact rows: rows [0, N/2) of W gate, [N/2, N) up
    a64 = a_cpu.double().numpy()
    w64 = w_cpu.double().numpy()
    h_ref = np.zeros((M * k, N // 2))
    for e in range(E):
        s0, s1 = lay["offsets"][e], lay["offsets"][e + 1]
        gu = a64[s0:s1] @ w64[e].T
        gate, up = gu[:, :N // 2], gu[:, N // 2:]
        h_ref[s0:s1] = gate / (1.0 + np.exp(-gate)) * up
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    common = dict(dtype=L.DTYPE_BF16, epilogue=L.EPI_SWIGLU, a=a_cpu.cuda(), w=w_cpu.cuda(),
                  offsets=cu(lay["offsets"]), tile_offsets=cu(lay["tile_offsets"]), block_m=bm)
    ref = torch.zeros(M * k, N // 2, dtype=torch.bfloat16, device="cuda")
    L.grouped_gemm(out=ref, ws=L.new_workspace(L.CTRL_BYTES), **common)
    torch.cuda.synchronize()
    _close(ref, h_ref, "workspace entry point vs numpy")
    for call in range(2):
        out = torch.zeros_like(ref)
        L.grouped_gemm_noalloc(out=out, **common)
        torch.cuda.synchronize()
        _close(out, ref, f"bf16 swiglu, call {call}, vs moe_grouped_gemm")
        _close(out, h_ref, f"bf16 swiglu, call {call}, vs numpy")


def test_noalloc_call_after_a_timed_out_call_is_correct():
    """A call whose producer issues no loads times out (bounded waits, no
    hang) and leaves whatever it left in the shared scratch; the next call
    clears the scratch first and must be correct."""
    ensure_built()
    common, shape, ref_oracle = _fp8_case()
    try:
        L.debug_set_pipeline_fault(True, 20_000_000)      # 20 ms wait limit
        junk = torch.zeros(*shape, device="cuda")
        L.grouped_gemm_noalloc(out=junk, **common)
        torch.cuda.synchronize()
    finally:
        L.debug_set_pipeline_fault(False, 0)
    for call in range(2):
        out = torch.zeros(*shape, device="cuda")
        L.grouped_gemm_noalloc(out=out, **common)
        torch.cuda.synchronize()
        _close(out, ref_oracle, f"after a timed-out call, call {call}")
