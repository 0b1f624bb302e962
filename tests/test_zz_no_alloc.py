"""moe_grouped_gemm_noalloc — the grouped GEMM for callers that cannot
allocate device memory (no workspace argument; the kernel's 256-byte control
block lives in a static array inside the library).  Its output must match
moe_grouped_gemm's, within the tolerance the parity tests use, on two calls
in a row (the second call finds the previous call's scratch contents)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL_L2, MAX_ABS_FRAC, bits, ensure_built
from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import inputs

pytestmark = pytest.mark.gpu


def _close(got: torch.Tensor, ref: torch.Tensor, what: str):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert np.abs(g - r).max() <= MAX_ABS_FRAC * max(np.abs(r).max(), 1e-30), what


def test_noalloc_fp8_scatter_matches_workspace_entry_point():
    ensure_built()
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
    ws = L.new_workspace(L.CTRL_BYTES)
    ref = torch.zeros(M, N, device="cuda")
    L.grouped_gemm(out=ref, ws=ws, **common)
    for call in range(2):
        out = torch.zeros(M, N, device="cuda")
        L.grouped_gemm_noalloc(out=out, **common)
        torch.cuda.synchronize()
        _close(out, ref, f"fp8 scatter, call {call}")


def test_noalloc_bf16_swiglu_matches_workspace_entry_point():
    ensure_built()
    g = torch.Generator().manual_seed(11)
    M, K, N, E, k, bm = 150, 256, 512, 6, 2, 64
    ids, _ = oracle.route(torch.randn(M, E, generator=g).numpy(), k)
    lay = oracle.layout(ids, E, block_m=bm)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    a = x[torch.from_numpy(lay["sorted_route_ids"] // k).long()].cuda()
    w = (torch.randn(E, N, K, generator=g) / 16).to(torch.bfloat16).cuda()
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    common = dict(dtype=L.DTYPE_BF16, epilogue=L.EPI_SWIGLU, a=a, w=w, offsets=cu(lay["offsets"]),
                  tile_offsets=cu(lay["tile_offsets"]), block_m=bm)
    ref = torch.zeros(M * k, N // 2, dtype=torch.bfloat16, device="cuda")
    L.grouped_gemm(out=ref, ws=L.new_workspace(L.CTRL_BYTES), **common)
    for call in range(2):
        out = torch.zeros_like(ref)
        L.grouped_gemm_noalloc(out=out, **common)
        torch.cuda.synchronize()
        _close(out, ref, f"bf16 swiglu, call {call}")
