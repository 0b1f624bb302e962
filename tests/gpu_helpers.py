"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import build as moe_build
from mixture_experts_forward_gb300 import inputs

THREADS = max(1, min(16, os.cpu_count() or 1))

# Output tolerance of the fused forward against the oracle's binary64 sum over
# the same quantised values: relative L2 <= 5e-3 and max-abs <= 1e-2 * max|ref|.
REL_L2 = 5e-3
MAX_ABS_FRAC = 1e-2


def ensure_built():
    moe_build.build()
    L.lib()


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bits(x_bf16: torch.Tensor) -> np.ndarray:
    return inputs.bf16_bits(x_bf16.cpu())


def assert_close(out: torch.Tensor, ref: np.ndarray, what: str = ""):
    got = out.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / max(denom, 1e-30)
    mx = np.abs(got - ref).max() if got.size else 0.0
    lim = MAX_ABS_FRAC * max(np.abs(ref).max() if ref.size else 0.0, 1e-30)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= lim, f"{what}: max-abs {mx:.3e} > {lim:.3e}"
    return rel, mx


def fp8_device_inputs(d):
    return dict(logits=d["logits"].cuda(), x=d["x"].cuda(), w_q=d["w_q"].cuda(),
                w_scales=d["w_scales"].cuda())


def run_forward_fp8(dev, cfg, block_m=0, sched=L.SCHED_QUEUE, k_splits=0, use_graph=1,
                    renorm=1, softcap=None, gather_rows=0):
    M, E = dev["logits"].shape
    K = dev["x"].shape[1]
    N = dev["w_q"].shape[1]
    args = L.forward_args(dtype=L.DTYPE_FP8, M=M, K=K, N=N, E=E, top_k=cfg["k"],
                          softcap=cfg["softcap"] if softcap is None else softcap, renorm=renorm,
                          logits=dev["logits"], x=dev["x"], w=dev["w_q"], w_scales=dev["w_scales"],
                          block_m=block_m, sched=sched, k_splits=k_splits, use_graph=use_graph,
                          gather_rows=gather_rows)
    ws = L.new_workspace(L.workspace_size(args))
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    L.forward(args, out, ws)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    return out, args, ws


def run_forward_bf16(dev, cfg, block_m=0, sched=L.SCHED_QUEUE, use_graph=1, gather_rows=0):
    T, E = dev["logits"].shape
    H = dev["x"].shape[1]
    I = dev["w_dn"].shape[2]
    args = L.forward_args(dtype=L.DTYPE_BF16, M=T, K=H, N=I, E=E, top_k=cfg["k"], softcap=0.0,
                          logits=dev["logits"], x=dev["x"], w=dev["w_up"], w2=dev["w_dn"],
                          block_m=block_m, sched=sched, use_graph=use_graph,
                          gather_rows=gather_rows)
    ws = L.new_workspace(L.workspace_size(args))
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    L.forward(args, out, ws)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    return out, args, ws


def sample_tokens(M: int, n: int, seed: int = 0) -> np.ndarray:
    if n >= M:
        return np.arange(M, dtype=np.int32)
    g = np.random.default_rng(seed)
    pick = np.sort(g.choice(M, size=n - 2, replace=False))
    return np.unique(np.concatenate([[0, M - 1], pick])).astype(np.int32)
