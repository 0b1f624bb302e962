"""Seeded synthetic inputs for the fused MoE forward.

This module is the only code shared by the oracle's tests and the CUDA path's
tests and benchmark.  It draws random numbers and lays them out; it performs
none of the forward's arithmetic.  The one transformation here is the
preparation of the FP8 expert weights (the forward takes them already
quantised): each 128x128 weight block gets scale = amax/448 and is cast to
``torch.float8_e4m3fn`` by PyTorch's own conversion.

Workloads (shapes, value distributions and routing structure follow the
source pages' workloads; no dataset is involved):

* ``tiny_fp8`` — M=16, K=256, N=128, E=8, top-2; logits, x ~ N(0,1);
  W ~ N(0, 1/sqrt(K)).  A correctness case.
* ``qwen_small_batch_fp8`` — M=128, K=2048, N=512, E=256, top-8, softcap 30:
  the shape of the problem table in "Fused MoE FP8: 8.09 -> 13.18 TFLOPS".
* ``skewed_large_batch_fp8`` — M=4096, same dims; logits N(0,1) plus a Zipf
  bias 2.5*ln(1/(e+1)) so expert loads differ by more than 10x.
* ``bf16_ffn`` — T=8192, H=3072, I=1536, E=16, top-8 gated FFN (the shape of
  section 3 "Benchmark design" of the H200 grouped-GEMM page) with balanced,
  uniform and Zipf(s=1.2) routing.
* ``imbalance_bf16`` — T=16384, H=4096, I=1024, E=8, top-2 (the Mixtral-like
  layer of the Weave retelling, section 1.2) with expert loads whose
  max/min ratio is rho in {1, 4, 16, 40}.
* ``ffn_fp8`` — the ``bf16_ffn`` shape and routing with FP8 expert weights
  (gate+up [E,2I,H] and down [E,H,I], each prepared like the FP8 workloads'
  weights: std 1/sqrt(fan_in), 128x128 blocks, amax/448 scales).

Routing structure for the BF16 cases is realised through the logits: the
chosen experts get +20 on top of N(0,1) noise and softcap is off, so top-k
recovers exactly the chosen set.
"""
from __future__ import annotations

import math

import numpy as np
import torch

FP8_CONFIGS = {
    "tiny_fp8": dict(M=16, K=256, N=128, E=8, k=2, softcap=0.0, zipf_bias=0.0),
    "qwen_small_batch_fp8": dict(M=128, K=2048, N=512, E=256, k=8, softcap=30.0, zipf_bias=0.0),
    "skewed_large_batch_fp8": dict(M=4096, K=2048, N=512, E=256, k=8, softcap=30.0,
                                   zipf_bias=2.5),
}

FFN_FP8_CONFIGS = {
    "ffn_fp8": dict(T=8192, H=3072, I=1536, E=16, k=8),
}

BF16_CONFIGS = {
    "bf16_ffn": dict(T=8192, H=3072, I=1536, E=16, k=8),
    "imbalance_bf16": dict(T=16384, H=4096, I=1024, E=8, k=2),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def quantize_weights_e4m3(w: torch.Tensor):
    """[E, N, K] float32 -> (uint8 codes [E,N,K], float32 scales [E,N/128,K/128]).

    Weight preparation only (the forward receives these as inputs)."""
    E, N, K = w.shape
    blocks = w.reshape(E, N // 128, 128, K // 128, 128)
    amax = blocks.abs().amax(dim=(2, 4))                       # [E, N/128, K/128]
    scale = amax / 448.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    q = (blocks / safe[:, :, None, :, None]).clamp(-448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(E, N, K)
    return codes.contiguous(), scale.to(torch.float32).contiguous()


def make_fp8_inputs(name_or_cfg, seed: int = 0, **overrides):
    """Inputs of one FP8 workload as CPU tensors:
    logits f32 [M,E], x bf16 [M,K], w_q uint8 [E,N,K], w_scales f32 [E,N/128,K/128]."""
    cfg = dict(FP8_CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    cfg.update(overrides)
    M, K, N, E = cfg["M"], cfg["K"], cfg["N"], cfg["E"]
    g = _gen(seed)
    logits = torch.randn(M, E, generator=g, dtype=torch.float32)
    if cfg.get("zipf_bias", 0.0):
        rank = torch.arange(1, E + 1, dtype=torch.float64)
        logits = (logits + (cfg["zipf_bias"] * torch.log(1.0 / rank)).to(torch.float32)).contiguous()
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    codes, scales = _normal_weights_e4m3(E, N, K, 1.0 / math.sqrt(K), g)
    return dict(cfg=cfg, logits=logits, x=x, w_q=codes, w_scales=scales)


def _normal_weights_e4m3(E: int, N: int, K: int, std: float, g: torch.Generator):
    """N(0, std) weights [E, N, K] drawn expert-chunk by expert-chunk, then
    prepared by quantize_weights_e4m3."""
    codes = torch.empty(E, N, K, dtype=torch.uint8)
    scales = torch.empty(E, N // 128, K // 128, dtype=torch.float32)
    chunk = max(1, (1 << 26) // (N * K))       # bound the float32 temporaries
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        w = torch.randn(e1 - e0, N, K, generator=g, dtype=torch.float32) * std
        codes[e0:e1], scales[e0:e1] = quantize_weights_e4m3(w)
    return codes, scales


def _chosen_to_logits(chosen: torch.Tensor, E: int, g: torch.Generator) -> torch.Tensor:
    T = chosen.shape[0]
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    bump = torch.zeros(T, E, dtype=torch.float32)
    bump.scatter_(1, chosen.long(), 20.0)
    return (logits + bump).contiguous()


def routing_choice(T: int, E: int, k: int, routing: str, g: torch.Generator,
                   rho: float = 1.0) -> torch.Tensor:
    """Chosen expert sets [T, k] (distinct per token) for the BF16 workloads."""
    if routing == "balanced":
        t = torch.arange(T)[:, None]
        j = torch.arange(k)[None, :]
        return ((k * t + j) % E).to(torch.int32)
    if routing == "uniform":
        return torch.rand(T, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32)
    if routing.startswith("zipf"):
        s = float(routing[4:] or 1.2)
        p = torch.arange(1, E + 1, dtype=torch.float64) ** (-s)
        return torch.multinomial(p.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    if routing == "loads":
        # expert loads proportional to rho^(-e/(E-1)), summing to T*k, each <= T
        assert k == 2, "the load-profile routing assigns two experts per token"
        raw = np.array([rho ** (-e / (E - 1)) for e in range(E)])
        target = raw / raw.sum() * T * k
        loads = np.floor(target).astype(np.int64)
        rem = T * k - loads.sum()
        for e in np.argsort(-(target - loads), kind="stable")[:rem]:
            loads[e] += 1
        assert loads.max() <= T and loads.sum() == T * k
        flat = np.repeat(np.arange(E), loads)
        pair = np.stack([flat[:T], flat[T:]], axis=1)
        perm = torch.randperm(T, generator=g).numpy()
        return torch.from_numpy(pair[perm].astype(np.int32))
    raise ValueError(routing)


def make_bf16_inputs(name_or_cfg, routing: str = "uniform", seed: int = 0, rho: float = 1.0,
                     **overrides):
    """Inputs of one BF16 gated-FFN workload as CPU tensors:
    logits f32 [T,E], x bf16 [T,H], w_up bf16 [E,2I,H] (rows [0,I) gate,
    [I,2I) up), w_dn bf16 [E,H,I]."""
    cfg = dict(BF16_CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    cfg.update(overrides)
    T, H, I, E, k = cfg["T"], cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    g = _gen(seed)
    chosen = routing_choice(T, E, k, routing, g, rho=rho)
    logits = _chosen_to_logits(chosen, E, g)
    x = torch.randn(T, H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    w_up = (torch.randn(E, 2 * I, H, generator=g, dtype=torch.float32) / math.sqrt(H)).to(torch.bfloat16)
    w_dn = (torch.randn(E, H, I, generator=g, dtype=torch.float32) / math.sqrt(I)).to(torch.bfloat16)
    cfg.update(routing=routing, rho=rho, softcap=0.0)
    return dict(cfg=cfg, logits=logits, x=x, w_up=w_up, w_dn=w_dn, chosen=chosen)


def make_fp8_ffn_inputs(name_or_cfg, routing: str = "uniform", seed: int = 0, **overrides):
    """Inputs of one FP8 gated-FFN workload as CPU tensors: logits f32 [T,E],
    x bf16 [T,H], wup_q uint8 [E,2I,H] (rows [0,I) gate, [I,2I) up) with
    wup_s f32 [E,2I/128,H/128], wdn_q uint8 [E,H,I] with wdn_s f32
    [E,H/128,I/128]."""
    cfg = dict(FFN_FP8_CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    cfg.update(overrides)
    T, H, I, E, k = cfg["T"], cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    g = _gen(seed)
    chosen = routing_choice(T, E, k, routing, g)
    logits = _chosen_to_logits(chosen, E, g)
    x = torch.randn(T, H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    wup_q, wup_s = _normal_weights_e4m3(E, 2 * I, H, 1.0 / math.sqrt(H), g)
    wdn_q, wdn_s = _normal_weights_e4m3(E, H, I, 1.0 / math.sqrt(I), g)
    cfg.update(routing=routing, softcap=0.0)
    return dict(cfg=cfg, logits=logits, x=x, wup_q=wup_q, wup_s=wup_s, wdn_q=wdn_q, wdn_s=wdn_s,
                chosen=chosen)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor -> numpy uint16 bit patterns (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
