"""Pins of the oracle's FP8 gated FFN (CPU only): the binary32 SwiGLU against
binary64 libm, the re-quantisation of h against the E4M3 error bound, the
token-major FFN against the slot-major pipeline assembled from the
separately pinned GEMM / quantiser / scatter, and a closed form that
constructed weights reduce the whole FFN to."""
import math

import numpy as np
import torch

import oracle
from mixture_experts_forward_gb300 import inputs


def _ulp32(y: np.ndarray) -> np.ndarray:
    a = np.abs(y).astype(np.float32)
    return (np.nextafter(a, np.float32(np.inf)) - a).astype(np.float64)


def _silu_mul_f64(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = g.astype(np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u.astype(np.float64)


def test_swiglu_f32_vs_binary64_libm():
    gen = np.random.default_rng(1)
    g = np.concatenate([np.linspace(-100.0, 100.0, 60_001, dtype=np.float32),
                        np.array([0.0, -0.0, 87.0, -87.0, 88.0, -88.0, 1e-30, -1e-30],
                                 np.float32)])
    u = gen.uniform(-4.0, 4.0, g.size).astype(np.float32)
    u[::7] = 1.0
    h = np.array([oracle.swiglu_f32(float(a), float(b)) for a, b in zip(g, u)], np.float32)
    ref = _silu_mul_f64(g, u)
    err = np.abs(h.astype(np.float64) - ref)
    # e = exp(-g) is within 2 ulp (pinned separately), then three binary32
    # roundings (1 + e, g / d, * u); below g = -88 the spec's exp overflows
    # to +inf and h is a signed zero where the true value is under 1e-35
    tiny = g < -88.0
    assert np.all(err[~tiny] <= 4.0 * _ulp32(ref[~tiny])), (err[~tiny] / _ulp32(ref[~tiny])).max()
    assert np.all(np.abs(ref[tiny]) < 1e-35) and np.all(h[tiny] == 0.0)
    assert oracle.swiglu_f32(0.0, 3.0) == 0.0
    assert oracle.swiglu_f32(40.0, 0.5) == 20.0          # silu(g) = g once exp(-g) < 2^-25


def test_swiglu_quant_error_bound_and_codes():
    gen = torch.Generator().manual_seed(21)
    R, I = 37, 384
    gu = (torch.randn(R, 2 * I, generator=gen) * 3.0).numpy().astype(np.float32)
    gu[0, 128:256] = 0.0                 # gate 0 -> h = 0: a zero block
    gu[1, I + 256:I + 384] = 0.0         # up 0 -> h = 0
    gu[2, 0:128] = -100.0                # exp(100) overflows: h = -0 (u > 0) or +0
    gu[3, 0:64] = -100.0                 # signed zeros inside a nonzero block
    h_q, h_s = oracle.swiglu_quant(gu)
    assert h_q.shape == (R, I) and h_s.shape == (I // 128, R)
    table = oracle.e4m3_decode_table()
    ref = _silu_mul_f64(gu[:, :I], gu[:, I:])
    for s in range(R):
        for b in range(I // 128):
            blk = ref[s, b * 128:(b + 1) * 128]
            codes = h_q[s, b * 128:(b + 1) * 128]
            sc = float(h_s[b, s])
            amax = np.abs(blk).max()
            # the scale is amax/448 of the binary32 h (within a few ulp of the exact h)
            assert abs(sc - amax / 448.0) <= 8 * 2.0 ** -24 * amax / 448.0 + 1e-40
            if sc == 0.0:
                assert np.all(codes == 0)
                continue
            deq = table[codes] * sc
            bound = (2.0 ** -4 + 2.0 ** -20) * np.abs(blk) + sc * 2.0 ** -10 * (1 + 2.0 ** -20)
            assert np.all(np.abs(deq - blk) <= bound), (s, b)
            assert np.abs(table[codes]).max() == 448.0
    assert np.all(h_q[0, 128:256] == 0) and h_s[1, 0] == 0.0
    assert np.all(h_q[1, 256:384] == 0) and h_s[2, 1] == 0.0
    assert h_s[0, 2] == 0.0 and np.all(h_q[2, 0:128] == 0)


def _ffn_fp8_case(seed: int, T=24, H=256, I=384, E=6, k=2):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g).numpy()
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wup_q, wup_s = inputs.quantize_weights_e4m3(torch.randn(E, 2 * I, H, generator=g) / math.sqrt(H))
    wdn_q, wdn_s = inputs.quantize_weights_e4m3(torch.randn(E, H, I, generator=g) / math.sqrt(I))
    return logits, x, wup_q.numpy(), wup_s.numpy(), wdn_q.numpy(), wdn_s.numpy()


def test_ffn_fp8_equals_slot_major_pipeline():
    """Token-major FFN == route -> layout -> quantise/gather -> up GEMM ->
    binary32 -> SwiGLU + quantise -> down GEMM -> scatter, each step the
    separately pinned oracle function, in the same order of operations."""
    k = 2
    logits, x, wup_q, wup_s, wdn_q, wdn_s = _ffn_fp8_case(31, k=k)
    E = wup_q.shape[0]
    ids, w = oracle.route(logits, k)
    lay = oracle.layout(ids, E)
    xb = inputs.bf16_bits(x)
    a_q, a_s = oracle.quant_gather(xb, k, lay["route_slot"])
    gu = oracle.grouped_gemm_fp8(a_q, a_s, wup_q, wup_s, lay["offsets"]).astype(np.float32)
    h_q, h_s = oracle.swiglu_quant(gu)
    Y = oracle.grouped_gemm_fp8(h_q, h_s, wdn_q, wdn_s, lay["offsets"])
    ref = oracle.scatter(Y, lay["route_slot"], w)
    got = oracle.ffn_fp8(xb, ids, w, wup_q, wup_s, wdn_q, wdn_s, threads=2)
    assert np.array_equal(got, ref)
    tok = np.array([23, 0, 11], np.int32)
    part = oracle.ffn_fp8(xb, ids, w, wup_q, wup_s, wdn_q, wdn_s, tokens=tok, threads=3)
    assert np.array_equal(part, ref[tok])


def test_ffn_fp8_constructed_weights_closed_form():
    """Gate rows read only column 0 (x[:,0] = 1, weight code 1.0, block scale
    G_e), so g = G_e = 32(e+1) and silu(g) = g in binary32; up rows and the down
    projection are identities.  Then h = G_e * u re-quantises to the token's
    own codes and out[t] = sum_j w[t,j] G_{e_j} dequant(x_t)."""
    T, H, E, k = 16, 256, 4, 2
    I = H
    one = oracle.e4m3_encode(1.0)
    G = np.array([32.0 * (e + 1) for e in range(E)])
    wup_q = np.zeros((E, 2 * I, H), np.uint8)
    wup_q[:, np.arange(I), 0] = one                          # gate: column 0
    wup_q[:, I + np.arange(I), np.arange(I)] = one           # up: identity
    wup_s = np.full((E, 2 * I // 128, H // 128), 5.0, np.float32)
    for e in range(E):
        wup_s[e, :I // 128, 0] = np.float32(G[e])
        wup_s[e, :I // 128, 1] = 3.0
        for b in range(H // 128):
            wup_s[e, I // 128 + b, b] = 1.0
    wdn_q = np.zeros((E, H, I), np.uint8)
    wdn_q[:, np.arange(H), np.arange(H)] = one
    wdn_s = np.full((E, H // 128, I // 128), 7.0, np.float32)
    for b in range(H // 128):
        wdn_s[:, b, b] = 1.0
    gen = torch.Generator().manual_seed(4)
    x = (torch.rand(T, H, generator=gen) * 1.8 - 0.9).to(torch.bfloat16)
    x[:, 0] = 1.0
    ids = np.stack([np.arange(T) % E, (np.arange(T) + 1) % E], axis=1).astype(np.int32)
    w = torch.softmax(torch.randn(T, k, generator=gen), dim=1).numpy().astype(np.float32)
    xb = inputs.bf16_bits(x)
    got = oracle.ffn_fp8(xb, ids, w, wup_q, wup_s, wdn_q, wdn_s)
    q, s = oracle.quant_gather(xb, 1, np.arange(T, dtype=np.int32))
    table = oracle.e4m3_decode_table()
    xdeq = (table[q].reshape(T, H // 128, 128) * s.T[:, :, None].astype(np.float64)).reshape(T, H)
    ref = np.zeros((T, H))
    for j in range(k):
        ref += (w[:, j].astype(np.float64) * G[ids[:, j]])[:, None] * xdeq
    assert np.all((got == 0) == (ref == 0))
    assert np.allclose(got, ref, rtol=4e-6, atol=0.0)
