"""Pins of the oracle's pipeline steps (CPU only): brute force on tiny inputs,
invariants that fix each step, special cases that reduce to textbook
routines, and an independent token-major dense path."""
import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_forward_gb300 import inputs


# ------------------------------------------------------------------ routing
def _brute_topk(z: np.ndarray, k: int) -> np.ndarray:
    """Exhaustive ordering of all experts by (value desc, id asc)."""
    M, E = z.shape
    out = np.zeros((M, k), np.int32)
    for t in range(M):
        order = sorted(range(E), key=lambda e: (-float(z[t, e]), e))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("M,E,k", [(37, 8, 2), (16, 256, 8), (9, 33, 33), (5, 1, 1)])
def test_route_topk_brute_force(M, E, k):
    g = torch.Generator().manual_seed(M * 1000 + E)
    logits = torch.randn(M, E, generator=g).numpy()
    ids, w = oracle.route(logits, k, softcap=0.0)
    assert np.array_equal(ids, _brute_topk(logits, k))
    # weights: softmax over the selected logits (binary64 textbook form)
    sel = np.take_along_axis(logits.astype(np.float64), ids, axis=1)
    ref = np.exp(sel - sel.max(axis=1, keepdims=True))
    ref /= ref.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-7)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= k * 2.0 ** -23 + 1e-7)
    assert np.all(np.diff(sel, axis=1) <= 0)


def test_route_ties_go_to_lower_id():
    logits = np.zeros((3, 8), np.float32)
    logits[0] = [1, 3, 3, 0, 3, 2, 2, 0]
    logits[1] = 0.5                                   # all equal
    logits[2] = [-1, -1, 5, 5, -1, 5, 5, 5]
    ids, w = oracle.route(logits, 4)
    assert ids[0].tolist() == [1, 2, 4, 5]
    assert ids[1].tolist() == [0, 1, 2, 3]
    assert ids[2].tolist() == [2, 3, 5, 6]
    assert np.allclose(w[1], 0.25) and np.all(w[2] == w[2][0])
    # -0.0 and +0.0 compare equal: the lower id wins
    z = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert oracle.route(z, 1)[0][0, 0] == 0


def test_route_softcap_matches_binary64_tanh():
    g = torch.Generator().manual_seed(7)
    logits = (torch.randn(64, 256, generator=g) * 3).numpy()
    ids, w = oracle.route(logits, 8, softcap=30.0)
    z = 30.0 * np.tanh(logits.astype(np.float64) / 30.0)
    assert np.array_equal(ids, _brute_topk(z, 8))       # no near-ties in this seed
    sel = np.take_along_axis(z, ids, axis=1)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=2e-6, atol=1e-7)


def test_route_full_softmax_equals_textbook():
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(20, 16, generator=g).numpy()
    ids, w = oracle.route(logits, 16, renorm=0)
    ref = torch.softmax(torch.from_numpy(logits).double(), dim=1).numpy()
    got = np.zeros_like(ref)
    np.put_along_axis(got, ids, w.astype(np.float64), axis=1)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-8)
    # renorm=0 with k<E: the selected full-softmax values, summing below 1
    ids4, w4 = oracle.route(logits, 4, renorm=0)
    assert np.allclose(w4, np.take_along_axis(ref, ids4, axis=1), rtol=1e-6)


# ------------------------------------------------------------------ layout
def _check_layout(ids, E, lay, block_m):
    M, k = ids.shape
    R = M * k
    cnt, off = lay["counts"], lay["offsets"]
    assert np.array_equal(cnt, np.bincount(ids.ravel(), minlength=E))
    assert cnt.sum() == R and off[0] == 0 and off[-1] == R
    assert np.all(np.diff(off) == cnt)
    srt, slot = lay["sorted_route_ids"], lay["route_slot"]
    assert np.array_equal(np.sort(srt), np.arange(R))           # every route once
    assert np.array_equal(slot[srt], np.arange(R))              # inverse permutation
    flat = ids.ravel()
    for e in range(E):
        seg = srt[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                         # stable: ascending route id
    # task list of the Weave retelling (section 4.3): per expert, tiles of
    # block_m rows starting at offsets[e] + tile_start
    tasks = []
    for e in range(E):
        for start in range(0, int(cnt[e]), block_m):
            tasks.append((e, int(off[e]) + start, min(block_m, int(cnt[e]) - start)))
    tile_off = lay["tile_offsets"]
    assert tile_off[-1] == len(tasks)
    for e in range(E):
        mine = [t for t in tasks if t[0] == e]
        assert tile_off[e + 1] - tile_off[e] == len(mine)
        if mine:
            assert tasks[tile_off[e]] == mine[0]


@pytest.mark.parametrize("M,E,k,bm", [(16, 8, 2, 16), (128, 256, 8, 16), (333, 16, 8, 64),
                                      (1, 4, 4, 128), (50, 1024, 3, 32)])
def test_layout_invariants(M, E, k, bm):
    g = torch.Generator().manual_seed(M + E)
    ids = torch.rand(M, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32).numpy()
    lay = oracle.layout(ids, E, block_m=bm)
    _check_layout(ids, E, lay, bm)


def test_layout_skewed_and_empty_experts():
    ids = np.zeros((40, 2), np.int32)
    ids[:, 1] = 5
    ids[3, 0] = 7
    lay = oracle.layout(ids, 9, block_m=16)
    _check_layout(ids, 9, lay, 16)
    assert lay["counts"].tolist() == [39, 0, 0, 0, 0, 40, 0, 1, 0]
    with pytest.raises(ValueError):
        oracle.layout(np.array([[0, 9]], np.int32), 9)


# ------------------------------------------------------------------ quantisation
def test_quant_gather_bounds_and_torch_cast():
    d = inputs.make_fp8_inputs("tiny_fp8", seed=0)
    x = d["x"]
    ids, _ = oracle.route(d["logits"].numpy(), 2)
    lay = oracle.layout(ids, 8)
    a_q, a_s = oracle.quant_gather(inputs.bf16_bits(x), 2, lay["route_slot"])
    M, K = x.shape
    xf = x.float().numpy()
    table = oracle.e4m3_decode_table()
    blocks = np.abs(xf).reshape(M, K // 128, 128).max(axis=2)
    for t in range(M):
        for j in range(2):
            s = lay["route_slot"][t * 2 + j]
            q = a_q[s]
            sc = a_s[:, s]
            assert np.array_equal(sc, (blocks[t] / np.float32(448.0)).astype(np.float32))
            # the codes equal torch's own E4M3 cast of x * (1/s)
            inv = (np.float32(1.0) / sc).astype(np.float32)
            scaled = (xf[t].reshape(-1, 128) * inv[:, None]).astype(np.float32)
            ref = torch.from_numpy(scaled.ravel()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q, ref)
            # per-element error bound of a 3-bit-mantissa RNE code
            deq = table[q].reshape(-1, 128) * sc[:, None].astype(np.float64)
            err = np.abs(deq - xf[t].reshape(-1, 128))
            bound = 2.0 ** -4 * np.abs(xf[t].reshape(-1, 128)) + sc[:, None] * 2.0 ** -10 \
                + 2.0 ** -23 * np.abs(xf[t].reshape(-1, 128)) * 2
            assert np.all(err <= bound)
            # the block maximum maps to the top code 448
            assert np.all(np.abs(table[q].reshape(-1, 128)).max(axis=1) == 448.0)


def test_quant_zero_block():
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    x[1, 128:] = 1.5
    a_q, a_s = oracle.quant_gather(inputs.bf16_bits(x), 1, np.array([1, 0], np.int32))
    assert np.all(a_q[1] == 0) and np.all(a_s[:, 1] == 0)     # token 0 -> slot 1
    assert np.all(a_q[0, :128] == 0) and a_s[0, 0] == 0
    assert np.all(a_q[0, 128:] == 0x7E) and a_s[1, 0] == np.float32(1.5) / np.float32(448)


# ------------------------------------------------------------------ GEMM + scatter
def test_forward_matches_independent_dense_path():
    d = inputs.make_fp8_inputs("tiny_fp8", seed=0)
    for softcap in (0.0, 30.0):
        r = oracle.forward_fp8(d["logits"].numpy(), inputs.bf16_bits(d["x"]), d["w_q"].numpy(),
                               d["w_scales"].numpy(), k=2, softcap=softcap)
        dense = oracle.dense_fp8(inputs.bf16_bits(d["x"]), r["ids"], r["weights"],
                                 d["w_q"].numpy(), d["w_scales"].numpy())
        assert np.allclose(r["out"], dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_gemm_single_expert_is_textbook_matmul():
    """E=1, k=1: Y = diag(sa) dq(A) (dq(W) * sb)^T computed with numpy matmul."""
    g = torch.Generator().manual_seed(11)
    M, K, N = 24, 384, 256
    w = torch.randn(1, N, K, generator=g) * 0.05
    w_q, w_s = inputs.quantize_weights_e4m3(w)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ids = np.zeros((M, 1), np.int32)
    lay = oracle.layout(ids, 1)
    a_q, a_s = oracle.quant_gather(inputs.bf16_bits(x), 1, lay["route_slot"])
    Y = oracle.grouped_gemm_fp8(a_q, a_s, w_q.numpy(), w_s.numpy(), lay["offsets"])
    table = oracle.e4m3_decode_table()
    A = table[a_q].reshape(M, K // 128, 128) * a_s.T[:, :, None].astype(np.float64)
    W = table[w_q.numpy()[0]].reshape(N // 128, 128, K // 128, 128) \
        * w_s.numpy()[0][:, None, :, None].astype(np.float64)
    ref = A.reshape(M, K) @ W.reshape(N, K).T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    out = oracle.scatter(Y, lay["route_slot"], np.ones((M, 1), np.float32))
    assert np.array_equal(out, Y[lay["route_slot"]])


def test_gemm_identity_weights_return_dequantised_rows():
    M, K, N, E = 8, 256, 256, 2
    w_q = np.zeros((E, N, K), np.uint8)
    one = oracle.e4m3_encode(1.0)
    for e in range(E):
        w_q[e, np.arange(N), np.arange(N) % K] = one
    w_s = np.full((E, N // 128, K // 128), 0.5, np.float32)
    g = torch.Generator().manual_seed(5)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ids = (np.arange(M * 1) % E).astype(np.int32).reshape(M, 1)
    lay = oracle.layout(ids, E)
    a_q, a_s = oracle.quant_gather(inputs.bf16_bits(x), 1, lay["route_slot"])
    Y = oracle.grouped_gemm_fp8(a_q, a_s, w_q, w_s, lay["offsets"])
    table = oracle.e4m3_decode_table()
    deq = table[a_q].reshape(M, K // 128, 128) * a_s.T[:, :, None].astype(np.float64)
    assert np.array_equal(Y, 0.5 * deq.reshape(M, K)[:, :N])


def test_gemm_bf16_single_expert_is_textbook_matmul():
    """E=1: Y = A W^T of the bf16 values, against numpy's matmul in binary64."""
    g = torch.Generator().manual_seed(12)
    R, K, N = 19, 320, 96
    a = torch.randn(R, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(1, N, K, generator=g) / 16).to(torch.bfloat16)
    Y = oracle.grouped_gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(w),
                                 np.array([0, R], np.int32), threads=2)
    ref = a.double().numpy() @ w[0].double().numpy().T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_bf16_scaled_identity_per_expert():
    """Expert e's weights are (e + 1) * I: every slot's row comes back scaled by
    its own expert's factor, exactly (a wrong expert index or row fails)."""
    g = torch.Generator().manual_seed(13)
    E, K = 3, 64
    counts = [5, 0, 7]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    a = torch.randn(R, K, generator=g).to(torch.bfloat16)
    w = torch.zeros(E, K, K)
    for e in range(E):
        w[e] = (e + 1) * torch.eye(K)
    w = w.to(torch.bfloat16)
    Y = oracle.grouped_gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(w), offsets)
    A = a.double().numpy()
    for e in range(E):
        s0, s1 = offsets[e], offsets[e + 1]
        assert np.array_equal(Y[s0:s1], (e + 1) * A[s0:s1])


def test_forward_token_subset_equals_full():
    d = inputs.make_fp8_inputs("tiny_fp8", seed=3)
    args = (d["logits"].numpy(), inputs.bf16_bits(d["x"]), d["w_q"].numpy(), d["w_scales"].numpy())
    full = oracle.forward_fp8(*args, k=2)
    tok = np.array([15, 0, 7], np.int32)
    part = oracle.forward_fp8(*args, k=2, tokens=tok, threads=3)
    assert np.array_equal(part["out"], full["out"][tok])


# ------------------------------------------------------------------ BF16 gated FFN
def test_ffn_bf16_against_numpy_and_torch_rounding():
    g = torch.Generator().manual_seed(9)
    T, H, I, E, k = 12, 64, 32, 4, 2
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w_up = (torch.randn(E, 2 * I, H, generator=g) / 8).to(torch.bfloat16)
    w_dn = (torch.randn(E, H, I, generator=g) / 6).to(torch.bfloat16)
    ids = torch.rand(T, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32).numpy()
    wts = torch.softmax(torch.randn(T, k, generator=g), dim=1).numpy().astype(np.float32)
    got = oracle.ffn_bf16(inputs.bf16_bits(x), ids, wts, inputs.bf16_bits(w_up),
                          inputs.bf16_bits(w_dn), threads=2)
    X = x.double().numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            gu = X[t] @ w_up[e].double().numpy().T
            gate, up = gu[:I], gu[I:]
            h = torch.from_numpy(gate / (1 + np.exp(-gate)) * up).float().to(torch.bfloat16).double()
            ref[t] += float(wts[t, j]) * (h.numpy() @ w_dn[e].double().numpy().T)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-9)


def test_ffn_zero_gate_gives_zero():
    T, H, I, E = 4, 16, 8, 2
    x = torch.ones(T, H, dtype=torch.bfloat16)
    w_up = torch.ones(E, 2 * I, H, dtype=torch.bfloat16)
    w_up[:, :I] = 0
    w_dn = torch.ones(E, H, I, dtype=torch.bfloat16)
    ids = np.array([[0, 1]] * T, np.int32)
    out = oracle.ffn_bf16(inputs.bf16_bits(x), ids, np.full((T, 2), 0.5, np.float32),
                          inputs.bf16_bits(w_up), inputs.bf16_bits(w_dn))
    assert np.all(out == 0.0)
