"""Oracle for the fused MoE forward — TEST INFRASTRUCTURE ONLY.

A ctypes binding over ``liboracle.so`` (built from ``moe_oracle.cpp`` with
``build()``).  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline legs may import this package; the product path never does.

The C++ file states, function by function, which passage of the source pages
each step follows:

* "Fused MoE FP8: 8.09 -> 13.18 TFLOPS (1.63x)" — pipeline overview, section
  "Baseline: 7 kernels" items 1-7, sections "Fusion 1/2/3";
* "H200 MoE Grouped GEMM: accounting fix, online replay, SM90 tuning" —
  section 4 (compact routed rows) and the config-tuning benchmark design
  (gated up projection + down projection);
* the blog retelling of "Weave" — section 4.3 (histogram, prefix, per-expert
  tiles);
* the FP8 gated FFN (gate+up projection, SiLU, down projection: the closing
  "Reference: vLLM full MLP" section of the Fused MoE FP8 page and the H200
  page's config-tuning section 3), with h re-quantised by the 1x128 rule.

Parity status: every function is pinned by a ``-m "not gpu"`` test
(brute force, closed forms, libm, torch's float8 cast); none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (plain g++, no fast-math, no contraction)."""
    hdr = os.path.join(_HERE, "moe_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i = ctypes.c_int
        f = ctypes.c_float
        L.oracle_exp_spec.argtypes = [f]
        L.oracle_exp_spec.restype = f
        L.oracle_tanh_spec.argtypes = [f]
        L.oracle_tanh_spec.restype = f
        L.oracle_e4m3_encode.argtypes = [f]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_bf16_round.argtypes = [ctypes.c_double]
        L.oracle_bf16_round.restype = ctypes.c_uint16
        for nm in ("oracle_exp_spec_array", "oracle_tanh_spec_array", "oracle_e4m3_encode_array"):
            getattr(L, nm).argtypes = [P, ctypes.c_int64, P]
        L.oracle_route.argtypes = [P, i, i, i, f, i, P, P]
        L.oracle_layout.argtypes = [P, i, i, i, i, P, P, P, P, P]
        L.oracle_layout.restype = i
        L.oracle_quant_gather.argtypes = [P, i, i, i, P, P, P]
        L.oracle_grouped_gemm_fp8.argtypes = [P, P, i, i, P, P, i, i, P, P, i, P]
        L.oracle_scatter.argtypes = [P, P, P, i, i, P, i, P]
        L.oracle_grouped_gemm_bf16.argtypes = [P, i, i, P, i, i, P, i, P]
        L.oracle_forward_fp8.argtypes = [P, P, P, P, i, i, i, i, i, f, i, i, P, i, i,
                                         P, P, P, P, P, P, P, P, P, P]
        L.oracle_dense_fp8.argtypes = [P, P, P, P, P, i, i, i, i, i, P, i, i, P]
        L.oracle_ffn_bf16.argtypes = [P, P, P, P, P, i, i, i, i, i, P, i, i, P]
        L.oracle_swiglu_f32.argtypes = [f, f]
        L.oracle_swiglu_f32.restype = f
        L.oracle_swiglu_quant.argtypes = [P, i, i, P, P]
        L.oracle_ffn_fp8.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, i, P]
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- scalars
def exp_spec(x: float) -> float:
    return lib().oracle_exp_spec(x)


def tanh_spec(t: float) -> float:
    return lib().oracle_tanh_spec(t)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def e4m3_decode(c: int) -> float:
    return lib().oracle_e4m3_decode(c)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def exp_spec_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_exp_spec_array(_p(x), x.size, _p(y))
    return y


def tanh_spec_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_tanh_spec_array(_p(x), x.size, _p(y))
    return y


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), x.size, _p(y))
    return y


def bf16_round(v: float) -> int:
    return lib().oracle_bf16_round(v)


# ----------------------------------------------------------------- steps
def route(logits: np.ndarray, k: int, softcap: float = 0.0, renorm: int = 1):
    logits = _c(logits, np.float32)
    M, E = logits.shape
    ids = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float32)
    lib().oracle_route(_p(logits), M, E, k, softcap, renorm, _p(ids), _p(w))
    return ids, w


def layout(ids: np.ndarray, E: int, block_m: int = 16):
    ids = _c(ids, np.int32)
    M, k = ids.shape
    R = M * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    sorted_ids = np.zeros(R, np.int32)
    route_slot = np.zeros(R, np.int32)
    tile_off = np.zeros(E + 1, np.int32)
    rc = lib().oracle_layout(_p(ids), M, E, k, block_m, _p(counts), _p(offsets),
                             _p(sorted_ids), _p(route_slot), _p(tile_off))
    if rc != 0:
        raise ValueError("expert id out of range")
    return dict(counts=counts, offsets=offsets, sorted_route_ids=sorted_ids,
                route_slot=route_slot, tile_offsets=tile_off)


def quant_gather(x_bf16_bits: np.ndarray, k: int, route_slot: np.ndarray):
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    R = M * k
    a_q = np.zeros((R, K), np.uint8)
    a_s = np.zeros((K // 128, R), np.float32)
    lib().oracle_quant_gather(_p(x), M, K, k, _p(_c(route_slot, np.int32)), _p(a_q), _p(a_s))
    return a_q, a_s


def grouped_gemm_fp8(a_q, a_scales, w_q, w_scales, offsets, row_mask=None, threads=1):
    a_q = _c(a_q, np.uint8)
    a_scales = _c(a_scales, np.float32)
    w_q = _c(w_q, np.uint8)
    w_scales = _c(w_scales, np.float32)
    R, K = a_q.shape
    E, N, _ = w_q.shape
    Y = np.zeros((R, N), np.float64)
    mask = None if row_mask is None else _c(row_mask, np.uint8)
    lib().oracle_grouped_gemm_fp8(_p(a_q), _p(a_scales), R, K, _p(w_q), _p(w_scales), E, N,
                                  _p(_c(offsets, np.int32)), _p(mask), threads, _p(Y))
    return Y


def grouped_gemm_bf16(a_bits, w_bits, offsets, threads=1):
    """BF16 grouped GEMM on expert-compact rows: a u16 bf16 bits [R, K], w u16
    bf16 bits [E, N, K] -> Y f64 [R, N] (slots outside every expert: 0)."""
    a = _c(a_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    R, K = a.shape
    E, N, _ = w.shape
    Y = np.zeros((R, N), np.float64)
    lib().oracle_grouped_gemm_bf16(_p(a), R, K, _p(w), E, N, _p(_c(offsets, np.int32)),
                                   int(threads), _p(Y))
    return Y


def scatter(Y, route_slot, weights, tokens=None):
    Y = _c(Y, np.float64)
    weights = _c(weights, np.float32)
    M, k = weights.shape
    N = Y.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    n = M if tok is None else len(tok)
    out = np.zeros((n, N), np.float64)
    lib().oracle_scatter(_p(Y), _p(_c(route_slot, np.int32)), _p(weights), N, k, _p(tok), n,
                         _p(out))
    return out


def forward_fp8(logits, x_bf16_bits, w_q, w_scales, k, softcap=0.0, renorm=1, block_m=16,
                tokens=None, threads=1):
    """All steps of the FP8 path; returns a dict of intermediates and the
    binary64 output rows of ``tokens`` (all tokens when None)."""
    logits = _c(logits, np.float32)
    x = _c(x_bf16_bits, np.uint16)
    w_q = _c(w_q, np.uint8)
    w_scales = _c(w_scales, np.float32)
    M, E = logits.shape
    K = x.shape[1]
    N = w_q.shape[1]
    R = M * k
    tok = None if tokens is None else _c(tokens, np.int32)
    n = M if tok is None else len(tok)
    r = dict(ids=np.zeros((M, k), np.int32), weights=np.zeros((M, k), np.float32),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             sorted_route_ids=np.zeros(R, np.int32), route_slot=np.zeros(R, np.int32),
             tile_offsets=np.zeros(E + 1, np.int32), a_q=np.zeros((R, K), np.uint8),
             a_scales=np.zeros((K // 128, R), np.float32), out=np.zeros((n, N), np.float64))
    lib().oracle_forward_fp8(_p(logits), _p(x), _p(w_q), _p(w_scales), M, K, N, E, k,
                             float(softcap), int(renorm), int(block_m), _p(tok), n, int(threads),
                             _p(r["ids"]), _p(r["weights"]), _p(r["counts"]), _p(r["offsets"]),
                             _p(r["sorted_route_ids"]), _p(r["route_slot"]),
                             _p(r["tile_offsets"]), _p(r["a_q"]), _p(r["a_scales"]),
                             _p(r["out"]))
    return r


def dense_fp8(x_bf16_bits, ids, weights, w_q, w_scales, tokens=None, threads=1):
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    w_q = _c(w_q, np.uint8)
    w_scales = _c(w_scales, np.float32)
    M, K = x.shape
    E, N, _ = w_q.shape
    k = ids.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    n = M if tok is None else len(tok)
    out = np.zeros((n, N), np.float64)
    lib().oracle_dense_fp8(_p(x), _p(ids), _p(weights), _p(w_q), _p(w_scales), M, K, N, E, k,
                           _p(tok), n, int(threads), _p(out))
    return out


def ffn_bf16(x_bf16_bits, ids, weights, w_up_bits, w_dn_bits, tokens=None, threads=1):
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    w_up = _c(w_up_bits, np.uint16)
    w_dn = _c(w_dn_bits, np.uint16)
    T, H = x.shape
    E, I2, _ = w_up.shape
    I = I2 // 2
    k = ids.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else len(tok)
    out = np.zeros((n, H), np.float64)
    lib().oracle_ffn_bf16(_p(x), _p(ids), _p(weights), _p(w_up), _p(w_dn), T, H, I, E, k,
                          _p(tok), n, int(threads), _p(out))
    return out


# ----------------------------------------------------------------- FP8 gated FFN
def swiglu_f32(g: float, u: float) -> float:
    return lib().oracle_swiglu_f32(g, u)


def swiglu_quant(gu: np.ndarray):
    """gu f32 [R, 2I] (gate columns, then up columns) -> (h_q u8 [R, I],
    h_scales f32 [I/128, R])."""
    gu = _c(gu, np.float32)
    R, I2 = gu.shape
    I = I2 // 2
    h_q = np.zeros((R, I), np.uint8)
    h_s = np.zeros((I // 128, R), np.float32)
    lib().oracle_swiglu_quant(_p(gu), R, I, _p(h_q), _p(h_s))
    return h_q, h_s


def ffn_fp8(x_bf16_bits, ids, weights, wup_q, wup_s, wdn_q, wdn_s, tokens=None, threads=1):
    """Token-major FP8 gated FFN; binary64 output rows of ``tokens`` (all when None)."""
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    wup_q = _c(wup_q, np.uint8)
    wup_s = _c(wup_s, np.float32)
    wdn_q = _c(wdn_q, np.uint8)
    wdn_s = _c(wdn_s, np.float32)
    T, H = x.shape
    E, I2, _ = wup_q.shape
    I = I2 // 2
    k = ids.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else len(tok)
    out = np.zeros((n, H), np.float64)
    lib().oracle_ffn_fp8(_p(x), _p(ids), _p(weights), _p(wup_q), _p(wup_s), _p(wdn_q), _p(wdn_s),
                         T, H, I, E, k, _p(tok), n, int(threads), _p(out))
    return out
