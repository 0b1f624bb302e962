"""The C-ABI library loads without a GPU, exports every entry point that
include/moe.h declares, and rejects bad arguments on the host before any
CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return L.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_pipeline():
    names = declared_functions()
    for n in ("moe_route", "moe_layout", "moe_quant_gather", "moe_grouped_gemm", "moe_scatter",
              "moe_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(L.EXPORTS) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        assert L.status_string(code)


FAKE = 1 << 20  # a non-null, aligned fake device address; never dereferenced


def test_route_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.moe_route(None, 4, 8, 2, 0.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_route(P(FAKE), 4, 8, 9, 0.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(P(FAKE), 4, 2000, 2, 0.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(P(FAKE), 4, 64, 33, 0.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(P(FAKE), 0, 8, 2, 0.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_route(P(FAKE), 4, 8, 2, -1.0, 1, P(FAKE), P(FAKE), None) == L.MOE_ERR_INVALID_ARG


def test_layout_and_quant_argument_errors(lib):
    P = ctypes.c_void_p
    f = P(FAKE)
    assert lib.moe_layout(f, 4, 8, 2, 24, f, f, f, f, f, f, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_layout(f, 4, 8, 2, 16, f, f, f, f, f, None, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_layout(f, 4, 8, 2, 16, f, f, f, f, f, P(FAKE + 16), None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_quant_gather(f, 4, 200, 2, f, f, f, None, 0, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_quant_gather(P(FAKE + 4), 4, 256, 2, f, f, f, None, 0, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_gather(f, 4, 256, 2, f, f, f, f, 6, None) == L.MOE_ERR_INVALID_ARG


def _gemm(**kw):
    base = dict(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER, sched=L.SCHED_QUEUE, block_m=16, E=8,
                N=256, K=256, R=32, M=16, top_k=2, a=FAKE, a_scales=FAKE, w=FAKE, w_scales=FAKE,
                offsets=FAKE, tile_offsets=FAKE, sorted_route_ids=FAKE, route_weights=FAKE,
                out=FAKE, k_splits=0, num_ctas=0)
    base.update(kw)
    return L.GemmArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(block_m=24), L.MOE_ERR_UNSUPPORTED), (dict(block_m=256), L.MOE_ERR_UNSUPPORTED),
    (dict(K=200), L.MOE_ERR_UNSUPPORTED), (dict(N=200), L.MOE_ERR_UNSUPPORTED),
    (dict(E=2000), L.MOE_ERR_UNSUPPORTED),
    (dict(epilogue=L.EPI_SWIGLU, out_scales=None), L.MOE_ERR_INVALID_ARG),
    (dict(epilogue=L.EPI_SWIGLU, out_scales=FAKE + 2), L.MOE_ERR_INVALID_ARG),
    (dict(epilogue=L.EPI_SWIGLU, N=384, out_scales=FAKE), L.MOE_ERR_UNSUPPORTED),
    (dict(epilogue=L.EPI_SWIGLU, out_scales=FAKE, gather_rows=1), L.MOE_ERR_UNSUPPORTED),
    (dict(a=None), L.MOE_ERR_INVALID_ARG), (dict(a_scales=None), L.MOE_ERR_INVALID_ARG),
    (dict(R=33), L.MOE_ERR_INVALID_ARG), (dict(sorted_route_ids=None), L.MOE_ERR_INVALID_ARG),
    (dict(epilogue=L.EPI_STORE, k_splits=2), L.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), L.MOE_ERR_INVALID_ARG), (dict(out=FAKE + 8), L.MOE_ERR_INVALID_ARG),
    (dict(dtype=L.DTYPE_BF16, epilogue=L.EPI_SWIGLU, N=384), L.MOE_ERR_UNSUPPORTED),
    (dict(epilogue=4), L.MOE_ERR_INVALID_ARG), (dict(epilogue=-1), L.MOE_ERR_INVALID_ARG),
    (dict(epilogue=L.EPI_STORE_BF16, k_splits=2), L.MOE_ERR_UNSUPPORTED),
    (dict(cta_pairs=1), L.MOE_ERR_INVALID_ARG), (dict(cta_pairs=-2), L.MOE_ERR_INVALID_ARG),
])
def test_gemm_argument_errors(lib, kw, code):
    g = _gemm(**kw)
    assert lib.moe_grouped_gemm(ctypes.byref(g), ctypes.c_void_p(FAKE), 4096, None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(gather_rows=2), L.MOE_ERR_INVALID_ARG), (dict(gather_rows=-1), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=1, sorted_route_ids=None), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=1, epilogue=L.EPI_STORE, M=0), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=1, epilogue=L.EPI_STORE, M=15), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=1, dtype=L.DTYPE_BF16, a_scales=None, w_scales=None),
     L.MOE_ERR_UNSUPPORTED),
    (dict(gather_rows=1, dtype=L.DTYPE_BF16, epilogue=L.EPI_STORE_BF16, a_scales=None,
          w_scales=None), L.MOE_ERR_UNSUPPORTED),
])
def test_gemm_gather_rows_argument_errors(lib, kw, code):
    """Gathered rows need the route ids and R = M * top_k (slot s reads token
    row ids[s] // top_k); BF16 gathers only in the gated up projection."""
    g = _gemm(**kw)
    assert lib.moe_grouped_gemm(ctypes.byref(g), ctypes.c_void_p(FAKE), 4096, None) == code


def _fwd(**kw):
    a = L.forward_args(**kw)
    a.w = FAKE
    a.w_scales = FAKE
    a.w2 = FAKE
    a.w2_scales = FAKE
    return a


def test_forward_gather_rows_workspace(lib):
    """With gathered rows the forward keeps one token-major copy of the
    activations ([M, K] FP8 codes and [K/128, M] scales) in place of the
    expert-compact [R, K] one; BF16 reads x directly and keeps no copy.
    Small FP8 batches (the fused quantise + layout path) ignore the flag."""
    big = dict(M=4096, K=2048, N=512, E=256, top_k=8)
    M, K, R = big["M"], big["K"], big["M"] * big["top_k"]
    plain = L.workspace_size(_fwd(dtype=L.DTYPE_FP8, **big))
    gath = L.workspace_size(_fwd(dtype=L.DTYPE_FP8, gather_rows=1, **big))
    saved = (R - M) * (K + (K // 128) * 4)
    assert abs((plain - gath) - saved) <= 512          # two 256-byte alignments
    bf = dict(M=4096, K=2048, N=1024, E=64, top_k=8)
    plain = L.workspace_size(_fwd(dtype=L.DTYPE_BF16, **bf))
    gath = L.workspace_size(_fwd(dtype=L.DTYPE_BF16, gather_rows=1, **bf))
    assert abs((plain - gath) - bf["M"] * bf["top_k"] * bf["K"] * 2) <= 256
    small = dict(M=128, K=2048, N=512, E=256, top_k=8)
    assert (L.workspace_size(_fwd(dtype=L.DTYPE_FP8, gather_rows=1, **small)) ==
            L.workspace_size(_fwd(dtype=L.DTYPE_FP8, **small)))
    for bad in (2, -1):
        assert lib.moe_workspace_size(ctypes.byref(_fwd(dtype=L.DTYPE_FP8, gather_rows=bad,
                                                        **big))) == 0


def test_forward_cta_pairs_argument(lib):
    """cta_pairs is 0 (CTA pairs where that form exists) or -1 (single CTAs);
    it does not change the workspace."""
    big = dict(M=4096, K=2048, N=512, E=256, top_k=8)
    on = L.workspace_size(_fwd(dtype=L.DTYPE_FP8, **big))
    assert on > 0 and L.workspace_size(_fwd(dtype=L.DTYPE_FP8, cta_pairs=-1, **big)) == on
    for bad in (1, -2):
        assert lib.moe_workspace_size(ctypes.byref(_fwd(dtype=L.DTYPE_FP8, cta_pairs=bad,
                                                        **big))) == 0


def test_scatter_argument_errors(lib):
    P = ctypes.c_void_p
    f = P(FAKE)
    assert lib.moe_scatter(f, f, f, 4, 256, 2, f, None, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_scatter(f, f, f, 4, 256, 2, f, P(FAKE + 16), None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_scatter(None, f, f, 4, 256, 2, f, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_scatter(f, f, f, 0, 256, 2, f, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_scatter(f, f, f, 4, 256, 33, f, f, None) == L.MOE_ERR_UNSUPPORTED


def test_swiglu_quant_argument_errors(lib):
    P = ctypes.c_void_p
    f = P(FAKE)
    assert lib.moe_swiglu_quant(None, 4, 128, f, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_swiglu_quant(f, 4, 128, None, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_swiglu_quant(f, 0, 128, f, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_swiglu_quant(f, 4, 200, f, f, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_swiglu_quant(P(FAKE + 4), 4, 128, f, f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_swiglu_quant(f, 4, 128, P(FAKE + 8), f, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_swiglu_quant(f, 4, 128, f, P(FAKE + 2), None) == L.MOE_ERR_INVALID_ARG


def test_forward_fp8_gated_checks_and_workspace(lib):
    """The FP8 gated FFN needs both projections' codes and scales; its
    workspace holds h's codes [R, N] and scales (written by the up
    projection's fused SwiGLU epilogue: no f32 [R, 2N] rows), and an
    accumulator as wide as the token features K."""
    shape = dict(M=8192, K=3072, N=1536, E=16, top_k=8)
    R = shape["M"] * shape["top_k"]
    a = L.forward_args(dtype=L.DTYPE_FP8, gated=1, **shape)
    a.w = FAKE
    a.w_scales = FAKE
    assert lib.moe_workspace_size(ctypes.byref(a)) == 0          # w2 missing
    a.w2 = FAKE
    assert lib.moe_workspace_size(ctypes.byref(a)) == 0          # w2_scales missing
    a.w2_scales = FAKE
    n = L.workspace_size(a)
    K, N, M = shape["K"], shape["N"], shape["M"]
    assert n >= R * N + (N // 128) * R * 4 + R * K + M * K * 4
    assert n < R * N + (N // 128) * R * 4 + R * K + M * K * 4 + R * 2 * N * 4
    single = L.forward_args(dtype=L.DTYPE_FP8, **shape)
    single.w = FAKE
    single.w_scales = FAKE
    assert L.workspace_size(single) < n
    for bad in (2, -1):
        a.gated = bad
        assert lib.moe_workspace_size(ctypes.byref(a)) == 0
    bf = L.forward_args(dtype=L.DTYPE_BF16, gated=1, M=64, K=256, N=256, E=4, top_k=2)
    bf.w = FAKE
    bf.w2 = FAKE
    assert lib.moe_workspace_size(ctypes.byref(bf)) > 0         # BF16 is always gated


def test_forward_plan_of_the_gated_fp8_ffn(lib):
    """The plan's K split is that of the scatter-add GEMM: for the FP8 gated
    FFN the down projection, whose contraction is the intermediate size N
    (here 8 K blocks, and 20 tiles of 256 outputs: split in 2), not the single
    FP8 GEMM's K (2 K blocks: no split)."""
    def plan(**kw):
        a = _fwd(dtype=L.DTYPE_FP8, M=16, K=256, N=1024, E=8, top_k=2, **kw)
        return L.forward_plan(a)
    assert plan(gated=1) == (16, 2)
    assert plan() == (16, 1)
    assert plan(gated=1, k_splits=3) == (16, 3)
    assert plan(k_splits=3) == (16, 2)                     # capped at the 2 K blocks
    big = _fwd(dtype=L.DTYPE_FP8, gated=1, M=16384, K=2048, N=256, E=8, top_k=2)
    assert L.forward_plan(big)[1] == 1                     # bf16-rows form: one split


@pytest.mark.parametrize("kw,code", [
    (dict(block_m=24), L.MOE_ERR_UNSUPPORTED), (dict(K=200), L.MOE_ERR_UNSUPPORTED),
    (dict(E=2000), L.MOE_ERR_UNSUPPORTED), (dict(epilogue=L.EPI_SWIGLU), L.MOE_ERR_INVALID_ARG),
    (dict(a=None), L.MOE_ERR_INVALID_ARG), (dict(a_scales=None), L.MOE_ERR_INVALID_ARG),
    (dict(R=33), L.MOE_ERR_INVALID_ARG), (dict(sorted_route_ids=None), L.MOE_ERR_INVALID_ARG),
    (dict(epilogue=L.EPI_STORE, k_splits=2), L.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), L.MOE_ERR_INVALID_ARG), (dict(out=FAKE + 8), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=2), L.MOE_ERR_INVALID_ARG),
    (dict(gather_rows=1, dtype=L.DTYPE_BF16, a_scales=None, w_scales=None),
     L.MOE_ERR_UNSUPPORTED),
])
def test_gemm_noalloc_argument_errors_match(lib, kw, code):
    """The allocation-free GEMM rejects bad arguments exactly as the
    workspace entry point does, before touching its scratch or the GPU."""
    g = _gemm(**kw)
    assert lib.moe_grouped_gemm(ctypes.byref(g), ctypes.c_void_p(FAKE), 4096, None) == code
    assert lib.moe_grouped_gemm_noalloc(ctypes.byref(g), None) == code
    assert lib.moe_grouped_gemm_noalloc(None, None) == L.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(dtype=L.DTYPE_FP8, M=128, K=2048, N=512, E=256, top_k=8),           # fused quant+layout
    dict(dtype=L.DTYPE_FP8, M=4096, K=2048, N=512, E=256, top_k=8),          # route+rank path
    dict(dtype=L.DTYPE_FP8, M=4096, K=2048, N=512, E=256, top_k=8, gather_rows=1),
    dict(dtype=L.DTYPE_FP8, gated=1, M=8192, K=3072, N=1536, E=16, top_k=8),
    dict(dtype=L.DTYPE_BF16, M=8192, K=3072, N=1536, E=16, top_k=8),
    dict(dtype=L.DTYPE_BF16, M=8192, K=3072, N=1536, E=16, top_k=8, gather_rows=1),
])
def test_forward_workspace_map(lib, kw):
    """Every intermediate the map names lies inside the workspace, 256-byte
    aligned, without overlapping another; a_rows and block_m follow the
    forward's plan and gathered rows."""
    a = _fwd(**kw)
    n = L.workspace_size(a)
    m = L.workspace_map(a)
    M, K, N, E, k = kw["M"], kw["K"], kw["N"], kw["E"], kw["top_k"]
    R = M * k
    fp8 = kw["dtype"] == L.DTYPE_FP8
    gather = kw.get("gather_rows", 0) == 1 and not (fp8 and R <= 4096)
    assert m["block_m"] == L.forward_plan(a)[0]
    assert m["a_rows"] == (M if gather else R)
    sizes = dict(ids=R * 4, weights=R * 4, counts=E * 4, offsets=(E + 1) * 4,
                 tile_offsets=(E + 1) * 4, sorted_route_ids=R * 4, route_slot=R * 4)
    if m["a"] is not None:
        sizes["a"] = m["a_rows"] * K * (1 if fp8 else 2)
    if m["a_scales"] is not None:
        sizes["a_scales"] = (K // 128) * m["a_rows"] * 4
    if m["h_q"] is not None:
        sizes["h_q"] = R * N
        sizes["h_scales"] = (N // 128) * R * 4
    assert (m["a"] is None) == (not fp8 and gather)
    assert (m["a_scales"] is None) == (not fp8)
    assert (m["h_q"] is None) == (kw.get("gated", 0) != 1 or not fp8)
    spans = sorted((m[name], m[name] + sz) for name, sz in sizes.items())
    assert spans[0][0] >= L.CTRL_BYTES
    for (b0, e0), (b1, _) in zip(spans, spans[1:]):
        assert e0 <= b1
    assert spans[-1][1] <= n
    assert all(b % 256 == 0 for b, _ in spans)
    assert lib.moe_forward_workspace_map(ctypes.byref(a), None) == L.MOE_ERR_INVALID_ARG


def test_gemm_workspace_errors(lib):
    g = _gemm()
    assert lib.moe_grouped_gemm(ctypes.byref(g), None, 4096, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_grouped_gemm(ctypes.byref(g), ctypes.c_void_p(FAKE), 100, None) == L.MOE_ERR_WORKSPACE


def test_workspace_size_and_forward_errors(lib):
    a = L.forward_args(dtype=L.DTYPE_FP8, M=128, K=2048, N=512, E=256, top_k=8, softcap=30.0)
    a.w = FAKE
    a.w_scales = FAKE
    n = L.workspace_size(a)
    R = 128 * 8
    assert n >= R * 2048 + 16 * R * 4 + 128 * 512 * 4      # codes, scales, accumulator
    a2 = L.forward_args(dtype=L.DTYPE_FP8, M=256, K=2048, N=512, E=256, top_k=8)
    a2.w = FAKE
    a2.w_scales = FAKE
    assert L.workspace_size(a2) > n
    bad = L.forward_args(dtype=L.DTYPE_FP8, M=128, K=2000, N=512, E=256, top_k=8)
    bad.w = FAKE
    bad.w_scales = FAKE
    assert lib.moe_workspace_size(ctypes.byref(bad)) == 0
    a.logits = FAKE
    a.x = FAKE
    assert lib.moe_forward(ctypes.byref(a), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 16,
                           None) == L.MOE_ERR_WORKSPACE
    bf = L.forward_args(dtype=L.DTYPE_BF16, M=64, K=256, N=256, E=4, top_k=2)
    bf.w = FAKE
    assert lib.moe_workspace_size(ctypes.byref(bf)) == 0        # w2 missing
    bf.w2 = FAKE
    assert lib.moe_workspace_size(ctypes.byref(bf)) > 0


@pytest.mark.parametrize("cname,pyclass", [("moe_gemm_args", "GemmArgs"),
                                           ("moe_forward_args", "ForwardArgs"),
                                           ("moe_workspace_map", "WorkspaceMap")])
def test_argument_structs_match_the_binding(tmp_path, cname, pyclass):
    """The ctypes mirrors of the argument structs have the header's size and
    field offsets (a C program built against include/moe.h prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cls = getattr(L, pyclass)
    fields = [f[0] for f in cls._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {",
             f'  printf("size %zu\\n", sizeof({cname}));']
    lines += [f'  printf("{f} %zu\\n", offsetof({cname}, {f}));' for f in fields]
    lines += ["  return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(cls)
    for f in fields:
        assert int(out[f]) == getattr(cls, f).offset, f
