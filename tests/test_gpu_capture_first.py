"""A grouped GEMM captured into the caller's own CUDA graph as the process's
first use of the library: the launch must not run the CTA-pair occupancy
query inside the capture, so it takes the single-CTA form, and the replayed
graph is still correct.  Runs in a fresh child process (the query result is
cached per process)."""
import os
import subprocess
import sys
import textwrap

import pytest

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import oracle
    from gpu_helpers import assert_close, bits
    from mixture_experts_forward_gb300 import _lib as L
    from mixture_experts_forward_gb300 import inputs

    torch.cuda.set_device(0)
    M, K, N, E, k, bm = 700, 1024, 512, 8, 3, 128      # FP8 scatter: a CTA-pair shape
    d = inputs.make_fp8_inputs(dict(M=M, K=K, N=N, E=E, k=k, softcap=0.0, zipf_bias=1.5),
                               seed=0)
    rid, rw = oracle.route(d["logits"].numpy(), k)
    lay = oracle.layout(rid, E, block_m=bm)
    a_q, a_s = oracle.quant_gather(bits(d["x"]), k, lay["route_slot"])
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = dict(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER, a=cu(a_q), a_scales=cu(a_s),
                w=d["w_q"].cuda(), w_scales=d["w_scales"].cuda(), offsets=cu(lay["offsets"]),
                tile_offsets=cu(lay["tile_offsets"]), block_m=bm,
                sorted_route_ids=cu(lay["sorted_route_ids"]), route_weights=cu(rw), M=M,
                top_k=k)
    ws = L.new_workspace(L.CTRL_BYTES)
    out = torch.zeros(M, N, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        L.grouped_gemm(out=out, ws=ws, stream=s, **args)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    ref = oracle.scatter(oracle.grouped_gemm_fp8(a_q, a_s, d["w_q"].numpy(),
                                                 d["w_scales"].numpy(), lay["offsets"]),
                         lay["route_slot"], rw)
    assert_close(out, ref, "captured first")
    # outside the capture the query runs, and a fresh launch takes the pairs
    assert L.gemm_cta_pairs() > 0
    out2 = torch.zeros(M, N, device="cuda")
    L.grouped_gemm(out=out2, ws=ws, **args)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    assert_close(out2, ref, "pairs after the capture")
    print("ok")
""")


def test_first_use_inside_a_capture_takes_single_ctas():
    ensure_built()
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
