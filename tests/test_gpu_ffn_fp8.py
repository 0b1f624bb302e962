"""GPU parity of the FP8 gated FFN through the C ABI against the oracle.

Bit-exact: the SwiGLU + 1x128 re-quantisation step on the same f32 inputs
(codes and scales; a zero code's sign is not part of the result, 0x00 and
0x80 both decode to 0).  Within the output tolerance (rel-L2 <= 5e-3,
max-abs <= 1e-2 max|ref| against the oracle's binary64 sums): the whole
forward, whose up projection accumulates in fp32 in another order than the
oracle's binary64 sum, so an h that sits on an E4M3 rounding boundary may
take the neighbouring code."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import THREADS, assert_close, bits, ensure_built, np_, sample_tokens
from mixture_experts_forward_gb300 import _lib as L
from mixture_experts_forward_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _codes_equal(got: np.ndarray, ref: np.ndarray):
    zero = (ref & 0x7F) == 0
    assert np.array_equal(got[~zero], ref[~zero])
    assert np.all((got[zero] & 0x7F) == 0)


@pytest.mark.parametrize("R,I", [(1, 128), (300, 384), (4097, 1536)])
def test_swiglu_quant_bit_exact(R, I):
    g = torch.Generator().manual_seed(R + I)
    gu = torch.randn(R, 2 * I, generator=g) * torch.exp(torch.randn(R, 1, generator=g) * 2)
    gu[0, I:I + 64] *= 1e-3                      # small codes, some subnormal
    if R > 3:
        gu[1, :128] = 0.0                        # gate 0: an all-zero block
        gu[2, I + 128:I + 256] = 0.0             # up 0 (block 1 when I > 128)
        gu[3, :64] = -100.0                      # exp overflows: signed zeros in a block
        gu[-1, :128] = -95.0                     # a whole block of signed zeros
        gu[-1, 128:192] = 95.0                   # silu(g) = g
    gu = gu.float().contiguous()
    h_q, h_s = L.swiglu_quant(gu.cuda())
    torch.cuda.synchronize()
    rq, rs = oracle.swiglu_quant(gu.numpy())
    _codes_equal(np_(h_q), rq)
    assert np.array_equal(np_(h_s).view(np.uint32), rs.view(np.uint32))


def _run_ffn_fp8(d, block_m=0, sched=L.SCHED_QUEUE, use_graph=1, gather_rows=0, cta_pairs=0):
    c = d["cfg"]
    dev = {k: d[k].cuda() for k in ("logits", "x", "wup_q", "wup_s", "wdn_q", "wdn_s")}
    args = L.forward_args(dtype=L.DTYPE_FP8, gated=1, M=c["T"], K=c["H"], N=c["I"], E=c["E"],
                          top_k=c["k"], softcap=0.0, logits=dev["logits"], x=dev["x"],
                          w=dev["wup_q"], w_scales=dev["wup_s"], w2=dev["wdn_q"],
                          w2_scales=dev["wdn_s"], block_m=block_m, sched=sched,
                          use_graph=use_graph, gather_rows=gather_rows, cta_pairs=cta_pairs)
    ws = L.new_workspace(L.workspace_size(args))
    out = torch.empty(c["T"], c["H"], dtype=torch.bfloat16, device="cuda")
    L.forward(args, out, ws)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK
    return out


def _check_ffn_fp8(d, out, n_tok, what):
    c = d["cfg"]
    ids, w = oracle.route(d["logits"].numpy(), c["k"])
    assert np.array_equal(np.sort(ids, axis=1), np.sort(d["chosen"].numpy(), axis=1))
    tok = sample_tokens(c["T"], n_tok)
    ref = oracle.ffn_fp8(bits(d["x"]), ids, w, d["wup_q"].numpy(), d["wup_s"].numpy(),
                         d["wdn_q"].numpy(), d["wdn_s"].numpy(), tokens=tok, threads=THREADS)
    assert_close(out[torch.from_numpy(tok).long().cuda()], ref, what)


@pytest.mark.parametrize("use_graph", [0, 1])
def test_forward_ffn_fp8_small_batch_all_rows(use_graph):
    """600 routes: the fused quantise + layout front end, then up -> SwiGLU
    + re-quantise -> down with the scatter-add epilogue."""
    d = inputs.make_fp8_ffn_inputs("ffn_fp8", T=200, H=256, I=256, E=8, k=3, seed=1)
    out = _run_ffn_fp8(d, use_graph=use_graph)
    _check_ffn_fp8(d, out, 10**9, f"ffn fp8 small graph={use_graph}")


@pytest.mark.parametrize("bm,gather,pairs", [(64, 0, 0), (128, 0, 0), (128, 1, 0), (128, 0, -1)])
def test_forward_ffn_fp8_large_batch_all_rows(bm, gather, pairs):
    """6000 routes (ragged expert tiles, three blocks of I): route + rank,
    quantise + gather (or token-major codes gathered by the up projection);
    at block_m 128 both projections on CTA pairs, or (pairs = -1) on single
    CTAs."""
    d = inputs.make_fp8_ffn_inputs("ffn_fp8", routing="zipf1.2", T=1500, H=512, I=384, E=16,
                                   k=4, seed=2)
    out = _run_ffn_fp8(d, block_m=bm, gather_rows=gather, cta_pairs=pairs)
    _check_ffn_fp8(d, out, 10**9, f"ffn fp8 large bm={bm} gather={gather} pairs={pairs}")


def test_forward_ffn_fp8_bf16_rows_path_sampled():
    """An fp32 accumulator of 16384 x 2048 x 4 B is above the on-chip limit:
    the down projection stores bf16 rows and a reduction applies the weights."""
    d = inputs.make_fp8_ffn_inputs("ffn_fp8", T=16384, H=2048, I=256, E=8, k=2, seed=3)
    out = _run_ffn_fp8(d)
    _check_ffn_fp8(d, out, 1024, "ffn fp8 rows path")


@pytest.mark.parametrize("routing", ["uniform", "zipf1.2"])
def test_forward_ffn_fp8_full_shape_sampled(routing):
    d = inputs.make_fp8_ffn_inputs("ffn_fp8", routing=routing, seed=0)
    out = _run_ffn_fp8(d)
    _check_ffn_fp8(d, out, 1024, f"ffn fp8 {routing}")
