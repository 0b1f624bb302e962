"""The shape facts the pages print for their 128-token / 256-expert FP8
workload, checked against this repository's workload definition and the
accounting the benchmark uses (compact routed rows)."""
import json
import os

import oracle
from mixture_experts_forward_gb300 import inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden", "qwen_shape_facts.json")


def test_qwen_shape_facts():
    g = json.load(open(GOLD))
    c = inputs.FP8_CONFIGS["qwen_small_batch_fp8"]
    assert (c["M"], c["K"], c["N"], c["E"], c["k"]) == (g["M"], g["K"], g["N"], g["E"], g["top_k"])
    R = c["M"] * c["k"]                                  # compact routed rows
    assert 2 * R * c["N"] * c["K"] == g["flops"]
    assert round(g["flops"] / 1e9, 2) == g["flops_rounded_gflop"]
    assert c["K"] // g["block"] == g["k_blocks"]
    assert c["E"] * (c["N"] // g["block"]) == g["grid_ctas"]
    assert R * c["K"] == g["lhs_bytes"]                  # one E4M3 byte per element
    assert g["block"] * g["block"] * g["k_blocks"] == g["rhs_bytes_per_cta"]
    assert R // c["E"] == g["routes_per_expert"]
    assert oracle.e4m3_decode(0x7E) == g["e4m3_max"]


FULL_MLP = os.path.join(os.path.dirname(__file__), "golden", "full_mlp_flops.json")


def test_full_mlp_flops_match_the_gated_ffn_accounting():
    """The pages' full-MLP FLOP count (gate+up, SiLU, down) on the 128-token
    shape equals the gated-FFN accounting the benchmark reports
    (2*R*2I*H + 2*R*H*I on compact routed rows), and the single GEMM's count
    its FP8 accounting."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "bench", os.path.join(os.path.dirname(os.path.dirname(__file__)), "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    g = json.load(open(FULL_MLP))
    ffn = dict(T=g["M"], H=g["hidden"], I=g["intermediate"], k=g["top_k"])
    single = dict(M=g["M"], K=g["hidden"], N=g["intermediate"], k=g["top_k"])
    assert round(bench.flops_per_step("fp8ffn", ffn) / 1e9, 2) == g["full_mlp_gflop"]
    assert round(bench.flops_per_step("bf16", ffn) / 1e9, 2) == g["full_mlp_gflop"]
    assert round(bench.flops_per_step("fp8", single) / 1e9, 2) == g["single_gemm_gflop"]
    assert bench.flops_per_step("fp8ffn", ffn) == 3 * bench.flops_per_step("fp8", single)
