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
