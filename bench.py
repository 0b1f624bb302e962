#!/usr/bin/env python
"""Benchmark of the fused MoE forward on GB300.

One step = one full forward (route -> layout -> quantise/gather -> grouped
GEMM with fused weighted scatter -> bf16 finalize) over one batch of seeded
synthetic inputs resident in HBM.  Default workload: the 128-token /
256-expert FP8 shape (M=128, K=2048, N=512, E=256, top-8, softcap 30).
Metric: TFLOPS on compact routed rows (2*R*N*K per forward, R = M*top_k);
µs per forward and the fraction of the roofline are reported beside it.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                  [--config qwen_small_batch_fp8 | tiny_fp8 | skewed_large_batch_fp8 |
                            bf16_ffn | imbalance_bf16 | ffn_fp8]

The gated-FFN workloads (bf16_ffn, imbalance_bf16, ffn_fp8) count the FLOPs of
both projections, 2*R*2I*H + 2*R*H*I; ffn_fp8 is the FP8 gated FFN (h
re-quantised in 1x128 blocks between the projections).

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(token data-parallel, no collective on the data path); rank 0 prints the
aggregate.  ``--impl reference`` times the CPU oracle (the only reference
implementation this workload has) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_forward_gb300 import inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024


class L2Flush:
    """Evicts a step's data from L2 between timed steps: a 256 MiB write, then
    a 256 MiB read of a second buffer, so L2 is left holding clean lines only
    (dirty flush lines would otherwise be written back inside the next timed
    step).  The two operations are captured once in a CUDA graph, so a flush
    costs the host one graph launch: the host then stays ahead of the GPU and
    no host submission gap falls inside a timed step."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)
        self._eager()
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._eager()

    def _eager(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)

    def __call__(self):
        self.graph.replay()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)   # ~2-3 s timed: room for clock samples
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="qwen_small_batch_fp8",
                    choices=list(inputs.FP8_CONFIGS) + list(inputs.BF16_CONFIGS)
                    + list(inputs.FFN_FP8_CONFIGS))
    ap.add_argument("--routing", default=None,
                    help="gated-FFN routing: balanced | uniform | zipf1.2 | loads "
                         "(default: loads for imbalance_bf16, else uniform)")
    ap.add_argument("--rho", type=float, default=None,
                    help="max/min expert load for --routing loads (default 40)")
    ap.add_argument("--block-m", type=int, default=0)
    ap.add_argument("--k-splits", type=int, default=0)
    ap.add_argument("--sched", choices=["queue", "static"], default="queue")
    ap.add_argument("--cta-pairs", choices=["on", "off"], default="on",
                    help="grouped GEMMs on clusters of two CTAs where that form exists (on), "
                         "or single CTAs only (off)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--measure-fp8-peak", action="store_true",
                    help="measure the dense FP8 (e4m3) tensor peak with torch._scaled_mm "
                         "(cuBLASLt) on 8192^3, print one JSON line and exit")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workload facts
def workload(cfg_name, args, seed):
    if cfg_name in inputs.FP8_CONFIGS:
        d = inputs.make_fp8_inputs(cfg_name, seed=seed)
        c = d["cfg"]
        desc = (f"{cfg_name} M={c['M']} K={c['K']} N={c['N']} E={c['E']} top{c['k']} "
                f"softcap={c['softcap']:g} fp8-e4m3 128x128/1x128 blocks")
        return "fp8", d, desc
    if cfg_name in inputs.FFN_FP8_CONFIGS:
        routing = args.routing or "uniform"
        d = inputs.make_fp8_ffn_inputs(cfg_name, routing=routing, seed=seed)
        c = d["cfg"]
        desc = (f"{cfg_name} T={c['T']} H={c['H']} I={c['I']} E={c['E']} top{c['k']} "
                f"routing={routing} fp8-e4m3 gated FFN (h re-quantised 1x128)")
        return "fp8ffn", d, desc
    routing = args.routing or ("loads" if cfg_name == "imbalance_bf16" else "uniform")
    rho = args.rho if args.rho is not None else (40.0 if routing == "loads" else 1.0)
    d = inputs.make_bf16_inputs(cfg_name, routing=routing, rho=rho, seed=seed)
    c = d["cfg"]
    desc = (f"{cfg_name} T={c['T']} H={c['H']} I={c['I']} E={c['E']} top{c['k']} "
            f"routing={routing} rho={rho:g} bf16 gated FFN")
    return "bf16", d, desc


def flops_per_step(kind, c):
    if kind == "fp8":
        return 2.0 * c["M"] * c["k"] * c["N"] * c["K"]
    R = c["T"] * c["k"]
    return 2.0 * R * (2 * c["I"]) * c["H"] + 2.0 * R * c["H"] * c["I"]


def peaks():
    """Roofline denominators: HBM and bf16 from MEASURED_PEAKS.json (else the
    fallback figures); FP8 from the committed measurement of the vendor FP8
    GEMM (profiles/fp8_dense_peak.json, written from `--measure-fp8-peak`),
    else twice the bf16 burst."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        pk = dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j["bf16_tflops_sustained"],
                  src="measured")
    else:
        pk = dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")
    pk["fp8_nominal"] = 2 * pk["bf16"]
    f = os.path.join(ROOT, "profiles", "fp8_dense_peak.json")
    if os.path.exists(f):
        pk["fp8"] = json.load(open(f))["fp8_e4m3_tflops"]
        pk["fp8_src"] = "measured cuBLASLt e4m3 8192^3 burst"
    else:
        pk["fp8"] = pk["fp8_nominal"]
        pk["fp8_src"] = f"2 x {pk['src']} bf16 burst"
    return pk


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples around a timed region: one
    query when it starts, a 50 ms polling loop while it runs, and one query
    right after the last step has been enqueued (while the GPU still works
    through the queue), so even a region of a few milliseconds has a record."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.lines = []

    def _cmd(self):
        return ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                "--format=csv,noheader,nounits"]

    def sample_now(self):
        try:
            r = subprocess.run(self._cmd(), capture_output=True, text=True, timeout=10)
            self.lines += r.stdout.splitlines()
        except (FileNotFoundError, OSError, subprocess.TimeoutExpired):
            pass

    def start(self):
        self.sample_now()
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        try:
            self.proc = subprocess.Popen(self._cmd() + ["-lms", "50"], stdout=fd,
                                         stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        os.close(fd)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.path is not None:
            with open(self.path) as f:
                self.lines += f.read().splitlines()
            os.unlink(self.path)
            self.path = None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def bench_ours(args, rank, world, local):
    from mixture_experts_forward_gb300 import _lib as L
    from mixture_experts_forward_gb300 import build as moe_build
    moe_build.build()
    L.lib()
    dev = torch.device("cuda", local)
    kind, d, desc = workload(args.config, args, args.seed + rank)
    c = d["cfg"]
    sched = L.SCHED_QUEUE if args.sched == "queue" else L.SCHED_STATIC
    pairs = 0 if args.cta_pairs == "on" else -1
    if kind == "fp8":
        logits, x = d["logits"].to(dev), d["x"].to(dev)
        w, ws_ = d["w_q"].to(dev), d["w_scales"].to(dev)
        M, K, N, E, k = c["M"], c["K"], c["N"], c["E"], c["k"]
        fa = L.forward_args(dtype=L.DTYPE_FP8, M=M, K=K, N=N, E=E, top_k=k, softcap=c["softcap"],
                            logits=logits, x=x, w=w, w_scales=ws_, block_m=args.block_m,
                            sched=sched, k_splits=args.k_splits, use_graph=1, cta_pairs=pairs)
        out_cols = N
    elif kind == "fp8ffn":
        logits, x = d["logits"].to(dev), d["x"].to(dev)
        wu, wus = d["wup_q"].to(dev), d["wup_s"].to(dev)
        wd, wds = d["wdn_q"].to(dev), d["wdn_s"].to(dev)
        M, K, N, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
        fa = L.forward_args(dtype=L.DTYPE_FP8, gated=1, M=M, K=K, N=N, E=E, top_k=k, softcap=0.0,
                            logits=logits, x=x, w=wu, w_scales=wus, w2=wd, w2_scales=wds,
                            block_m=args.block_m, sched=sched, k_splits=args.k_splits,
                            use_graph=1, cta_pairs=pairs)
        out_cols = K
    else:
        logits, x = d["logits"].to(dev), d["x"].to(dev)
        w, w2 = d["w_up"].to(dev), d["w_dn"].to(dev)
        M, K, N, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
        fa = L.forward_args(dtype=L.DTYPE_BF16, M=M, K=K, N=N, E=E, top_k=k, softcap=0.0,
                            logits=logits, x=x, w=w, w2=w2, block_m=args.block_m, sched=sched,
                            use_graph=1, cta_pairs=pairs)
        out_cols = K
    ws = L.new_workspace(L.workspace_size(fa), device=dev)
    out = torch.empty(M, out_cols, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    block_m, k_splits = L.forward_plan(fa)

    for _ in range(max(3, args.warmup)):
        flush()
        L.forward(fa, out, ws)
    torch.cuda.synchronize()
    assert L.get_error(ws) == L.MOE_OK

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()                          # L2 flushed between steps (untimed)
        starts[i].record(stream)
        L.forward(fa, out, ws)
        ends[i].record(stream)
    sampler.sample_now()                 # while the GPU still drains the queued steps
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    status = L.get_error(ws)
    assert status == L.MOE_OK, L.status_string(status)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = all_max(sum(step_ms), world)
    fl = flops_per_step(kind, c)
    value = world * fl * args.steps / (total_ms * 1e-3) / 1e12
    ms_per_step = total_ms / args.steps
    # route+layout, quant/gather, GEMM(s) (the FP8 FFN's up projection carries
    # the SwiGLU + re-quantisation), finalize
    launches_per_step = {"fp8": 4, "bf16": 5, "fp8ffn": 5}[kind]

    # routing facts of this batch (for bytes and the roofline)
    ids, _ = L.route(logits, k, softcap=c.get("softcap", 0.0))
    lay = L.layout(ids, E, block_m, L.new_workspace(L.CTRL_BYTES, device=dev))
    counts = lay["counts"].cpu().numpy()
    touched = int((counts > 0).sum())
    pk = peaks()

    roof = dominant_kernel(L, kind, c, fa, d, dev, block_m, k_splits, sched, lay, ids, flush,
                           touched, pk, cfg_name=args.config, cta_pairs=pairs)
    if kind == "fp8":
        alg_bytes = touched * (N * K + (N // 128) * (K // 128) * 4) + M * E * 4 + M * K * 2 + M * N * 2
        t_roof = max(fl / (pk["fp8"] * 1e12), alg_bytes / (pk["hbm"] * 1e9))
    elif kind == "fp8ffn":
        # both projections' codes and block scales of every touched expert
        w_bytes = 3 * N * K + ((2 * N // 128) * (K // 128) + (K // 128) * (N // 128)) * 4
        alg_bytes = touched * w_bytes + M * E * 4 + M * K * 2 + M * K * 2
        t_roof = max(fl / (pk["fp8"] * 1e12), alg_bytes / (pk["hbm"] * 1e9))
    else:
        alg_bytes = touched * (2 * N * K + K * N) * 2 + M * E * 4 + M * K * 2 + M * K * 2
        t_roof = max(fl / (pk["bf16"] * 1e12), alg_bytes / (pk["hbm"] * 1e9))
    fwd_roof_frac = t_roof / (ms_per_step * 1e-3)

    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(L, fa, d, kind, dev, args, flush, fl, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(kind, d, c)

    res = {
        "metric": "fused-MoE fwd TFLOPS on compact routed rows",
        "value": round(value, 4), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_forward": round(ms_per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if kind == "bf16" else "fp8_e4m3", "data": "synthetic (seeded)",
        "config": {"workload": desc, "l2": "flushed between steps (256 MiB write, then 256 MiB read)",
                   "block_m": block_m, "k_splits": k_splits, "sched": args.sched,
                   "cta_pairs": args.cta_pairs,
                   "touched_experts": touched, "compact_rows": int(M * k),
                   "parallelism": f"replicas x{world} (token data-parallel, no collective)"},
        "forward_roofline": {"bound": "hbm" if t_roof == alg_bytes / (pk["hbm"] * 1e9) else "tensor",
                             "alg_bytes": int(alg_bytes), "roofline_us": round(t_roof * 1e6, 3),
                             "frac": round(fwd_roof_frac, 4), "peak_source": pk["src"],
                             "fp8_peak_source": pk["fp8_src"] if kind != "bf16" else None},
        "roofline": roof,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0:
        print(json.dumps(res), flush=True)


def dominant_kernel(L, kind, c, fa, d, dev, block_m, k_splits, sched, lay, ids, flush, touched, pk,
                    cfg_name="", cta_pairs=0):
    """Time the grouped GEMM alone (same inputs and tiling as the forward) with
    CUDA events on its stream and report it against its roofline."""
    stream = torch.cuda.current_stream(dev)
    ws = L.new_workspace(L.CTRL_BYTES, device=dev)
    if kind == "fp8":
        M, K, N, E, k = c["M"], c["K"], c["N"], c["E"], c["k"]
        _, wts = L.route(d["logits"].to(dev), k, softcap=c["softcap"])
        R = M * k
        # the forward's epilogue: weighted fp32 scatter-add (small batches) or
        # bf16 expert-compact rows (large batches, reduced afterwards)
        small = M * N * 4 <= (112 << 20)   # the forward's choice (fp32 accumulator on chip)
        acc = torch.zeros(M, N, dtype=torch.float32, device=dev) if small else \
            torch.zeros(R, N, dtype=torch.bfloat16, device=dev)
        a_q, a_s = L.quant_gather(d["x"].to(dev), k, lay["route_slot"],
                                  zero_acc=acc if small else None)
        w, w_s = d["w_q"].to(dev), d["w_scales"].to(dev)

        def launch():
            L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SCATTER if small else L.EPI_STORE_BF16,
                           a=a_q, a_scales=a_s, w=w,
                           w_scales=w_s, offsets=lay["offsets"], tile_offsets=lay["tile_offsets"],
                           out=acc, ws=ws, block_m=block_m, sorted_route_ids=lay["sorted_route_ids"],
                           route_weights=wts, M=M, top_k=k, sched=sched, k_splits=k_splits,
                           cta_pairs=cta_pairs)
        out_bytes = M * N * 4 if small else R * N * 2
        alg = touched * (N * K + (N // 128) * (K // 128) * 4) + R * K + (K // 128) * R * 4 + out_bytes
        fl = 2.0 * R * N * K
        name = "grouped_gemm_kernel<fp8, scatter>" if small else "grouped_gemm_kernel<fp8, store_bf16>"
        src = "grouped_gemm.cu"
    elif kind == "fp8ffn":
        # the forward's largest kernel: the FP8 up projection (gate and up
        # tiles) with the fused SwiGLU + 1x128 re-quantisation epilogue
        T, H, I, k = c["T"], c["H"], c["I"], c["k"]
        R = T * k
        a_q, a_s = L.quant_gather(d["x"].to(dev), k, lay["route_slot"])
        w, w_s = d["wup_q"].to(dev), d["wup_s"].to(dev)
        h_q = torch.empty(R, I, dtype=torch.uint8, device=dev)
        h_s = torch.empty(I // 128, R, dtype=torch.float32, device=dev)

        def launch():
            L.grouped_gemm(dtype=L.DTYPE_FP8, epilogue=L.EPI_SWIGLU, a=a_q, a_scales=a_s, w=w,
                           w_scales=w_s, offsets=lay["offsets"], tile_offsets=lay["tile_offsets"],
                           out=h_q, out_scales=h_s, ws=ws, block_m=block_m, M=T, top_k=k,
                           sched=sched, k_splits=1, cta_pairs=cta_pairs)
        alg = touched * (2 * I * H + (2 * I // 128) * (H // 128) * 4) + R * H + (H // 128) * R * 4 \
            + R * I + (I // 128) * R * 4
        fl = 2.0 * R * (2 * I) * H
        name = "grouped_gemm_kernel<fp8, swiglu>"
        src = "grouped_gemm.cu"
    else:
        # the forward's largest kernel: the gated up-projection with the SwiGLU
        # epilogue, on the expert-compact rows the sort/gather produces
        T, H, I, k = c["T"], c["H"], c["I"], c["k"]
        R = T * k
        x = d["x"].to(dev)
        a = x[(lay["sorted_route_ids"].long() // k)].contiguous()   # untimed setup
        w = d["w_up"].to(dev)
        h = torch.empty(R, I, dtype=torch.bfloat16, device=dev)

        def launch():
            L.grouped_gemm(dtype=L.DTYPE_BF16, epilogue=L.EPI_SWIGLU, a=a, w=w,
                           offsets=lay["offsets"], tile_offsets=lay["tile_offsets"], out=h,
                           ws=ws, block_m=block_m, M=T, top_k=k, sched=sched, cta_pairs=cta_pairs)
        alg = touched * (2 * I) * H * 2 + R * H * 2 + R * I * 2
        fl = 2.0 * R * (2 * I) * H
        name = "grouped_gemm_kernel<bf16, swiglu>"
        src = "grouped_gemm.cu"
    for _ in range(3):
        flush()
        launch()
    # n launches back to back (each after an L2 flush) between two events, minus
    # the same n flushes alone: the GPU never waits for the host inside the
    # measured span, so no submission latency is counted
    n = 50

    def span(with_gemm):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(n):
            flush()
            if with_gemm:
                launch()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3

    spans = [(span(True), span(False)) for _ in range(3)]
    assert L.get_error(ws) == L.MOE_OK
    avg_s = statistics.median(g - f for g, f in spans) / n
    t_hbm = alg / (pk["hbm"] * 1e9)
    fp8 = kind in ("fp8", "fp8ffn")
    t_tc = fl / ((pk["fp8"] if fp8 else pk["bf16"]) * 1e12)
    # (the committed captures are of the default build: CTA pairs on)
    traffic = stored_traffic(src, name, cfg_name) if cta_pairs == 0 else None
    if t_hbm >= t_tc:
        achieved = alg / avg_s / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": pk["hbm"], "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4),
                "traffic": traffic, "alg_bytes_per_launch": int(alg),
                "avg_launch_us": round(avg_s * 1e6, 3),
                "peak_note": f"{pk['src']} copy bandwidth (burst)"}
    achieved = fl / avg_s / 1e12
    peak = pk["fp8"] if fp8 else pk["bf16"]
    note = pk["fp8_src"] if fp8 else f"{pk['src']} bf16 burst"
    res = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
           "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
           "flops_per_launch": fl, "avg_launch_us": round(avg_s * 1e6, 3),
           "peak_note": note}
    if fp8:
        res["frac_of_nominal_2x_bf16"] = round(achieved / pk["fp8_nominal"], 4)
    return res


def code_sha(path: str) -> str:
    """Hash of a CUDA source's code: comments and whitespace removed, so that
    editing a comment does not mark a capture of the same kernel as stale."""
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def stored_traffic(src_name: str, kernel: str, config_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and the current kernel code (else null)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    j = json.load(open(p))
    src = os.path.join(ROOT, "mixture_experts_forward_gb300", "csrc", src_name)
    sha = code_sha(src)
    e = j.get(f"{kernel}@{config_name}")
    if not e or e.get("source_sha") != sha or e.get("config") != config_name:
        return None
    return e.get("dram_bytes_per_launch")


def bench_e2e(L, fa, d, kind, dev, args, flush, fl, world):
    """Same metric through moe_forward_host with pinned host buffers: the
    inputs move host -> device and the bf16 result device -> host inside every
    timed step (for small buffers the forward's kernels access the pinned
    buffers over the host link directly; otherwise staging copies)."""
    stream = torch.cuda.current_stream(dev)
    c = d["cfg"]
    if kind == "fp8":
        M, K, N = c["M"], c["K"], c["N"]
        out_cols = N
    else:
        M, K, N = c["T"], c["H"], c["I"]
        out_cols = K
    h_logits = d["logits"].contiguous().pin_memory()
    h_x = d["x"].contiguous().pin_memory()
    h_out = torch.empty(M, out_cols, dtype=torch.bfloat16).pin_memory()
    ws = L.new_workspace(L.workspace_size(fa), device=dev)
    for _ in range(3):
        L.forward_host(fa, h_logits, h_x, h_out, ws)
    torch.cuda.synchronize()
    steps = max(10, min(args.steps // 2, 5000))
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        st[i].record(stream)
        L.forward_host(fa, h_logits, h_x, h_out, ws)
        en[i].record(stream)
    torch.cuda.synchronize()
    total = all_max(sum(s.elapsed_time(e) for s, e in zip(st, en)), world)
    h2d = h_logits.numel() * 4 + h_x.numel() * 2
    d2h = h_out.numel() * 2
    return {"value": round(world * fl * steps / (total * 1e-3) / 1e12, 4), "unit": "TFLOPS",
            "us_per_forward": round(total / steps * 1e3, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ---------------------------------------------------------------- CPU oracle
def oracle_step(kind, d, c, tokens, threads):
    import oracle
    if kind == "fp8":
        oracle.forward_fp8(d["logits"].numpy(), inputs.bf16_bits(d["x"]), d["w_q"].numpy(),
                           d["w_scales"].numpy(), k=c["k"], softcap=c["softcap"], tokens=tokens,
                           threads=threads)
        return 2.0 * len(tokens) * c["k"] * c["N"] * c["K"]
    ids, w = oracle.route(d["logits"].numpy(), c["k"])
    if kind == "fp8ffn":
        oracle.ffn_fp8(inputs.bf16_bits(d["x"]), ids, w, d["wup_q"].numpy(), d["wup_s"].numpy(),
                       d["wdn_q"].numpy(), d["wdn_s"].numpy(), tokens=tokens, threads=threads)
    else:
        oracle.ffn_bf16(inputs.bf16_bits(d["x"]), ids, w, inputs.bf16_bits(d["w_up"]),
                        inputs.bf16_bits(d["w_dn"]), tokens=tokens, threads=threads)
    R = len(tokens) * c["k"]
    return 2.0 * R * 2 * c["I"] * c["H"] + 2.0 * R * c["H"] * c["I"]


def cpu_baseline(kind, d, c, budget_s=12.0):
    """The oracle as it stands, on this host's cores, over a bounded sample of
    the workload's tokens (repeated until about budget_s of CPU work)."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    M = c["M"] if kind == "fp8" else c["T"]
    n_tok = M if kind == "fp8" else 16
    tokens = np.arange(min(M, n_tok), dtype=np.int32)
    flops, t0, reps = 0.0, time.perf_counter(), 0
    while True:
        flops += oracle_step(kind, d, c, tokens, threads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= 2000:
            break
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOPS", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} oracle forwards of the first {len(tokens)} tokens "
                      f"(all routing/layout/quantisation steps, binary64 GEMM) in {dt:.1f} s"}


def bench_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    kind, d, desc = workload(args.config, args, args.seed)
    c = d["cfg"]
    threads = os.cpu_count() or 1
    M = c["M"] if kind == "fp8" else c["T"]
    tokens = np.arange(min(M, 16 if kind == "fp8" else 4), dtype=np.int32)
    for _ in range(args.warmup):
        oracle_step(kind, d, c, tokens, threads)
    fl, t0 = 0.0, time.perf_counter()
    for _ in range(args.steps):
        fl += oracle_step(kind, d, c, tokens, threads)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    sample = (f"each step: oracle forward of {len(tokens)} of {M} tokens (routing, layout and "
              f"quantisation of all tokens; binary64 GEMM for the sampled tokens' routes)")
    res = {"impl": "reference", "metric": "fused-MoE fwd TFLOPS on compact routed rows",
           "value": round(value, 6), "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
           "config": {"workload": desc},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": threads,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def measure_fp8_peak():
    """Dense E4M3 x E4M3 -> bf16 GEMM throughput of the vendor library on this
    GPU, the FP8 counterpart of the driver's bf16 measurement: 8192^3
    (2 * 8192^3 FLOPs), best of 10 single launches (burst) and the mean over
    back-to-back launches for about 4 s (sustained), CUDA events on the
    launching stream, with the clocks sampled meanwhile."""
    n = 8192
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()  # column-major
    one = torch.ones((), device=dev)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    fl = 2.0 * n ** 3
    stream = torch.cuda.current_stream()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mm()
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    sampler = ClockSampler(0)
    sampler.start()
    reps, total = 0, 0.0
    while total < 4.0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(100):
            mm()
        e1.record(stream)
        sampler.sample_now()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1) * 1e-3
        reps += 100
    clocks = sampler.stop()
    print(json.dumps({"fp8_e4m3_tflops": round(fl / best / 1e12, 1),
                      "fp8_e4m3_tflops_sustained": round(fl * reps / total / 1e12, 1),
                      "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, unit tensor scales, 8192^3: "
                             "best of 10 (burst); 100-launch batches back to back for ~4 s "
                             "(sustained); CUDA events",
                      "torch": torch.__version__, "gpu": torch.cuda.get_device_name(0),
                      "clocks": clocks}), flush=True)


def main():
    args = parse()
    if args.measure_fp8_peak:
        measure_fp8_peak()
        return
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            bench_reference(args, rank, world)
        else:
            bench_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
