"""The N > 1 launch path on CPU: bench.py's rank helpers over world_size-2
gloo process groups, and the reference arm under torch.distributed.run (rank 0
prints the only line, the other rank exits cleanly).  The forward itself has no
collective on its data path (every rank runs an independent replica)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _needs_cpu_ranks():
    # with CUDA present bench.py takes NCCL and one GPU per rank
    import torch
    if torch.cuda.is_available() and torch.cuda.device_count() < 2:
        pytest.skip("two ranks need two GPUs here (NCCL); this test runs its ranks on CPU")


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    worst = bench.all_max(1.5 + r, w)   # each rank's "time"; the job's is the slowest
    import torch.distributed as dist
    backend = dist.get_backend()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "max": worst, "backend": backend}, f)


def test_rank_helpers_gloo_world2(tmp_path):
    _needs_cpu_ranks()
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["backend"] == "gloo"
        assert d["max"] == pytest.approx(1.5 + world - 1)   # max over ranks, seen by every rank


def test_reference_arm_under_torchrun():
    _needs_cpu_ranks()
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--config", "tiny_fp8"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
