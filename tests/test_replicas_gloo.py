"""The multi-process side of bench.py on the CPU (gloo, world size 2): replicas are timed by
the slowest rank, the whole-job throughput counts every rank's tokens, and under torchrun the
reference arm prints exactly one line (rank 0) while every rank exits cleanly."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank: int, world: int, port: int, local_ms, results):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(local_ms[rank], world)
        bench.barrier(world)
        results[rank] = (slowest, bench.replica_throughput(8, slowest, world))
    finally:
        dist.destroy_process_group()


def test_replicas_are_timed_by_the_slowest_rank():
    world, local_ms = 2, [0.05, 0.08]
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_replica, args=(world, _free_port(), local_ms, results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        slowest, tput = got[rank]
        assert slowest == max(local_ms)
        assert tput == world * 8 / (max(local_ms) * 1e-3)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(0.07, 1) == 0.07
    assert bench.replica_throughput(8, 0.05, 1) == 8 / 0.05e-3


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"
