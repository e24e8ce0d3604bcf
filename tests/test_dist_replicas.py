"""The N > 1 host path of bench.py on CPU: two gloo ranks (one process each, as torchrun would
start them) use its process-group set-up, barrier and max/sum reductions over ranks, and the
reference arm does its work on rank 0 only."""
import json
import os
import socket
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import importlib.util, json, os, sys, time
spec = importlib.util.spec_from_file_location("bench_rank", os.path.join(sys.argv[1], "bench.py"))
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)
import torch
world, rank, local = bench.dist_env()
bench.init_dist(world, "gloo")
cpu = torch.device("cpu")
time.sleep(0.2 * rank)            # ranks reach the barrier at different times
bench.barrier(cpu)
out = {
    "rank": rank,
    "max": bench.reduce_max(1.5 + rank, cpu),      # per-rank timing -> max over ranks
    "sum": bench.reduce_sum(10.0 * (rank + 1), cpu),  # per-rank work -> whole-job total
}
bench.barrier(cpu)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps(out))
"""


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_barrier_and_reductions():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        finally:
            if p.poll() is None:
                p.kill()
        assert p.returncode == 0, err[-2000:]
        results.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(r["rank"] for r in results) == [0, 1]
    for r in results:
        assert r["max"] == 2.5   # max(1.5, 2.5) seen by both ranks
        assert r["sum"] == 30.0  # 10 + 20 seen by both ranks


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_ref", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = types.SimpleNamespace(steps=3, warmup=3)
    # Rank 1 returns before touching the oracle or the workload (nothing to build or time).
    assert bench.run_reference(args, w=None) is None
