"""The bench's multi-rank logic on CPU: two gloo ranks, no GPU.

The path shards without a data exchange (rows, key heads and prompt tiles are
independent), so several GPUs each run their own copy of the workload; the
only collective is the max of the ranks' step times.  These tests cover that
reduction, the weak-scaling aggregate, and the reference arm's rule that only
rank 0 runs and prints.
"""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        results[rank] = bench.reduce_max(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    # the result store is started by spawn, like the ranks: a fork of a threaded process can deadlock
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.25, None, None) == 3.25


def test_weak_scaling_value_counts_every_rank():
    import bench
    # 27.6 ms of roofline work per rank, 40 ms per step on the slowest rank
    one = bench.weak_scaling_value(0.0276, 40.0, 1)
    two = bench.weak_scaling_value(0.0276, 40.0, 2)
    assert one == pytest.approx(0.69)
    assert two == pytest.approx(2 * one)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """Rank 0 of the reference arm prints one JSON line with the contract's keys: the oracle's
    own cpu_baseline and an e2e that moves no bytes."""
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--parts", "decode_sliding", "--ref-budget", "0.4"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["warmup"] >= 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "decode_sliding"
