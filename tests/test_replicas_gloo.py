"""Multi-rank (replica) path of bench.py, on the CPU with the gloo backend.

The decode path shards by sequence with no data exchange, so N GPUs run N
independent replicas; the benchmark takes the slowest rank's time and the sum
of the ranks' work.  These tests run that aggregation with world_size 2 over
gloo, and check that the reference arm does its work on rank 0 only.
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


def _worker(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        # rank r pretends its K steps took (10 + 5r) ms and moved (1 + r) MB per step
        job = bench.whole_job(10.0 + 5.0 * rank, 5, (1 + rank) * 1_000_000, 32 * (1 + rank),
                              world, torch.device("cpu"))
        results[rank] = job
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_whole_job_takes_slowest_rank_and_sums_work():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        r0, r1 = results[0], results[1]
    for r in (r0, r1):  # every rank reaches the same figures
        assert r["ms_per_step"] == pytest.approx(15.0 / 5)
        assert r["total_bytes_per_step"] == 3_000_000
        t = 15.0e-3 / 5
        assert r["value_gbs"] == pytest.approx(3_000_000 / t / 1e9)
        assert r["query_heads_per_s"] == pytest.approx(96 / t)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    job = bench.whole_job(8.0, 4, 2_000_000, 64, 1, torch.device("cpu"))
    assert job["ms_per_step"] == 2.0
    assert job["value_gbs"] == pytest.approx(2_000_000 / 2e-3 / 1e9)


def test_reference_arm_works_on_rank_zero_only():
    # a non-zero rank of the reference arm exits 0 without running the oracle
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line_on_rank_zero():
    # rank 0 times the oracle on the host cores and prints the JSON line the
    # driver parses; the small workload keeps the run to a fraction of a second
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "small", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    import json
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    # value = algorithmic bytes of one step / time per step
    assert line["value"] == pytest.approx(413696 / (line["ms_per_step"] * 1e-3) / 1e9, rel=1e-6)
