"""The benchmark's multi-rank path on the CPU: two gloo ranks.

bench.py under torchrun runs one independent replica per GPU (cache rows are
independent; nothing is exchanged on the data path), waits at a barrier on
both sides of the timed region, takes the slowest rank's time and reports the
whole job's units over it. These tests run that host logic with world size 2
on the gloo backend, and the reference arm's rank handling (rank 0 alone runs
and prints; the other ranks exit 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, dist = bench.init_ranks("gloo")
    bench.barrier(dist)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, device="cpu")   # rank 1 is slower
    bench.barrier(dist)
    out[rank] = (w, r, slowest, bench.job_rate(w, 100, slowest))
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (w, r, slowest, rate) in res.items():
        assert (w, r) == (world, rank)
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 100 / 15.0)


def test_single_process_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    w, r, dist = bench.init_ranks("gloo")
    assert (w, r, dist) == (1, 0, None)
    assert bench.max_over_ranks(3.5, dist) == 3.5
    assert bench.job_rate(1, 10, 2.0) == 5.0


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny_h2o", "--steps", "1", "--warmup", "0",
                           "--gpus", str(world)],
                          env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_on_rank_zero_only():
    other = _reference(1, 2)
    assert other.returncode == 0 and other.stdout.strip() == ""
    first = _reference(0, 2)
    assert first.returncode == 0, first.stderr
    line = json.loads(first.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
