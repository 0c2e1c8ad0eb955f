"""The benchmark's multi-process host logic on CPU: two gloo ranks. Every
rank ends with the maximum of the ranks' timings (the job ends with its
slowest rank), the whole-job rate counts all ranks' tokens over that time,
and the reference arm does its work on rank 0 only (the others return)."""
import argparse
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([10.0 + 3 * rank, 20.0 - rank], world, "cpu")
        q.put((rank, got, bench.job_rate(8, world, got[0] / 200)))
    finally:
        dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [13.0, 20.0], (rank, got)  # rank 1's 13.0 and rank 0's 20.0
        assert rate == pytest.approx(8 * 2 / (13.0 / 200 / 1e3))


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.job_rate(8, 1, 0.5) == pytest.approx(16000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    out = io.StringIO()
    with redirect_stdout(out):
        bench.reference_arm(argparse.Namespace(workload="decode", steps=1, warmup=0))
    assert out.getvalue() == ""
