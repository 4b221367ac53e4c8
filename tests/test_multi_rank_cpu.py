"""The bench's multi-GPU bookkeeping, run as two gloo ranks on the CPU.

Rows are independent, so N GPUs run N replicas with no data exchange; the
only cross-rank step is the timing: every rank takes the slowest rank's
time and the job's throughput counts the rows of all replicas.
"""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 20.0][rank]
        worst = bench.max_over_ranks(my_ms, world)
        value = bench.job_rows_per_s(8192, 100, world, worst)
        out.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [20.0, 20.0]
    # 2 replicas x 8192 rows x 100 steps over 20 ms
    assert all(abs(g[2] - 2 * 8192 * 100 / 0.020) < 1e-6 for g in got)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_rows_per_s(128, 10, 1, 2.0) == 128 * 10 / 0.002


def test_cpu_baseline_all_cores_splits_the_rows():
    """The all-cores oracle baseline: every row in exactly one block, one
    spawned process per block, throughput over the common timed window."""
    import bench
    import workloads
    w = workloads.WORKLOADS["c1"]
    r = bench.cpu_baseline_all_cores(w, 0.2, start_delay_s=2.0)
    assert r["kind"] == "oracle" and r["unit"] == "rows/s"
    assert 1 <= r["cores"] <= max(1, min(os.cpu_count() or 1, w.M))
    assert r["value"] > 0 and r["gbs"] > 0
