"""Host threads calling the library at once, each on its own stream.

ctypes releases the GIL during a foreign call, so these calls run inside the
library concurrently: the per-(device, stream) workspace cache, the device
table and the error words are shared state behind a mutex or atomics, and
each thread's messages are its own.  Each thread runs a different path (row
registers, cluster split in both forms, two-pass split with its
workspace, split row sum with its workspace) many times on its own buffers;
every result is then compared with the float64 oracle.
"""
from __future__ import annotations

import threading

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import check_row_sum, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# (op, workload recipe, M, N, ld, the path the planner picks)
JOBS = [("softmax", "c2", 256, 1024, 1024, "row_regs"),
        ("softmax", "c3", 8, 32768, 32768, "cluster"),
        ("softmax", "c4", 4, 140000, 140001, "two_pass"),   # unaligned past 131072: the scalar two-pass path
        ("softmax", "c2", 6, 40000, 40001, "cluster"),      # unaligned: the scalar cluster split
        ("row_sum", "c3", 8, 200000, 200000, "split"),
        ("softmax", "c4", 64, 4096, 4096, "row_regs"),
        ("row_sum", "c5", 16, 4096, 4096, "row")]


def test_host_threads_on_their_own_streams(lib):
    props = torch.cuda.get_device_properties(0)
    rrs.force_path("auto", "auto")
    inputs, outs, streams = [], [], []
    for op, name, M, N, ld, path in JOBS:
        if op == "softmax":
            plan = rrs.plan_softmax(M, N, ld, ld % 4 == 0, props.multi_processor_count,
                                    props.shared_memory_per_block_optin)
        else:
            plan = rrs.plan_row_sum(M, N, ld, ld % 4 == 0, props.multi_processor_count,
                                    props.shared_memory_per_block_optin)
        assert plan["path_name"] == path, (op, M, N, plan["path_name"])
        x_host = workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N), ld=ld)
        inputs.append((x_host, torch.from_numpy(x_host).cuda()))
        outs.append(torch.full((M, ld) if op == "softmax" else (M,), float("nan"), device="cuda"))
        streams.append(torch.cuda.Stream())
    torch.cuda.synchronize()
    start = threading.Barrier(len(JOBS))
    errors: list = []

    def work(i):
        op, _, M, N, ld, _ = JOBS[i]
        x, y, s = inputs[i][1], outs[i], streams[i].cuda_stream
        try:
            start.wait()
            for _ in range(50):
                if op == "softmax":
                    rrs.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), M, N, ld, s)
                else:
                    rrs.row_sum_ptr(x.data_ptr(), y.data_ptr(), M, N, ld, s)
        except Exception as e:   # reported below, on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(JOBS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert rrs.device_error() == 0
    for (op, name, M, N, ld, path), (x_host, _), y in zip(JOBS, inputs, outs):
        got = y.cpu().numpy()
        where = f"thread {op} {path} {M}x{N}"
        if op == "softmax":
            check_softmax(got[:, :N], x_host[:, :N], where)
            if ld > N:
                assert np.all(np.isnan(got[:, N:])), f"{where}: the ld gap was written"
        else:
            check_row_sum(got, x_host[:, :N], where)
