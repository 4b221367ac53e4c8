"""Failure detection on the GPU, without faulting it.

The split-row GRID path waits for the partials of other CTAs.  Every such
wait is bounded (about a second): when it runs out, the kernel records the
failure in a device error word and returns, and the host reads the status.
Here the failure is made on purpose from the host -- rrs_inject_fault makes
one CTA skip publishing a partial, a flag nothing else sets -- and the test
checks the reported status and that the context is still usable.
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import check_every_row, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIMEOUT = 4


def test_grid_wait_runs_out_and_is_reported(lib):
    path = "grid"
    M, N = 4, 65536
    x_host = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    try:
        rrs.force_path(path)
        assert rrs.device_error() == 0
        assert lib.rrs_inject_fault(1) == 0
        rrs.softmax_rows(x, y)                      # the launch itself succeeds
        assert rrs.device_error() == TIMEOUT         # ... and its waits ran out
        assert rrs.device_error() == 0               # the word was cleared
    finally:
        lib.rrs_inject_fault(0)
        rrs.force_path("auto", "auto")
    # the context is still usable and results are right again
    rrs.force_path(path)
    try:
        rrs.softmax_rows(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax(y.cpu().numpy(), x_host, "after an injected timeout")
    finally:
        rrs.force_path("auto", "auto")


def test_cols_two_pass_wait_runs_out_and_is_reported(lib):
    """COLS_TWO_PASS: the second passes wait for the first passes' column
    partials.  With item 0's partials withheld, band 0's second passes give
    up after their bounded wait and leave their rows unwritten; the status
    is reported, later calls are refused until it is collected, and the
    path is right again afterwards."""
    M, N = 1024, 256
    x_host = workloads.matrix(workloads.WORKLOADS["c4"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = torch.full_like(x, float("nan"))
    try:
        rrs.force_cols_path("two_pass")
        assert rrs.device_error() == 0
        assert lib.rrs_inject_fault(2) == 0
        rrs.softmax_cols(x, y)                      # enqueued: RRS_OK
        lib.rrs_inject_fault(0)
        torch.cuda.synchronize()
        with pytest.raises(rrs.RRSError) as e:
            rrs.softmax_cols(x, y)
        assert e.value.status == TIMEOUT
        assert rrs.device_error() == TIMEOUT
        assert rrs.device_error() == 0
        assert bool(torch.isnan(y[:, :32]).all())   # band 0 was never written
        rrs.softmax_cols(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        from gpu_helpers import check_softmax_cols
        check_softmax_cols(y.cpu().numpy(), x_host, "cols two-pass after an injected timeout")
    finally:
        lib.rrs_inject_fault(0)
        rrs.force_cols_path("auto")


def test_grid_timeout_is_refused_until_collected(lib):
    """After a GRID kernel's wait ran out (and the kernel finished), later
    calls on the device return RRS_ERR_TIMEOUT without a synchronising poll,
    until rrs_device_error collects it."""
    M, N = 4, 65536
    x_host = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    s = torch.empty(M, device="cuda")
    try:
        rrs.force_path("grid")
        assert rrs.device_error() == 0
        assert lib.rrs_inject_fault(1) == 0
        rrs.softmax_rows(x, y)                       # enqueued: RRS_OK
        lib.rrs_inject_fault(0)
        torch.cuda.synchronize()                     # the kernel gave up and finished
        for call in (lambda: rrs.softmax_rows(x, y), lambda: rrs.row_sum(x, s),
                     lambda: rrs.softmax_cols(x)):
            with pytest.raises(rrs.RRSError) as e:
                call()
            assert e.value.status == TIMEOUT
        assert lib.softmax_rows_noalloc(x.data_ptr(), y.data_ptr(), M, N, N,
                                        torch.cuda.current_stream().cuda_stream) == TIMEOUT
        assert rrs.device_error() == TIMEOUT         # collected ...
        assert rrs.device_error() == 0               # ... and cleared
        rrs.softmax_rows(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax(y.cpu().numpy(), x_host, "after a collected timeout")
    finally:
        lib.rrs_inject_fault(0)
        rrs.force_path("auto", "auto")


@pytest.mark.parametrize("held", [0.5, 0.66, 0.9])
def test_grid_runs_while_other_work_holds_sms(lib, held):
    """A fraction of the SMs held for 50 ms by CTAs of another stream whose
    shared memory leaves no room for a GRID CTA: the GRID CTAs draw their
    rows in arrival order, so a complete row group runs as soon as it fits
    (with 90 % held, not until the hold ends: the bounded waits, a second,
    outlast it) and the rest follow; the result is right (a timeout would
    have to be reported, never an incomplete y behind RRS_OK)."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    w = workloads.WORKLOADS["c5"]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    other = torch.cuda.Stream()
    try:
        rrs.force_path("auto", "auto")
        assert rrs.plan_softmax(w.M, w.N)["path_name"] == "grid"
        for trial in range(2):
            y = torch.full_like(x, float("nan"))
            torch.cuda.synchronize()
            assert lib.rrs_test_occupy(int(props.multi_processor_count * held),
                                       props.shared_memory_per_block_optin, 50_000_000,
                                       other.cuda_stream) == 0
            rrs.softmax_rows(x, y)
            torch.cuda.synchronize()
            st = rrs.device_error()
            assert st in (0, TIMEOUT), st
            if st == 0:
                check_every_row(check_softmax, y, x_host, f"c5 beside {held:.0%} held SMs, trial {trial}")
    finally:
        rrs.force_path("auto", "auto")


def test_two_grid_calls_at_once_on_two_streams(lib):
    """Two c5 calls on two streams at the same time: 304 grid CTAs for 152 SMs,
    so each launch gets only part of the GPU while the other runs.  Each CTA
    draws its row in arrival order from its own stream's workspace, so a
    complete row group of either launch always runs; both results are right."""
    w = workloads.WORKLOADS["c5"]
    xs = [workloads.matrix(w), np.flip(workloads.matrix(w), axis=1).copy()]
    dx = [torch.from_numpy(a).cuda() for a in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    try:
        rrs.force_path("auto", "auto")
        assert rrs.plan_softmax(w.M, w.N)["path_name"] == "grid"
        ys = [torch.full_like(dx[0], float("nan")) for _ in range(2)]
        torch.cuda.synchronize()
        for _ in range(3):
            for s, x, y in zip(streams, dx, ys):
                with torch.cuda.stream(s):
                    rrs.softmax_rows(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        for k in range(2):
            check_every_row(check_softmax, ys[k], xs[k], f"c5 concurrent stream {k}")
    finally:
        rrs.force_path("auto", "auto")


@pytest.mark.parametrize("held", [0.5, 0.9])
def test_cols_two_pass_runs_while_other_work_holds_sms(lib, held):
    """The column two-pass path waits only for items drawn before the waiting
    CTA (so by CTAs that run), never for co-residency: with most SMs held for
    50 ms by another stream's CTAs, it runs on the rest, never times out, and
    every column is right."""
    from gpu_helpers import check_softmax_cols
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    M, N = 4096, 8192
    x_host = workloads.matrix(workloads.WORKLOADS["c4"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    other = torch.cuda.Stream()
    rrs.force_cols_path("auto")
    assert rrs.plan_softmax_cols(M, N, sm_count=props.multi_processor_count)["path_name"] == "two_pass"
    for trial in range(2):
        y = torch.full_like(x, float("nan"))
        torch.cuda.synchronize()
        assert lib.rrs_test_occupy(int(props.multi_processor_count * held),
                                   props.shared_memory_per_block_optin, 50_000_000, other.cuda_stream) == 0
        rrs.softmax_cols(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax_cols(y.cpu().numpy(), x_host, f"cols two-pass beside {held:.0%} held SMs, trial {trial}")


def test_two_cols_two_pass_calls_at_once_on_two_streams(lib):
    """Two two-pass column calls on two streams at the same time, each with its
    own stream's workspace (arrival counter and ticketed slots): both right."""
    from gpu_helpers import check_softmax_cols
    M, N = 4096, 8192
    w = workloads.WORKLOADS["c4"].with_shape(M, N)
    xs = [workloads.matrix(w), np.flip(workloads.matrix(w), axis=0).copy() * np.float32(0.5)]
    dx = [torch.from_numpy(a).cuda() for a in xs]
    dy = [torch.full_like(d, float("nan")) for d in dx]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    rrs.force_cols_path("auto")
    for k in range(2):   # eager first calls make each stream's workspace
        rrs.softmax_cols(dx[k], dy[k], stream=streams[k])
    torch.cuda.synchronize()
    for _ in range(3):
        for k in range(2):
            rrs.softmax_cols(dx[k], dy[k], stream=streams[k])
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    for k in range(2):
        check_softmax_cols(dy[k].cpu().numpy(), xs[k], f"cols two-pass on stream {k}")


def test_rows_two_pass_wait_runs_out_and_is_reported(lib):
    """The rows' two-pass path: with item 0's pair withheld, row 0's second
    passes give up after their bounded wait and leave their chunks unwritten;
    the status is reported, later calls are refused until it is collected,
    and the path is right again afterwards."""
    M, N = 4, 100003
    x_host = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = torch.full_like(x, float("nan"))
    try:
        rrs.force_path("two_pass")
        assert rrs.device_error() == 0
        assert lib.rrs_inject_fault(2) == 0
        rrs.softmax_rows(x, y)                      # enqueued: RRS_OK
        lib.rrs_inject_fault(0)
        torch.cuda.synchronize()
        with pytest.raises(rrs.RRSError) as e:
            rrs.softmax_rows(x, y)
        assert e.value.status == TIMEOUT
        assert rrs.device_error() == TIMEOUT
        assert rrs.device_error() == 0
        assert bool(torch.isnan(y[0]).all())        # row 0 was never written
        rrs.softmax_rows(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax(y.cpu().numpy(), x_host, "rows two-pass after an injected timeout")
    finally:
        lib.rrs_inject_fault(0)
        rrs.force_path("auto", "auto")


@pytest.mark.parametrize("held", [0.5, 0.9])
def test_rows_two_pass_runs_while_other_work_holds_sms(lib, held):
    """Unaligned long rows (the two-pass path) beside another stream's CTAs
    holding most SMs for 50 ms: no timeout, every row right."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    M, N, ld = 16, 1048577, 1048579
    x_host = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(M, N))
    xb = torch.zeros(M * ld + 4, device="cuda")
    xv = xb[1:1 + M * ld].view(M, ld)
    xv[:, :N].copy_(torch.from_numpy(x_host))
    yb = torch.full((M * ld + 4,), float("nan"), device="cuda")
    yv = yb[1:1 + M * ld].view(M, ld)
    assert rrs.plan_softmax(M, N, ld, False, props.multi_processor_count)["path_name"] == "two_pass"
    other = torch.cuda.Stream()
    for trial in range(2):
        torch.cuda.synchronize()
        assert lib.rrs_test_occupy(int(props.multi_processor_count * held),
                                   props.shared_memory_per_block_optin, 50_000_000, other.cuda_stream) == 0
        rrs.softmax_rows_ptr(xv.data_ptr(), yv.data_ptr(), M, N, ld, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_every_row(check_softmax, yv[:, :N], x_host, f"rows two-pass beside {held:.0%} held SMs, trial {trial}")
