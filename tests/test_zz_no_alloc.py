"""softmax_rows_noalloc: the entry point for callers that cannot allocate device memory.

Callers such as an inference engine's plugin execute hook (the engine owns all
device memory) or a latency-critical loop (an allocation could synchronise the
device or fail mid-step) may not call cudaMalloc.  softmax_rows_noalloc keeps
its partials in a fixed array inside the library instead.  These tests call it
through the C ABI twice in a row -- on different inputs, so a stale scratch
would show -- and check each result against softmax_rows on the same input,
with the tolerances every softmax test here uses.  This file is collected
last on purpose.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import ABS_TOL, ROW_SUM_TOL, Guarded, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OK, INVALID, ALIAS = 0, 1, 2


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _call_noalloc(lib, xp, yp, M, N, ld):
    return lib.softmax_rows_noalloc(xp, yp, M, N, ld, _stream())


def _twice_against_softmax_rows(lib, x_host, ld, offset=0):
    """Two calls in a row (the second on a different input), each compared with
    softmax_rows on the same input and with the oracle on a few rows; the gap
    [N, ld) and the guard floats around y stay untouched."""
    M, N = x_host.shape
    inputs = [x_host, np.flip(x_host, axis=0).copy() * np.float32(0.5)]
    for k, xh in enumerate(inputs):
        xg, yg, rg = Guarded(M, ld, offset), Guarded(M, ld, offset), Guarded(M, ld, offset)
        xg.mat[:, :N].copy_(torch.from_numpy(xh))
        assert lib.softmax_rows(xg.ptr, rg.ptr, M, N, ld, _stream()) == OK
        assert _call_noalloc(lib, xg.ptr, yg.ptr, M, N, ld) == OK
        torch.cuda.synchronize()
        y, ref = yg.mat[:, :N].double(), rg.mat[:, :N].double()
        diff = (y - ref).abs().max().item()
        assert diff <= ABS_TOL, (k, diff)
        assert (y.sum(dim=1) - 1.0).abs().max().item() <= ROW_SUM_TOL
        assert yg.untouched_outside(N)
        rows = sorted({0, M // 2, M - 1})
        check_softmax(yg.mat[rows, :N].cpu().numpy(), xh[rows], f"noalloc {M}x{N} ld {ld} call {k}")


@pytest.mark.parametrize("name,M,N", [("c5", 32, 1 << 20), ("c4", 300, 4096), ("c3", 7, 40003)])
def test_noalloc_matches_softmax_rows_twice(lib, name, M, N):
    rrs.force_path("auto", "auto")
    _twice_against_softmax_rows(lib, workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N)), N)


def test_noalloc_strided_scalar_path(lib):
    """ld = N + 3: rows not 16-byte aligned, so the scalar loads; the gap is never written."""
    rrs.force_path("auto", "auto")
    M, N = 37, 9000
    _twice_against_softmax_rows(lib, workloads.matrix(workloads.WORKLOADS["c2"].with_shape(M, N)), N + 3)


def test_noalloc_takes_the_planned_kernels(lib):
    """Where softmax_rows runs the register kernel or the cluster split (no
    workspace) or the grid split (its workspace in a fixed array here), the
    no-allocation call runs the same kernel: the results are bitwise equal,
    also past the two-phase kernels' row limit, and on a second grid call
    (the fixed workspace left ready by the first)."""
    rrs.force_path("auto", "auto")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    smem = torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    for name, M, N, path in [("c2", 8192, 1024, "row_regs"), ("c3", 64, 32768, "cluster"),
                             ("c4", 200000, 36, "row_regs"), ("c5", 32, 1 << 20, "grid"),
                             ("c5", 16, 1 << 20, "grid")]:
        assert rrs.plan_softmax(M, N, N, True, sms, smem)["path_name"] == path
        x_host = workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N))
        x = torch.from_numpy(x_host).cuda()
        ref, y = torch.empty_like(x), torch.full_like(x, float("nan"))
        assert lib.softmax_rows(x.data_ptr(), ref.data_ptr(), M, N, N, _stream()) == OK
        assert _call_noalloc(lib, x.data_ptr(), y.data_ptr(), M, N, N) == OK
        torch.cuda.synchronize()
        assert torch.equal(y, ref), (name, M, N)
        rows = sorted({0, M // 2, M - 1})
        check_softmax(y[rows].cpu().numpy(), x_host[rows], f"noalloc {path} {M}x{N}")


def test_noalloc_at_the_row_limit(lib):
    """M = 131072 rows on the two-phase kernels (forced), the most the scratch
    holds (one (max, sum) pair per row)."""
    rrs.force_path("two_phase", "auto")
    M, N = 131072, 2048
    w = workloads.WORKLOADS["c2"].with_shape(M, N)
    rows = [0, 1, 4097, M // 2, M - 2, M - 1]
    x_rows = workloads.matrix(w, rows=rows)
    x = torch.empty(M, N, dtype=torch.float32, device="cuda")
    x.normal_(0.0, 2.0, generator=torch.Generator(device="cuda").manual_seed(131072))
    x[rows] = torch.from_numpy(x_rows).cuda()
    ref = torch.empty_like(x)
    for k in range(2):
        y = torch.full_like(x, float("nan"))
        assert lib.softmax_rows(x.data_ptr(), ref.data_ptr(), M, N, N, _stream()) == OK
        assert _call_noalloc(lib, x.data_ptr(), y.data_ptr(), M, N, N) == OK
        torch.cuda.synchronize()
        assert (y.double() - ref.double()).abs().max().item() <= ABS_TOL
        assert (y.double().sum(dim=1) - 1.0).abs().max().item() <= ROW_SUM_TOL
        check_softmax(y[rows].cpu().numpy(), x_rows, f"noalloc {M} x {N} call {k}")
        x.mul_(0.5)                        # the second call sees another input
        x_rows = x_rows * np.float32(0.5)
        del y
    rrs.force_path("auto", "auto")
    del x, ref
    torch.cuda.empty_cache()


def test_noalloc_in_place(lib):
    """y == x with one stride computes in place, the same result as softmax_rows out of place."""
    rrs.force_path("auto", "auto")
    for M, N in [(32, 1 << 20), (300, 4096)]:
        x_host = workloads.matrix(workloads.WORKLOADS["c4"].with_shape(M, N))
        x = torch.from_numpy(x_host).cuda()
        ref = torch.empty_like(x)
        assert lib.softmax_rows(x.data_ptr(), ref.data_ptr(), M, N, N, _stream()) == OK
        assert _call_noalloc(lib, x.data_ptr(), x.data_ptr(), M, N, N) == OK
        torch.cuda.synchronize()
        assert (x.double() - ref.double()).abs().max().item() <= ABS_TOL
        rows = [0, M // 2, M - 1]
        check_softmax(x[rows].cpu().numpy(), x_host[rows], f"noalloc in place {M}x{N}")


def test_noalloc_refusals_leave_y_untouched(lib):
    """Too many rows for the two-phase kernels (forced here; a shape that
    needs them past 131072 rows would take 68 GB) and partial overlaps are
    refused before anything is enqueued: y keeps its sentinel and
    rrs_last_error says why."""
    lib.rrs_last_error.restype = ctypes.c_char_p
    x = torch.zeros(131073, 4, device="cuda")
    y = Guarded(131073, 4)
    rrs.force_path("two_phase", "auto")
    try:
        assert _call_noalloc(lib, x.data_ptr(), y.ptr, 131073, 4, 4) == INVALID
        assert b"131072" in lib.rrs_last_error()
    finally:
        rrs.force_path("auto", "auto")
    assert _call_noalloc(lib, x.data_ptr(), y.ptr, 0, 4, 4) == OK            # nothing to do
    assert lib.rrs_last_error() == b""
    assert _call_noalloc(lib, x.data_ptr(), x.data_ptr() + 16, 4, 4, 4) == ALIAS   # y = x + 1 row
    assert b"overlap" in lib.rrs_last_error()
    assert _call_noalloc(lib, x.data_ptr(), x.data_ptr(), 4, 4, 3) == INVALID     # ld < N
    torch.cuda.synchronize()
    assert y.untouched_outside(0)
