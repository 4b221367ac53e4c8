"""Matrices past 2^31 elements (8 GiB of fp32 each way) on every path.

Row offsets, chunk bounds and work-item indices are 64-bit in every kernel;
these cases put rows (and, for the column softmax, elements of the last
row) past element 2^31, where a 32-bit offset would wrap.  Sampled rows at
the start, on both sides of element 2^31 and at the end are set from the
seeded workload generator and compared with the float64 oracle element by
element; every row is checked on the device against properties that hold
at any size (finite, non-negative, sums to one within the row-sum
tolerance; for the row sum, the normwise bound against float64 sums).
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import ROW_SUM_TOL, SUM_TOL, check_row_sum, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LIMIT = 1 << 31


@pytest.fixture(autouse=True)
def _release():
    yield
    rrs.force_path("auto", "auto")
    rrs.force_cols_path("auto")
    torch.cuda.synchronize()
    rrs.release_workspace()
    torch.cuda.empty_cache()


def sample_rows(M: int, N: int) -> list[int]:
    """First rows, the rows around element 2^31, the last rows."""
    r = LIMIT // N
    return sorted({0, 1, r - 1, r, min(r + 1, M - 1), M - 2, M - 1})


def big_input(M: int, N: int, w: workloads.Workload, rows: list[int]):
    """x on the device: Normal(0, 3^2) from a seeded torch generator, the
    sampled rows overwritten with the workload generator's rows."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    x = torch.randn(M, N, device="cuda", generator=g).mul_(3.0)
    x_rows = workloads.matrix(w.with_shape(M, N), rows=rows)
    x[torch.tensor(rows, device="cuda")] = torch.from_numpy(x_rows).cuda()
    return x, x_rows


def check_all_rows_sum_to_one(y, where: str):
    M, N = y.shape
    step = max(1, (1 << 24) // N)
    for r0 in range(0, M, step):
        blk = y[r0:r0 + step]
        assert bool(torch.isfinite(blk).all()), f"{where}: non-finite in rows {r0}+"
        assert bool((blk >= 0).all()), f"{where}: negative in rows {r0}+"
        s = blk.double().sum(dim=1)
        err = float((s - 1.0).abs().max())
        assert err <= ROW_SUM_TOL, f"{where}: rows {r0}+ sum to one within {err:.3e}"


@pytest.mark.parametrize("path,N", [("row_regs", 4096), ("cluster", 32768), ("grid", 1 << 20),
                                    ("two_phase", 1 << 20), ("two_phase", 4096), ("two_pass", 1 << 20)])
def test_softmax_rows_past_2_31_elements(lib, path, N):
    M = LIMIT // N + 3
    assert M * N > LIMIT
    rows = sample_rows(M, N)
    x, x_rows = big_input(M, N, workloads.WORKLOADS["c4"], rows)
    rrs.force_path(path, "auto")
    plan = rrs.plan_softmax(M, N, N, True, torch.cuda.get_device_properties(0).multi_processor_count,
                            torch.cuda.get_device_properties(0).shared_memory_per_block_optin)
    assert plan["path_name"] == path
    y = torch.empty_like(x)
    rrs.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), M, N, N, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    got = y[torch.tensor(rows, device="cuda")].cpu().numpy()
    check_softmax(got, x_rows, f"{path} {M}x{N} rows {rows}")
    check_all_rows_sum_to_one(y, f"{path} {M}x{N}")


@pytest.mark.parametrize("path", ["row", "split"])
def test_row_sum_past_2_31_elements(lib, path):
    N = 4096
    M = LIMIT // N + 3
    rows = sample_rows(M, N)
    x, x_rows = big_input(M, N, workloads.WORKLOADS["c3"], rows)
    rrs.force_path("auto", path)
    out = torch.empty(M, device="cuda")
    rrs.row_sum_ptr(x.data_ptr(), out.data_ptr(), M, N, N, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    check_row_sum(out[torch.tensor(rows, device="cuda")].cpu().numpy(), x_rows, f"row sum {path}")
    step = (1 << 24) // N
    for r0 in range(0, M, step):
        blk = x[r0:r0 + step].double()
        err = (out[r0:r0 + step].double() - blk.sum(dim=1)).abs()
        assert bool((err <= SUM_TOL * blk.abs().sum(dim=1)).all()), f"row sum {path}: rows {r0}+"


@pytest.mark.parametrize("path", ["auto", "band"])
def test_softmax_cols_past_2_31_elements(lib, path):
    """4096 x 524320: the last row holds elements past 2^31, on the planner's
    path (two-pass) and on the band path.  Sampled columns are the workload
    generator's rows of the transposed shape."""
    M = 4096
    N = LIMIT // M + 32
    assert M * N > LIMIT
    cross = LIMIT - (M - 1) * N            # first column of the last row past element 2^31
    cols = sorted({0, 1, cross - 1, cross, cross + 1, N - 1})
    g = torch.Generator(device="cuda")
    g.manual_seed(4321)
    x = torch.randn(M, N, device="cuda", generator=g).mul_(3.0)
    wt = workloads.WORKLOADS["c4"].with_shape(N, M)
    xt_cols = workloads.matrix(wt, rows=cols)                  # (len(cols), M)
    x[:, torch.tensor(cols, device="cuda")] = torch.from_numpy(np.ascontiguousarray(xt_cols.T)).cuda()
    y = torch.empty_like(x)
    rrs.force_cols_path(path)
    p = rrs.plan_softmax_cols(M, N, N, True, torch.cuda.get_device_properties(0).multi_processor_count)
    assert p["path_name"] == ("two_pass" if path == "auto" else path)
    rrs.softmax_cols_ptr(x.data_ptr(), N, y.data_ptr(), N, M, N, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    got = y[:, torch.tensor(cols, device="cuda")].cpu().numpy().T   # columns as rows
    check_softmax(got, xt_cols, f"cols {M}x{N} columns {cols}")
    acc = torch.zeros(N, dtype=torch.float64, device="cuda")
    for r0 in range(0, M, 256):
        blk = y[r0:r0 + 256]
        assert bool(torch.isfinite(blk).all()) and bool((blk >= 0).all()), f"cols rows {r0}+"
        acc += blk.double().sum(dim=0)
    assert float((acc - 1.0).abs().max()) <= ROW_SUM_TOL
