"""GPU parity of row_sum against the float64 oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import Guarded, check_row_sum

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 2), (5, 3), (7, 10), (4, 31), (9, 33), (128, 256), (33, 1000), (5, 4097),
          (3, 32768), (2, 65537), (3, 300001), (2, 1 << 20)]


@pytest.fixture(autouse=True)
def _auto_path(lib):
    rrs.force_path("auto", "auto")
    yield
    rrs.force_path("auto", "auto")


def run(x_host: np.ndarray, N: int, ld: int, path: str = "auto", x_off: int = 0):
    M = x_host.shape[0]
    xb = Guarded(M, ld, x_off)
    xb.mat[:, :N].copy_(torch.from_numpy(np.ascontiguousarray(x_host[:, :N], dtype=np.float32)))
    ob = Guarded(1, max(M, 1))
    rrs.force_path("auto", path)
    rrs.row_sum_ptr(xb.ptr, ob.ptr, M, N, ld, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = ob.mat[0, :M].cpu().numpy()
    return out, ob.untouched_outside(M) and xb.untouched_outside(N)


@pytest.mark.parametrize("path", ["row", "split"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_parity_small(path, M, N):
    x = workloads.matrix(workloads.WORKLOADS["c3"].with_shape(M, N))
    out, guards = run(x, N, N, path)
    check_row_sum(out, x, f"{path} {M}x{N}")
    assert guards


def test_worked_example_row():
    """The transcript's row 3,1,4,1,5,9,2,6,5,3 sums to 39, exactly, on every path."""
    row = np.array([[3, 1, 4, 1, 5, 9, 2, 6, 5, 3]], dtype=np.float32)
    for path in ("row", "split"):
        out, _ = run(row, 10, 10, path)
        assert out[0] == 39.0


@pytest.mark.parametrize("path", ["row", "split"])
def test_integer_rows_are_exact(path):
    N = 100000
    x = np.tile(np.arange(1, N + 1, dtype=np.float32) % 97, (3, 1))
    out, _ = run(x, N, N, path)
    assert np.array_equal(out.astype(np.int64), x.astype(np.int64).sum(axis=1))


@pytest.mark.parametrize("M,N,ld,off", [(4, 1000, 1001, 0), (3, 4096, 4096, 1), (6, 33, 40, 3)])
def test_unaligned_and_gaps(M, N, ld, off):
    x = workloads.matrix(workloads.WORKLOADS["c2"].with_shape(M, N))
    for path in ("row", "split"):
        out, guards = run(x, N, ld, path, off)
        check_row_sum(out, x, f"{path} ld={ld} off={off}")
        assert guards


def test_zero_columns_writes_zeros():
    x = np.zeros((5, 0), dtype=np.float32)
    ob = Guarded(1, 5)
    xb = Guarded(5, 1)
    rrs.row_sum_ptr(xb.ptr, ob.ptr, 5, 0, 1, 0)
    torch.cuda.synchronize()
    assert np.all(ob.mat[0].cpu().numpy() == 0.0)
    del x


@pytest.mark.parametrize("path", ["row", "split"])
def test_bitwise_deterministic(path):
    x = workloads.matrix(workloads.WORKLOADS["c3"].with_shape(16, 70001))
    a, _ = run(x, 70001, 70001, path)
    b, _ = run(x, 70001, 70001, path)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


def test_tensor_api():
    x = torch.randn(9, 333, device="cuda")
    s = rrs.row_sum(x)
    torch.cuda.synchronize()
    check_row_sum(s.cpu().numpy(), x.cpu().numpy(), "tensor api")


def test_full_size_workload():
    """Every row of the 4096 x 32768 row sum against the oracle's float64 sum."""
    w = workloads.WORKLOADS["c3"]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    out = rrs.row_sum(x)
    torch.cuda.synchronize()
    check_row_sum(out.cpu().numpy(), x_host, "c3 every row")
    del x
    torch.cuda.empty_cache()
