"""GPU parity of softmax_rows against the float64 oracle, through the C ABI.

Small shapes run on every execution path (forced), with canary regions
around x and y, leading-dimension gaps, misaligned bases and ragged tails;
full-size workloads run on the path the planner picks (the launch the bench
times) and are compared with the oracle element by element on every row.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import Guarded, check_every_row, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PATHS = ["row_regs", "cluster", "two_phase", "row_staged", "grid", "two_pass"]

SHAPES = [(1, 1), (3, 2), (5, 3), (7, 5), (4, 31), (9, 33), (16, 128), (17, 129), (128, 256),
          (33, 1000), (8, 1024), (5, 2047), (3, 2049), (6, 4097), (4, 8191), (2, 16385),
          (3, 32768), (2, 40000), (2, 131072), (2, 300001)]


def supports(path: str, N: int, ld: int) -> bool:
    """Whether a forced path takes this shape (vector paths need ld % 4 == 0)."""
    vector_ok = ld % 4 == 0
    if path == "row_regs":
        return N <= 32768                      # scalar loads when not vector_ok
    if path == "cluster":
        return N <= 131072                     # scalar loads when not vector_ok
    if path == "row_staged":
        return vector_ok and N % 4 == 0 and N <= 32912
    if path == "grid":
        return vector_ok and N % 4 == 0
    return True


@pytest.fixture(autouse=True)
def _auto_path(lib):
    rrs.force_path("auto", "auto")
    yield
    rrs.force_path("auto", "auto")


def run(x_host: np.ndarray, N: int, ld: int, path: str = "auto", x_off: int = 0, y_off: int = 0):
    """softmax_rows through the C ABI on guarded buffers; returns (y[:, :N], guards_ok)."""
    M = x_host.shape[0]
    xb = Guarded(M, ld, x_off)
    yb = Guarded(M, ld, y_off)
    # only the M x N window is written: the ld gap keeps the NaN sentinel, so
    # a kernel that reads past N poisons its row
    xb.mat[:, :N].copy_(torch.from_numpy(np.ascontiguousarray(x_host[:, :N], dtype=np.float32)))
    rrs.force_path(path)
    rrs.softmax_rows_ptr(xb.ptr, yb.ptr, M, N, ld, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    y = yb.mat[:, :N].cpu().numpy()
    return y, yb.untouched_outside(N) and xb.untouched_outside(N)


def recipe(name: str, M: int, N: int) -> np.ndarray:
    return workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N))


@pytest.mark.parametrize("path,M,N", [(p, M, N) for M, N in SHAPES for p in PATHS if supports(p, N, N)])
def test_parity_small(path, M, N):
    name = ["c1", "c2", "c3", "c4", "c5"][(M + N) % 5]
    x = recipe(name, M, N)
    y, guards = run(x, N, N, path)
    check_softmax(y, x, f"{path} {M}x{N} {name}")
    assert guards, "wrote outside the M x N window"


@pytest.mark.parametrize("path,M,N,gap", [(p, M, N, g) for M, N, g in [(5, 1000, 4), (3, 4096, 8), (4, 32768, 4),
                                                                        (6, 257, 11)]
                                           for p in PATHS if supports(p, N, N + g)])
def test_leading_dimension_gap(path, M, N, gap):
    x = recipe("c4", M, N)
    y, guards = run(x, N, N + gap, path)
    check_softmax(y, x, f"{path} ld={N + gap}")
    assert guards


@pytest.mark.parametrize("M,N,ld,x_off,y_off", [(4, 1000, 1001, 0, 0), (3, 4096, 4096, 1, 0),
                                                (3, 4096, 4096, 0, 3), (5, 33, 35, 2, 1),
                                                (2, 40000, 40003, 1, 1), (3, 50257, 50257, 0, 0),
                                                (2, 16385, 16387, 0, 1), (2, 131072, 131073, 1, 2),
                                                (2, 131075, 131075, 0, 0), (3, 8191, 8193, 1, 3),
                                                (3, 12287, 12289, 2, 1), (2, 16384, 16385, 0, 0)])
def test_unaligned_takes_scalar_path(M, N, ld, x_off, y_off):
    """Rows whose start or stride is not 16-byte aligned: the scalar register
    kernel up to 4096, the scalar register kernel or the scalar cluster split
    up to 16384, the scalar cluster split up to 131072 (each CTA's segment in
    four-scalar slots), the scalar two-pass split beyond; the two-pass split
    forced on every shape too."""
    x = recipe("c2", M, N)
    y, guards = run(x, N, ld, "auto", x_off, y_off)
    check_softmax(y, x, f"unaligned {M}x{N} ld={ld}")
    assert guards
    want = {"row_regs"} if N <= 4096 else ({"row_regs", "cluster"} if N <= 16384 else
                                           {"cluster"} if N <= 131072 else {"two_pass"})
    assert rrs.plan_softmax(M, N, ld, False, torch.cuda.get_device_properties(0).multi_processor_count)[
        "path_name"] in want
    if N <= 32768:
        y, guards = run(x, N, ld, "row_regs", x_off, y_off)    # the scalar row kernel
        check_softmax(y, x, f"unaligned row_regs {M}x{N} ld={ld}")
        assert guards
    y, guards = run(x, N, ld, "two_pass", x_off, y_off)        # the scalar two-pass kernel
    check_softmax(y, x, f"unaligned two_pass {M}x{N} ld={ld}")
    assert guards
    if N <= 131072:
        y, guards = run(x, N, ld, "cluster", x_off, y_off)     # the scalar cluster kernel
        check_softmax(y, x, f"unaligned cluster {M}x{N} ld={ld}")
        assert guards
    else:
        with pytest.raises(rrs.RRSError) as e:
            run(x, N, ld, "cluster", x_off, y_off)
        assert e.value.status == 6


@pytest.mark.parametrize("M,N,ld", [(3, 50257, 50260), (2, 16385, 16388), (2, 131073, 131076)])
def test_ragged_long_rows_take_the_cluster_split(M, N, ld):
    """Aligned rows with N % 4 != 0 past 16384 floats: the vector cluster
    kernel with the ragged tail in its last CTA."""
    x = recipe("c4", M, N)
    assert rrs.plan_softmax(M, N, ld, True, torch.cuda.get_device_properties(0).multi_processor_count)[
        "path_name"] == "cluster"
    y, guards = run(x, N, ld, "auto")
    check_softmax(y, x, f"ragged {M}x{N} ld={ld}")
    assert guards


@pytest.mark.parametrize("path,N", [(p, N) for N in [2, 8, 1024, 5000, 40000] for p in PATHS if supports(p, N, N)])
def test_special_values(path, N):
    rng = np.random.default_rng(N)
    x = rng.normal(0, 3, size=(8, N)).astype(np.float32)
    x[0] = -np.inf                              # all masked: NaN row
    x[1, :] = 7.25                              # constant row: uniform
    x[2, 1:] = -np.inf                          # one finite entry: one-hot
    x[3, N // 2] = np.inf                       # +inf: NaN row
    x[4, N - 1] = np.nan                        # NaN: NaN row
    x[5, ::2] = -np.inf                         # half masked
    x[6] += 1000.0                              # large offset (shift invariance)
    x[7, 0] = 88.0                              # a spike near exp's fp32 range
    y, guards = run(x, N, N, path)
    check_softmax(y, x, f"{path} specials N={N}")
    assert guards
    assert np.all(y[1] == y[1][0])
    assert y[2, 0] == 1.0 and np.all(y[2, 1:] == 0.0)


@pytest.mark.parametrize("path,N", [(p, N) for N in [6, 1003, 5000, 40000, 300000] for p in PATHS
                                    if supports(p, N, N)])
def test_extreme_magnitudes_and_tail_maxima(path, N):
    """Values near fp32's limits and maxima in awkward places, on every path:
    x - m overflowing to -inf (its exp is 0, as the true value is), a row at
    3.4e38, subnormal rows, a maximum only in the ragged tail or only in the
    first column, a row of huge negative values."""
    rng = np.random.default_rng(N + 7)
    x = rng.normal(0, 3, size=(8, N)).astype(np.float32)
    x[0, ::2] = 3.0e38                          # x - m = -6e38 overflows to -inf: exactly 0
    x[0, 1::2] = -3.0e38
    x[1, :] = np.float32(3.4e38)                # the largest magnitudes, all equal: uniform
    x[2, :] = (np.arange(N) % 7 + 1).astype(np.float32) * np.float32(1e-40)   # subnormals
    x[3, N - 1] = 20.0                          # the maximum only in the last column
    x[4, 0] = 20.0                              # ... only in the first
    x[5, :] = np.float32(-1e30) + x[5]          # huge negative: the noise rounds away, uniform
    x[6, :] = -np.inf
    x[6, N // 3] = np.float32(-1e30)            # one finite entry among -inf
    x[7, :] = np.float32(2.0) ** -126           # the smallest normal, all equal
    y, guards = run(x, N, N, path)
    check_softmax(y, x, f"{path} extremes N={N}")
    assert guards
    assert np.all(y[1] == y[1][0]) and np.all(y[5] == y[5][0]) and np.all(y[7] == y[7][0])
    assert y[6, N // 3] == 1.0 and np.count_nonzero(y[6]) == 1


@pytest.mark.parametrize("path", PATHS)
def test_shift_invariance_on_gpu(path):
    N = 40000 if path in ("cluster", "grid") else 4096
    # values on a 2^-8 grid, so x + 1000 is exact in fp32 and the shift is a true shift
    x = np.round(recipe("c2", 16, N) * 256.0).astype(np.float32) / np.float32(256.0)
    xs = x + np.float32(1000.0)
    assert np.array_equal(xs - np.float32(1000.0), x)
    y0, _ = run(x, N, N, path)
    y1, _ = run(xs, N, N, path)
    check_softmax(y1, xs, "shifted")
    assert np.max(np.abs(y0.astype(np.float64) - y1)) <= 2e-6


@pytest.mark.parametrize("path", PATHS)
def test_bitwise_deterministic(path):
    N = 50000 if path in ("cluster", "grid") else 2052
    x = recipe("c3", 32, N)
    a, _ = run(x, N, N, path)
    b, _ = run(x, N, N, path)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


def test_empty_and_tensor_api():
    x = torch.randn(0, 7, device="cuda")
    assert rrs.softmax_rows(x).shape == (0, 7)
    x = torch.randn(5, 0, device="cuda")
    assert rrs.softmax_rows(x).shape == (5, 0)
    x = torch.randn(6, 100, device="cuda")
    y = rrs.softmax_rows(x)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), x.cpu().numpy(), "tensor api")
    with pytest.raises(ValueError):
        rrs.softmax_rows(x.cpu())
    with pytest.raises(ValueError):
        rrs.softmax_rows(x.double())


def test_rejects_host_memory():
    host = np.zeros((4, 64), dtype=np.float32)
    dev = torch.zeros(4, 64, device="cuda")
    with pytest.raises(rrs.RRSError) as e:
        rrs.softmax_rows_ptr(host.ctypes.data, dev.data_ptr(), 4, 64, 64, 0)
    assert e.value.status == 1
    with pytest.raises(rrs.RRSError) as e:
        rrs.softmax_rows_ptr(dev.data_ptr(), dev.data_ptr() + 64, 4, 64, 64, 0)
    assert e.value.status == 2


# Rows of more than 128 chunks of 8192 floats: the two-pass kernel's merging
# warp loads a row's (max, sum) pairs 128 at a time, so these rows take two
# or three rounds of its loads (up to the planner's 256-chunk limit, and past
# it when the path is forced).
@pytest.mark.parametrize("M,N,ld,x_off,y_off,path", [
    (2, 2_097_152, 2_097_153, 1, 2, "auto"),       # 256 chunks, unaligned: the planner's two-pass limit
    (3, 1_500_001, 1_500_001, 0, 0, "two_pass"),   # 184 chunks, a ragged last chunk, scalar form
    (2, 2_105_344, 2_105_344, 0, 0, "two_pass"),   # 257 chunks, float4 form: three rounds
])
def test_two_pass_rows_of_many_chunks(M, N, ld, x_off, y_off, path):
    x = recipe("c5", M, N)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if path == "auto":
        assert rrs.plan_softmax(M, N, ld, False, sms)["path_name"] == "two_pass"
    y, guards = run(x, N, ld, path, x_off, y_off)
    assert rrs.device_error() == 0
    check_softmax(y, x, f"two_pass {M}x{N} ld={ld}")
    assert guards


@pytest.mark.parametrize("name", ["c2", "c4"])
@pytest.mark.parametrize("path", ["auto", "cluster", "two_phase", "two_pass"])
def test_input_written_just_before_reads_back_intact(name, path):
    """x written by kernels right before the call -- its lines still dirty in
    the L2 -- is read back unchanged by a later kernel, and the softmax of it
    is right: the library's streaming loads never drop or alter x."""
    rrs.force_path(path, "auto")
    try:
        w = workloads.WORKLOADS[name]
        x_host = workloads.matrix(w)
        src = torch.from_numpy(x_host).cuda()
        x = torch.zeros_like(src)
        y = torch.empty_like(src)
        rows = [0, 7, w.M // 2, w.M - 1]
        for _ in range(3):
            x.zero_()
            x.copy_(src)             # device writes of x: dirty in the L2
            x.mul_(1.0)              # and once more
            rrs.softmax_rows(x, y)
            back = x.clone()         # a later kernel reads x
            torch.cuda.synchronize()
            assert torch.equal(back, src)
            check_softmax(y[rows].cpu().numpy(), x_host[rows], f"{name} {path} after device writes")
    finally:
        rrs.force_path("auto", "auto")


def test_two_streams_use_separate_workspaces():
    rrs.force_path("two_phase")
    xs = [recipe("c5", 4, 300000 + 17 * i) for i in range(2)]
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    dev_x = [torch.from_numpy(x).cuda() for x in xs]
    torch.cuda.synchronize()
    for _ in range(3):
        for s, dx in zip(streams, dev_x):
            with torch.cuda.stream(s):
                outs.append(rrs.softmax_rows(dx))
    torch.cuda.synchronize()
    for k, y in enumerate(outs):
        check_softmax(y.cpu().numpy(), xs[k % 2], f"stream {k % 2}")


# ------------------------------------------------------- full-size workloads --

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_full_size_workload(name):
    """Every row of each of the five workloads, on the planner's path (the
    launch the bench times), against the oracle element by element."""
    w = workloads.WORKLOADS[name]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    rrs.softmax_rows(x, y)                     # the planner's path, as the bench launches it
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check_every_row(check_softmax, y, x_host, f"{name}")
    if name == "c4":
        assert bool((y[torch.isneginf(x)] == 0).all())
        spikes = x == 50.0
        assert int(spikes.sum()) == w.M * 205
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["grid", "two_phase", "two_pass"])
def test_full_size_long_rows_on_each_split_path(path):
    """32 rows of 2^20 on every path that splits a row over CTAs, every row checked."""
    w = workloads.WORKLOADS["c5"]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    rrs.force_path(path)
    for _ in range(3):                         # repeated launches reuse the workspace
        rrs.softmax_rows(x, y)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check_every_row(check_softmax, y, x_host, f"{path} c5")
    del x, y
    torch.cuda.empty_cache()


# ------------------------------------------------------------- size limits --

def test_one_row_of_two_to_the_28():
    """A single 1 GiB row: past what a cluster or the grid holds, so the two-phase path."""
    N = 1 << 28
    w = workloads.WORKLOADS["c5"].with_shape(1, N)
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    plan = rrs.plan_softmax(1, N)
    assert plan["path_name"] == "two_phase"
    rrs.softmax_rows(x, y)
    torch.cuda.synchronize()
    want = oracle.softmax_rows(x_host)[0]
    rng = np.random.default_rng(28)
    idx = np.concatenate([[0, N - 1, N // 2], rng.integers(0, N, size=200000)])
    got = y[0, torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - want[idx])) <= 2e-6
    big = want[idx] >= 1e-30
    assert np.max(np.abs(got[big] - want[idx][big]) / want[idx][big]) <= 1e-5
    assert abs(float(y.double().sum()) - 1.0) <= 1e-5
    s = torch.empty(1, device="cuda")
    rrs.row_sum(x, s)
    rrs_sum = float(s.cpu()[0])
    assert abs(rrs_sum - float(np.sum(x_host, dtype=np.float64))) <= 1e-5 * float(np.abs(x_host).sum(dtype=np.float64))
    del x, y
    torch.cuda.empty_cache()


def test_sixteen_million_rows_of_three():
    """M = 2^24 rows of N = 3 (ld = 3: the scalar two-phase path, one thread per row chunk)."""
    M, N = 1 << 24, 3
    rng = np.random.default_rng(24)
    x_host = rng.normal(0, 2, size=(M, N)).astype(np.float32)
    x = torch.from_numpy(x_host).cuda()
    y = rrs.softmax_rows(x)
    torch.cuda.synchronize()
    rows = sorted({0, M - 1, *rng.integers(0, M, size=5000).tolist()})
    check_softmax(y[rows].cpu().numpy(), x_host[rows], "2^24 x 3 sampled rows")
    sums = y.double().sum(dim=1)
    assert float((sums - 1.0).abs().max()) <= 1e-5
    del x, y
    torch.cuda.empty_cache()
