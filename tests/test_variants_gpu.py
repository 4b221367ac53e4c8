"""GPU parity of the variants on the softmax skeleton, through the C ABI.

* softmax_rows_ex: separate row strides for x and y, in place (y == x), and
  the log-softmax, on every execution path (forced);
* row_max and row_mean on both row-reduction paths;
* softmax_cols (softmax down each column) on both of its paths, including
  the log form, in place, separate strides and unaligned bases;
* gelu (elementwise) on ragged, unaligned and in-place vectors;
* full-size cases of each at the sizes the bench times, compared on sampled
  rows or columns plus properties of every row or column.

All comparisons are against the float64 oracle with the tolerances stated in
``gpu_helpers``.
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import (Guarded, check_every_row, check_gelu, check_log_softmax, check_row_max, check_row_mean,
                         check_softmax, check_softmax_cols)
from test_softmax_gpu import PATHS, supports

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOG = rrs.LOG_SOFTMAX


@pytest.fixture(autouse=True)
def _auto_paths(lib):
    rrs.force_path("auto", "auto")
    rrs.force_cols_path("auto")
    yield
    rrs.force_path("auto", "auto")
    rrs.force_cols_path("auto")


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def put(buf: Guarded, x_host: np.ndarray, N: int) -> None:
    buf.mat[:, :N].copy_(torch.from_numpy(np.ascontiguousarray(x_host[:, :N], dtype=np.float32)))


def run_ex(x_host, N, ldx, ldy, path="auto", flags=0, in_place=False, x_off=0, y_off=0):
    """softmax_rows_ex on guarded buffers; returns (y[:, :N], guards_ok)."""
    M = x_host.shape[0]
    xb = Guarded(M, ldx, x_off)
    put(xb, x_host, N)
    yb = xb if in_place else Guarded(M, ldy, y_off)
    rrs.force_path(path)
    rrs.softmax_rows_ex_ptr(xb.ptr, ldx, yb.ptr, ldx if in_place else ldy, M, N, flags, stream())
    torch.cuda.synchronize()
    y = yb.mat[:, :N].cpu().numpy()
    return y, yb.untouched_outside(N) and xb.untouched_outside(N)


def recipe(name, M, N):
    return workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N))


SHAPES = [(1, 1), (5, 3), (7, 33), (17, 129), (33, 1000), (5, 2047), (6, 4097), (3, 32768),
          (2, 40000), (2, 131072), (2, 300001)]


# ------------------------------------------------------------- strides ----

@pytest.mark.parametrize("path,M,N,gx,gy", [(p, M, N, gx, gy)
                                             for M, N, gx, gy in [(5, 1000, 0, 24), (4, 4096, 8, 0), (3, 40000, 4, 12),
                                                                  (6, 257, 3, 7), (2, 300000, 0, 4)]
                                             for p in PATHS if supports(p, N, N + gx) and supports(p, N, N + gy)])
def test_separate_strides(path, M, N, gx, gy):
    ldx, ldy = N + gx, N + gy
    x = recipe("c2", M, N)
    y, guards = run_ex(x, N, ldx, ldy, path)
    check_softmax(y, x, f"{path} ldx={ldx} ldy={ldy}")
    assert guards, "wrote outside the M x N window"


# ------------------------------------------------------------- in place ----

@pytest.mark.parametrize("path,M,N", [(p, M, N) for M, N in [(7, 33), (33, 1000), (6, 4097), (3, 32768), (2, 40000),
                                                              (2, 300000)]
                                      for p in PATHS if supports(p, N, N)])
def test_in_place(path, M, N):
    x = recipe("c4", M, N)
    y, guards = run_ex(x, N, N, N, path, in_place=True)
    check_softmax(y, x, f"{path} in place {M}x{N}")
    assert guards


def test_in_place_through_softmax_rows_and_tensor_api():
    x_host = recipe("c3", 64, 5000)
    x = torch.from_numpy(x_host).cuda()
    rrs.softmax_rows_ptr(x.data_ptr(), x.data_ptr(), 64, 5000, 5000, stream())
    torch.cuda.synchronize()
    check_softmax(x.cpu().numpy(), x_host, "softmax_rows in place")
    x = torch.from_numpy(x_host).cuda()
    y = rrs.softmax_rows(x, x)
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr()
    check_softmax(x.cpu().numpy(), x_host, "tensor api in place")


# ---------------------------------------------------------- log-softmax ----

@pytest.mark.parametrize("path,M,N", [(p, M, N) for M, N in SHAPES for p in PATHS if supports(p, N, N)])
def test_log_softmax_small(path, M, N):
    name = ["c1", "c2", "c3", "c4", "c5"][(M + N) % 5]
    x = recipe(name, M, N)
    if path == "row_staged":
        with pytest.raises(rrs.RRSError) as e:
            run_ex(x, N, N, N, path, LOG)
        assert e.value.status == 6
        return
    y, guards = run_ex(x, N, N, N, path, LOG)
    check_log_softmax(y, x, f"{path} log {M}x{N} {name}")
    assert guards


@pytest.mark.parametrize("path,N", [(p, N) for N in [2, 8, 1024, 5000, 40000]
                                    for p in ["row_regs", "cluster", "two_phase", "grid", "two_pass"] if supports(p, N, N)])
def test_log_softmax_special_values(path, N):
    rng = np.random.default_rng(N + 7)
    x = rng.normal(0, 3, size=(8, N)).astype(np.float32)
    x[0] = -np.inf
    x[1, :] = 7.25
    x[2, 1:] = -np.inf
    x[3, N // 2] = np.inf
    x[4, N - 1] = np.nan
    x[5, ::2] = -np.inf
    x[6] += 1000.0
    x[7, 0] = 88.0
    y, guards = run_ex(x, N, N, N, path, LOG)
    check_log_softmax(y, x, f"{path} log specials N={N}")
    assert guards
    assert y[2, 0] == 0.0 and np.all(np.isneginf(y[2, 1:]))


def test_log_softmax_unaligned_and_tensor_api():
    x_host = recipe("c4", 5, 3001)
    y, guards = run_ex(x_host, 3001, 3003, 3005, "auto", LOG, x_off=1, y_off=2)
    check_log_softmax(y, x_host, "log unaligned")
    assert guards
    x = torch.from_numpy(recipe("c2", 9, 700)).cuda()
    ly = rrs.log_softmax_rows(x)
    torch.cuda.synchronize()
    check_log_softmax(ly.cpu().numpy(), x.cpu().numpy(), "log tensor api")


# ---------------------------------------------------------- row max / mean ----

def run_reduce(fn, x_host, N, ld, path, x_off=0):
    M = x_host.shape[0]
    xb = Guarded(M, ld, x_off)
    put(xb, x_host, N)
    ob = Guarded(1, max(M, 1))
    rrs.force_path("auto", path)
    fn(xb.ptr, ob.ptr, M, N, ld, stream())
    torch.cuda.synchronize()
    return ob.mat[0, :M].cpu().numpy(), ob.untouched_outside(M) and xb.untouched_outside(N)


RED_SHAPES = [(1, 1), (3, 2), (7, 10), (9, 33), (128, 256), (33, 1000), (5, 4097), (3, 32768),
              (2, 65537), (3, 300001)]


@pytest.mark.parametrize("path", ["row", "split"])
@pytest.mark.parametrize("M,N", RED_SHAPES)
def test_row_max_and_mean(path, M, N):
    x = recipe("c4", M, N)
    got, guards = run_reduce(rrs.row_max_ptr, x, N, N, path)
    check_row_max(got, x, f"max {path} {M}x{N}")
    assert guards
    x = recipe("c3", M, N)
    got, guards = run_reduce(rrs.row_mean_ptr, x, N, N, path)
    check_row_mean(got, x, f"mean {path} {M}x{N}")
    assert guards


@pytest.mark.parametrize("path", ["row", "split"])
def test_row_max_specials_gaps_and_unaligned(path):
    N = 5000
    rng = np.random.default_rng(31)
    x = rng.normal(0, 2, size=(6, N)).astype(np.float32)
    x[0] = -np.inf
    x[1, 17] = np.nan
    x[2, N - 1] = np.inf
    x[3, :] = -3.5
    x[4, 4999] = 1e30
    got, guards = run_reduce(rrs.row_max_ptr, x, N, N + 3, path, x_off=1)
    check_row_max(got, x, f"max specials {path}")
    assert guards
    got, _ = run_reduce(rrs.row_mean_ptr, np.nan_to_num(x, neginf=0.0, posinf=0.0), N, N + 3,
                        path, x_off=1)
    check_row_mean(got, np.nan_to_num(x, neginf=0.0, posinf=0.0), f"mean unaligned {path}")


def test_empty_rows_fill_identities():
    out = torch.full((5,), 3.0, device="cuda")
    x = torch.empty(5, 0, device="cuda")
    rrs.row_max(x, out)
    torch.cuda.synchronize()
    assert bool(torch.isneginf(out).all())
    rrs.row_mean(x, out)
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all())
    rrs.row_sum(x, out)
    torch.cuda.synchronize()
    assert bool((out == 0).all())


# ---------------------------------------------------------- column softmax ----

def run_cols(x_host, N, ldx, ldy, path="auto", flags=0, in_place=False, x_off=0, y_off=0):
    M = x_host.shape[0]
    xb = Guarded(M, ldx, x_off)
    put(xb, x_host, N)
    yb = xb if in_place else Guarded(M, ldy, y_off)
    rrs.force_cols_path(path)
    rrs.softmax_cols_ptr(xb.ptr, ldx, yb.ptr, ldx if in_place else ldy, M, N, flags, stream())
    torch.cuda.synchronize()
    y = yb.mat[:, :N].cpu().numpy()
    return y, yb.untouched_outside(N) and xb.untouched_outside(N)


COL_SHAPES = [(1, 1), (2, 5), (7, 3), (8, 128), (9, 129), (64, 250), (100, 33), (129, 512),
              (1024, 300), (2047, 64), (2048, 131), (2049, 130), (5000, 40), (8192, 37),
              (8193, 20), (20000, 36)]


# the cluster path holds at most 8192 rows of a column
@pytest.mark.parametrize("path,M,N", [(p, M, N) for M, N in COL_SHAPES
                                      for p in ["cluster", "band", "two_phase", "two_pass"]
                                      if not (p == "cluster" and M > 8192)])
def test_cols_parity(path, M, N):
    x = recipe(["c2", "c4", "c3"][(M + N) % 3], M, N)
    ld = N if path == "two_phase" else -(-N // 4) * 4   # the other paths want ld % 4 == 0
    y, guards = run_cols(x, N, ld, ld, path)
    check_softmax_cols(y, x, f"cols {path} {M}x{N}")
    assert guards
    y, guards = run_cols(x, N, ld, ld, path, LOG)
    check_softmax_cols(y, x, f"cols log {path} {M}x{N}", log=True)
    assert guards


@pytest.mark.parametrize("path", ["cluster", "band", "two_phase", "two_pass"])
def test_cols_strides_in_place_and_specials(path):
    M, N = 300, 260
    rng = np.random.default_rng(32)
    x = rng.normal(0, 3, size=(M, N)).astype(np.float32)
    x[:, 0] = -np.inf                       # all-masked column: NaN
    x[:, 1] = 2.5                           # constant column: 1/M
    x[5, 2] = np.nan                        # NaN column
    x[::3, 3] = -np.inf                     # partly masked column
    x[:, 4] += 1000.0
    y, guards = run_cols(x, N, N + 4, N + 12, path)
    check_softmax_cols(y, x, f"cols strides {path}")
    assert guards
    assert np.all(y[:, 1] == y[0, 1])
    y, guards = run_cols(x, N, N + 8, N + 8, path, in_place=True)
    check_softmax_cols(y, x, f"cols in place {path}")
    assert guards


# Grids of many waves (at least nine CTAs per SM) on the band kernel: every
# column of such shapes, with a partial last batch of rows and a ragged last
# band.
@pytest.mark.parametrize("M,N", [(100, 44002), (1500, 11000)])
def test_cols_band_many_waves(M, N):
    ld = -(-N // 4) * 4
    rrs.force_cols_path("band")
    try:
        p = rrs.plan_softmax_cols(M, N, ld, sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
    finally:
        rrs.force_cols_path("auto")
    assert p["path_name"] == "band" and p["vec"] == 4 and p["grid"] >= 9 * torch.cuda.get_device_properties(0).multi_processor_count
    x = recipe("c4", M, N)
    for flags, log in ((0, False), (LOG, True)):
        y, guards = run_cols(x, N, ld, ld, "band", flags)
        check_softmax_cols(y, x, f"cols band many waves {M}x{N} log={log}", log=log)
        assert guards


def test_cols_unaligned_takes_the_scalar_paths():
    """x and y not 16-byte aligned, strides not multiples of 4: the planner's
    choice (the two-pass path's scalar form) and both scalar paths forced are
    right, in the log form too; the float4-only paths refuse."""
    x = recipe("c2", 77, 301)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rrs.plan_softmax_cols(77, 301, 305, vector_ok=False, sm_count=sms)["path_name"] == "two_pass"
    for path in ("auto", "two_pass", "two_phase"):
        for flags, log in ((0, False), (LOG, True)):
            y, guards = run_cols(x, 301, 303, 305, path, flags, x_off=1, y_off=3)
            check_softmax_cols(y, x, f"cols unaligned {path} log={log}", log=log)
            assert guards
    for path in ("cluster", "band"):
        with pytest.raises(rrs.RRSError) as e:
            run_cols(x, 301, 303, 305, path, x_off=1, y_off=3)
        assert e.value.status == 6


# Unaligned shapes on the scalar two-pass path with items enough to
# interleave, every column against the oracle, and in place.
@pytest.mark.parametrize("M,N,ld,off", [(4096, 4100, 4101, 1), (2048, 9001, 9003, 3)])
def test_cols_two_pass_scalar_form(M, N, ld, off):
    x = recipe("c4", M, N)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rrs.plan_softmax_cols(M, N, ld, vector_ok=False, sm_count=sms)["path_name"] == "two_pass"
    y, guards = run_cols(x, N, ld, ld, "auto", x_off=off, y_off=off)
    check_softmax_cols(y, x, f"cols scalar two-pass {M}x{N} ld={ld}")
    assert guards
    y, guards = run_cols(x, N, ld, ld, "auto", in_place=True, x_off=off)
    check_softmax_cols(y, x, f"cols scalar two-pass in place {M}x{N}")
    assert guards
    assert rrs.device_error() == 0


# The planner's boundary between the band and the two-pass paths: at least
# 912 items (slices of 512 rows x bands of 32 columns, twice the lag of
# 3 x 152) and at most 8 slices per band take the two-pass path.  Each side
# of both limits runs on the planner's choice, every column checked.
@pytest.mark.parametrize("M,N,path", [(4096, 3648, "two_pass"), (4096, 3616, "band"),
                                      (4097, 16384, "band"), (4096, 16388, "two_pass")])
def test_cols_auto_path_at_the_planner_boundary(M, N, path):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("the boundary shapes are laid out for 152 SMs")
    ld = -(-N // 4) * 4
    assert rrs.plan_softmax_cols(M, N, ld, sm_count=sms)["path_name"] == path
    x = recipe("c3", M, N)
    y, guards = run_cols(x, N, ld, ld, "auto")
    check_softmax_cols(y, x, f"cols auto {path} {M}x{N}")
    assert guards
    assert rrs.device_error() == 0


# Shapes with more items per pass than the lag, so that first and second
# passes interleave in one launch (and, with 20000 rows, 40 slices per band
# take five rounds of the merge's eight-slice polls); every column is
# compared with the oracle, in place too.
@pytest.mark.parametrize("M,N", [(2048, 5100), (20000, 1000), (600, 40000)])
def test_cols_two_pass_interleaved(M, N):
    ld = -(-N // 4) * 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rrs.force_cols_path("two_pass")
    try:
        p = rrs.plan_softmax_cols(M, N, ld, sm_count=sms)
    finally:
        rrs.force_cols_path("auto")
    bands = -(-N // 32)
    assert p["path_name"] == "two_pass" and p["stages"] < bands * p["ctas_per_row"]
    x = recipe("c4", M, N)
    for flags, log in ((0, False), (LOG, True)):
        y, guards = run_cols(x, N, ld, ld, "two_pass", flags)
        check_softmax_cols(y, x, f"cols two-pass {M}x{N} log={log}", log=log)
        assert guards
    y, guards = run_cols(x, N, ld, ld, "two_pass", in_place=True)
    check_softmax_cols(y, x, f"cols two-pass in place {M}x{N}")
    assert guards
    assert rrs.device_error() == 0


# ------------------------------------------------------- full-size variants ----

def sampled(n: int, seed: int, k: int = 12) -> list[int]:
    rng = np.random.default_rng(seed + 2000)
    idx = {0, n - 1, n // 2}
    idx.update(rng.choice(n, size=min(n, k), replace=False).tolist())
    return sorted(idx)


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_full_size_log_softmax(name):
    w = workloads.WORKLOADS[name]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    y = rrs.log_softmax_rows(x)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check_every_row(check_log_softmax, y, x_host, f"{name} log")
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,name", [(1024, 8192, "c2"), (4096, 16384, "c4")])
def test_full_size_columns(M, N, name):
    x_host = workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = rrs.softmax_cols(x)
    torch.cuda.synchronize()
    step = max(1, (1 << 23) // M)             # every column, a block of columns at a time
    for c0 in range(0, N, step):
        c1 = min(N, c0 + step)
        check_softmax_cols(y[:, c0:c1].cpu().numpy(), x_host[:, c0:c1], f"columns {M}x{N}, {c0}-{c1}")
    if name == "c4":
        assert bool((y[torch.isneginf(x)] == 0).all())
    del x, y
    torch.cuda.empty_cache()


def test_full_size_row_max_and_mean():
    w = workloads.WORKLOADS["c3"]
    x_host = workloads.matrix(w)
    x = torch.from_numpy(x_host).cuda()
    mx = rrs.row_max(x).cpu().numpy()
    mean = rrs.row_mean(x).cpu().numpy()
    check_row_max(mx, x_host, "c3 max, every row")                    # bit-exact
    check_row_mean(mean, x_host, "c3 mean, every row")
    del x
    torch.cuda.empty_cache()



# ------------------------------------------------------------------- GeLU ----

@pytest.mark.parametrize("n,off_x,off_y", [(1, 0, 0), (3, 0, 0), (4, 0, 0), (5, 1, 0), (1023, 0, 2),
                                           (4097, 3, 3), ((1 << 20) + 3, 0, 0), (1 << 22, 0, 0)])
def test_gelu_parity(n, off_x, off_y):
    rng = np.random.default_rng(n)
    x = rng.normal(0, 3, size=n).astype(np.float32)
    xb = Guarded(1, n, off_x)
    yb = Guarded(1, n, off_y)
    xb.mat[0].copy_(torch.from_numpy(x))
    rrs.gelu_ptr(xb.ptr, yb.ptr, n, stream())
    torch.cuda.synchronize()
    check_gelu(yb.mat[0].cpu().numpy(), x, f"gelu n={n}")
    assert yb.untouched_outside(n) and xb.untouched_outside(n)


def test_gelu_specials_and_in_place():
    x = np.array([0.0, -0.0, 1.0, -1.0, 1e-30, -1e-30, 5.0, -5.0, 9.0, -9.0, 20.0, -20.0, 1e20,
                  -1e20, np.inf, -np.inf, np.nan, 3.4e38, -3.4e38, 1e-45], dtype=np.float32)
    t = torch.from_numpy(x).cuda()
    rrs.gelu(t, t)
    torch.cuda.synchronize()
    got = t.cpu().numpy()
    check_gelu(got, x, "gelu specials in place")
    assert got[0] == 0.0 and got[14] == np.inf and np.isnan(got[15]) and np.isnan(got[16])


def test_full_size_gelu():
    n = 16384 * 16384
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn(n, device="cuda", generator=g)
    y = rrs.gelu(x)
    torch.cuda.synchronize()
    idx = torch.randint(0, n, (200000,), device="cuda", generator=g)
    idx[:3] = torch.tensor([0, n // 2, n - 1], device="cuda")
    check_gelu(y[idx].cpu().numpy(), x[idx].cpu().numpy(), "gelu 2^28 sampled")
    # every element: gelu(x) - gelu(-x) == x, the reflection the oracle is pinned by,
    # within the two outputs' error bounds (|a| <= 13 for |x| <= 6.5)
    y2 = rrs.gelu(-x)
    torch.cuda.synchronize()
    assert float(x.abs().max()) <= 6.5
    resid = (y.double() - y2.double() - x.double()).abs()
    assert bool((resid <= 3e-5 * x.double().abs() + 1e-30).all())
    del x, y, y2, idx, resid
    torch.cuda.empty_cache()


# ------------------------------------------- the scalar cluster split ----

@pytest.mark.parametrize("N,ldx,ldy,x_off,y_off", [(20000, 20001, 20003, 1, 2), (50257, 50257, 50260, 0, 0),
                                                   (131071, 131073, 131071, 3, 0)])
def test_scalar_cluster_specials_log_and_in_place(N, ldx, ldy, x_off, y_off):
    """Long rows with unaligned starts or strides on the cluster split's
    scalar form: special values, the log form, separate strides and in
    place (same stride), every row against the oracle."""
    rng = np.random.default_rng(N)
    x = rng.normal(0, 3, size=(8, N)).astype(np.float32)
    x[0] = -np.inf
    x[1, :] = 7.25
    x[2, 1:] = -np.inf
    x[3, N // 2] = np.inf
    x[4, N - 1] = np.nan
    x[5, ::2] = -np.inf
    x[6] += 1000.0
    x[7, N - 1] = 88.0                         # the row's maximum in the last CTA's last column
    for flags, check in ((0, check_softmax), (LOG, check_log_softmax)):
        y, guards = run_ex(x, N, ldx, ldy, "cluster", flags, x_off=x_off, y_off=y_off)
        check(y, x, f"scalar cluster N={N} flags={flags}")
        assert guards
    y, guards = run_ex(x, N, ldx, ldx, "cluster", 0, in_place=True, x_off=x_off)
    check_softmax(y, x, f"scalar cluster in place N={N}")
    assert guards


@pytest.mark.parametrize("N,pad,off", [(16385, 1, 0), (50257, 0, 1), (50257, 2, 3), (100003, 1, 2),
                                       (131069, 0, 0)])
def test_shifted_window_cluster(N, pad, off):
    """Rows that are not 16-byte aligned but whose x and y are misaligned
    alike (the same offset, the same stride): the cluster split reads and
    writes each row through a float4 window shifted back to the 16-byte
    boundary (the shift cycles through 0..3 when the stride is not a
    multiple of 4, and is the base offset when it is), masking the lanes
    outside the row.  Special values at both ends
    of rows, the log form and in place."""
    ld = N + pad
    assert ld % 4 != 0 or off % 4 != 0          # not a 16-byte-aligned layout
    props = torch.cuda.get_device_properties(0)
    p = rrs.plan_softmax(8, N, ld, 2, props.multi_processor_count, props.shared_memory_per_block_optin)
    assert p["path_name"] == "cluster" and p["vector_io"] == 2
    rng = np.random.default_rng(N + pad + off)
    x = rng.normal(0, 3, size=(8, N)).astype(np.float32)
    x[0, 0] = 60.0                             # the maximum in the first column
    x[1, N - 1] = 60.0                         # ... in the last column
    x[2, :3] = np.inf                          # +inf in the masked-edge float4: a NaN row
    x[3, N - 3:] = -np.inf
    x[4] = -np.inf
    x[5, 1:] = -np.inf                         # only the first column visible
    x[6, :-1] = -np.inf                        # only the last column visible
    x[7, ::3] = np.nan if N % 2 else -np.inf
    for flags, check in ((0, check_softmax), (LOG, check_log_softmax)):
        y, guards = run_ex(x, N, ld, ld, "auto", flags, x_off=off, y_off=off)
        check(y, x, f"shifted N={N} ld={ld} off={off} flags={flags}")
        assert guards
    y, guards = run_ex(x, N, ld, ld, "auto", 0, in_place=True, x_off=off)
    check_softmax(y, x, f"shifted in place N={N} ld={ld}")
    assert guards
