"""Seeded random cases through the C ABI, against the float64 oracle.

Each case draws a shape, strides, base offsets, a value recipe (Gaussian of
a random spread, +50 spikes, -inf masks, occasionally a whole row or column
of -inf) and an execution path; the tolerances are those of the other GPU
tests (gpu_helpers).  The generator is seeded, so a failing case is
reproduced by its index.  Sizes stay small enough for the oracle to check
every output.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import Guarded, attention_reference, check_log_softmax, check_softmax, check_softmax_cols
from test_softmax_gpu import PATHS, supports

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

UNSUPPORTED = 6


@pytest.fixture(autouse=True)
def _auto_paths(lib):
    rrs.force_path("auto", "auto")
    rrs.force_cols_path("auto")
    yield
    rrs.force_path("auto", "auto")
    rrs.force_cols_path("auto")


def values(rng: np.random.Generator, M: int, N: int) -> np.ndarray:
    x = rng.normal(0.0, float(rng.choice([0.1, 1.0, 5.0, 30.0])), size=(M, N)).astype(np.float32)
    if rng.random() < 0.3:                                   # spikes
        k = max(1, int(0.03 * M * N))
        x.flat[rng.choice(M * N, size=k, replace=False)] = 50.0
    if rng.random() < 0.3:                                   # masked entries
        k = max(1, int(0.01 * M * N))
        x.flat[rng.choice(M * N, size=k, replace=False)] = -np.inf
    if rng.random() < 0.1 and M > 1:                         # a fully masked row (a NaN row)
        x[rng.integers(M)] = -np.inf
    return x


def log_uniform(rng, lo: int, hi: int) -> int:
    return int(round(np.exp(rng.uniform(np.log(lo), np.log(hi)))))


@pytest.mark.parametrize("case", range(100))
def test_fuzz_softmax_rows(case):
    rng = np.random.default_rng(1000 + case)
    N = log_uniform(rng, 1, 300000)
    M = max(1, min(log_uniform(rng, 1, 400), 1_500_000 // N))
    aligned = rng.random() < 0.7
    pad = int(rng.choice([0, 4, 8, 64])) if aligned else int(rng.integers(0, 7))
    ldx = (-(-N // 4) * 4 if aligned else N) + pad
    ldy = ldx if rng.random() < 0.6 else ldx + (4 * int(rng.integers(0, 3)) if aligned else int(rng.integers(0, 5)))
    x_off = 0 if aligned else int(rng.integers(0, 4))
    y_off = 0 if aligned else int(rng.integers(0, 4))
    path = "auto"
    if aligned and rng.random() < 0.6:
        cands = [p for p in PATHS if supports(p, N, max(ldx, ldy))]
        path = cands[int(rng.integers(len(cands)))] if cands else "auto"
    log = rng.random() < 0.25
    if log and path == "row_staged":                          # the staged kernel has no log form
        path = "auto"
    x = values(rng, M, N)
    xb, yb = Guarded(M, ldx, x_off), Guarded(M, ldy, y_off)
    xb.mat[:, :N].copy_(torch.from_numpy(x))
    rrs.force_path(path, "auto")
    where = f"case {case}: {M}x{N} ldx={ldx} ldy={ldy} off={x_off},{y_off} path={path} log={log}"
    try:
        rrs.softmax_rows_ex_ptr(xb.ptr, ldx, yb.ptr, ldy, M, N, rrs.LOG_SOFTMAX if log else 0,
                                torch.cuda.current_stream().cuda_stream)
    except rrs.RRSError as e:
        assert e.status == UNSUPPORTED and path != "auto", f"{where}: {e}"
        pytest.skip(f"{where}: path not available for this shape")
    torch.cuda.synchronize()
    assert rrs.device_error() == 0, where
    y = yb.mat[:, :N].cpu().numpy()
    (check_log_softmax if log else check_softmax)(y, x, where)
    assert xb.untouched_outside(N) and yb.untouched_outside(N), f"{where}: a canary was overwritten"
    assert np.array_equal(xb.mat[:, :N].cpu().numpy(), x, equal_nan=True), f"{where}: x was modified"


@pytest.mark.parametrize("case", range(60))
def test_fuzz_softmax_cols(case):
    rng = np.random.default_rng(2000 + case)
    M = log_uniform(rng, 1, 9000)
    N = max(1, min(log_uniform(rng, 1, 3000), 1_000_000 // M))
    aligned = rng.random() < 0.75
    ld = (-(-N // 4) * 4 if aligned else N) + (4 * int(rng.integers(0, 3)) if aligned else int(rng.integers(0, 3)))
    path = "auto"
    if aligned and rng.random() < 0.6:
        path = str(rng.choice(["band", "two_phase", "two_pass"] + (["cluster"] if M <= 8192 else [])))
    log = rng.random() < 0.25
    x = values(rng, M, N)
    if rng.random() < 0.1:
        x[:, rng.integers(N)] = -np.inf                         # a fully masked column
    xb, yb = Guarded(M, ld), Guarded(M, ld)
    xb.mat[:, :N].copy_(torch.from_numpy(x))
    rrs.force_cols_path(path)
    where = f"case {case}: {M}x{N} ld={ld} path={path} log={log}"
    rrs.softmax_cols_ptr(xb.ptr, ld, yb.ptr, ld, M, N, rrs.LOG_SOFTMAX if log else 0,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0, where
    check_softmax_cols(yb.mat[:, :N].cpu().numpy(), x, where, log=log)
    assert xb.untouched_outside(N) and yb.untouched_outside(N), f"{where}: a canary was overwritten"


@pytest.mark.parametrize("case", range(24))
def test_fuzz_attention(case):
    rng = np.random.default_rng(3000 + case)
    BH = int(rng.integers(1, 4))
    L, S = log_uniform(rng, 1, 700), log_uniform(rng, 1, 700)
    d = int(rng.choice([64, 128]))
    causal = bool(rng.random() < 0.5)
    spread = float(rng.choice([0.5, 1.0, 3.0]))
    q, k, v = (workloads.to_bf16_bits(rng.normal(0, spread, size=(BH, n, d)).astype(np.float32))
               for n in (L, S, S))
    dev = lambda bits: torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    o, lse = rrs.attention(dev(q), dev(k), dev(v), causal=causal)
    torch.cuda.synchronize()
    where = f"case {case}: BH={BH} L={L} S={S} d={d} causal={causal} spread={spread}"
    assert rrs.device_error() == 0, where
    f64 = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want_o, want_l, bound = attention_reference(f64(q), f64(k), f64(v), causal)
    got_o, got_l = o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    dead = np.isnan(want_o).any(axis=-1)
    assert np.all(np.isnan(got_o[dead])) and np.all(np.isneginf(got_l[dead])), f"{where}: rows with no key"
    ok = ~dead
    assert np.all(np.abs(got_o - want_o)[ok] <= bound[ok]), f"{where}: O"
    lerr = np.abs(got_l[ok] - want_l[ok])
    assert np.all(lerr <= 1e-5 * np.maximum(1.0, np.abs(want_l[ok])) + 1e-5), f"{where}: LSE"
