"""Helpers for the GPU parity tests: guarded device buffers and the tolerance checks.

Tolerances (floating point, fp32 kernel against the float64 oracle):
  * max |y - y_oracle| <= 2e-6 over every finite row;
  * max_i |sum_j y_ij - 1| <= 1e-5 (sum taken in float64 on the host);
  * |y - y_oracle| <= 1e-5 * y_oracle wherever y_oracle >= 1e-30;
  * y == 0 exactly where x == -inf (rows with a finite entry);
  * rows the oracle makes NaN (all -inf, +inf, NaN inside) are all NaN;
  * row sums: |r - r_oracle| <= 1e-5 * sum_j |x_ij| (an absolute 1e-5 is
    below one fp32 ulp of sums of magnitude 100+); row means the same over N;
  * row max: bit-exact (a max of fp32 values is one of them);
  * log-softmax: |log y - oracle| <= 1e-5 + 2^-21 |oracle| (x - m rounds at
    2^-24 |x - m|, log(s) carries s's relative error, about 2e-6, as an
    absolute one, and the final subtraction rounds at 2^-24 |log y|);
    exactly -inf where x == -inf; NaN rows as for the softmax;
  * column softmax: the row tolerances applied to each column;
  * GeLU: |y - oracle| <= 1e-6 (2 + |a|) |oracle| + 2^-50 |x| + 1e-36 with
    a = 0.79788456 (x + 0.044715 x^3): the kernel forms x / (1 + e^(-2a)),
    whose relative error is a few ulps of fp32 times |a| (the rounding of a
    scales e^(-2a) by e^(2 |a| u)); the oracle evaluates the pages' form
    0.5 x (1 + tanh(a)) in float64, where 1 + tanh(a) keeps nothing below
    2^-53 (it is exactly 0 once a < -19), hence 2^-50 |x|; 1e-36 absorbs
    results below the normal range.  +inf -> +inf; -inf, NaN -> NaN.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

SENTINEL_BITS = 0x7FC0DEAD        # a quiet NaN nobody computes
GUARD = 64                        # floats of canary before and after each buffer

ABS_TOL = 2e-6
ROW_SUM_TOL = 1e-5
REL_TOL = 1e-5
REL_FLOOR = 1e-30
SUM_TOL = 1e-5


def sentinel_fill(t: torch.Tensor) -> None:
    t.view(torch.int32).fill_(SENTINEL_BITS - (1 << 32) if SENTINEL_BITS >= 1 << 31 else SENTINEL_BITS)


class Guarded:
    """A device buffer of ``M`` rows of stride ``ld`` with canaries around it.

    ``offset`` shifts the matrix start by that many floats (misaligned bases).
    """

    def __init__(self, M: int, ld: int, offset: int = 0, device="cuda"):
        self.M, self.ld, self.offset = M, ld, offset
        self.n = M * ld
        self.raw = torch.empty(self.n + 2 * GUARD + offset, dtype=torch.float32, device=device)
        sentinel_fill(self.raw)
        self.start = GUARD + offset
        self.mat = self.raw[self.start:self.start + self.n].view(M, ld) if M * ld else \
            self.raw[self.start:self.start].view(M, ld)

    @property
    def ptr(self) -> int:
        return self.raw.data_ptr() + 4 * self.start

    def load(self, host: np.ndarray) -> None:
        self.mat.copy_(torch.from_numpy(np.ascontiguousarray(host, dtype=np.float32)))

    def untouched_outside(self, N: int) -> bool:
        """True if every float outside the M x N window still holds the sentinel."""
        bits = self.raw.view(torch.int32).cpu().numpy().astype(np.int64) & 0xFFFFFFFF
        mask = np.ones(bits.shape, dtype=bool)
        for i in range(self.M):
            a = self.start + i * self.ld
            mask[a:a + N] = False
        return bool(np.all(bits[mask] == SENTINEL_BITS))


def check_softmax(got: np.ndarray, x: np.ndarray, where: str = "") -> dict:
    """Assert the tolerances above; returns the measured errors."""
    got = np.asarray(got, dtype=np.float64)
    want = oracle.softmax_rows(x)
    M, N = want.shape
    assert got.shape == (M, N), where
    nan_rows = np.isnan(want).any(axis=1)
    for i in np.nonzero(nan_rows)[0]:
        assert np.all(np.isnan(got[i])), f"{where}: row {i} should be NaN"
    ok = ~nan_rows
    res = {"max_abs": 0.0, "row_sum": 0.0, "max_rel": 0.0}
    if not ok.any() or N == 0:
        return res
    g, w, xv = got[ok], want[ok], np.asarray(x, dtype=np.float64)[ok]
    assert np.all(np.isfinite(g)), f"{where}: non-finite output"
    abs_err = float(np.max(np.abs(g - w)))
    row_err = float(np.max(np.abs(g.sum(axis=1) - 1.0)))
    big = w >= REL_FLOOR
    rel_err = float(np.max(np.abs(g[big] - w[big]) / w[big])) if big.any() else 0.0
    assert abs_err <= ABS_TOL, f"{where}: max abs err {abs_err:.3e}"
    assert row_err <= ROW_SUM_TOL, f"{where}: row-sum err {row_err:.3e}"
    assert rel_err <= REL_TOL, f"{where}: max rel err {rel_err:.3e}"
    neg = np.isneginf(xv)
    assert np.all(g[neg] == 0.0), f"{where}: -inf entries must give exactly 0"
    res.update(max_abs=abs_err, row_sum=row_err, max_rel=rel_err)
    return res


def check_row_sum(got: np.ndarray, x: np.ndarray, where: str = "") -> float:
    xv = np.asarray(x, dtype=np.float64)
    want = oracle.row_sum(xv)
    scale = np.sum(np.abs(xv), axis=1)
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    assert np.all(err <= SUM_TOL * scale + 0.0), f"{where}: row-sum err {float(np.max(err)):.3e}"
    return float(np.max(err / np.maximum(scale, 1e-300))) if err.size else 0.0


LOG_ABS_TOL = 1e-5
LOG_REL_TOL = 2.0 ** -21


def check_log_softmax(got: np.ndarray, x: np.ndarray, where: str = "") -> float:
    got = np.asarray(got, dtype=np.float64)
    want = oracle.log_softmax_rows(x)
    assert got.shape == want.shape, where
    nan_rows = np.isnan(want).any(axis=1)
    for i in np.nonzero(nan_rows)[0]:
        assert np.all(np.isnan(got[i])), f"{where}: row {i} should be NaN"
    ok = ~nan_rows
    if not ok.any() or want.shape[1] == 0:
        return 0.0
    g, w = got[ok], want[ok]
    neg = np.isneginf(w)
    assert np.all(np.isneginf(g[neg])), f"{where}: -inf entries must give -inf"
    fin = ~neg
    err = np.abs(g[fin] - w[fin])
    bound = LOG_ABS_TOL + LOG_REL_TOL * np.abs(w[fin])
    assert np.all(err <= bound), f"{where}: log-softmax err {float(np.max(err)):.3e}"
    return float(np.max(err)) if err.size else 0.0


def check_row_max(got: np.ndarray, x: np.ndarray, where: str = "") -> None:
    want = oracle.row_max(np.asarray(x, dtype=np.float64))
    g = np.asarray(got, dtype=np.float64)
    same = (g == want) | (np.isnan(g) & np.isnan(want))
    assert np.all(same), f"{where}: row max differs at rows {np.nonzero(~same)[0][:5]}"


def check_row_mean(got: np.ndarray, x: np.ndarray, where: str = "") -> float:
    xv = np.asarray(x, dtype=np.float64)
    want = oracle.row_mean(xv)
    g = np.asarray(got, dtype=np.float64)
    if xv.shape[1] == 0:
        assert np.all(np.isnan(g)), where
        return 0.0
    scale = np.sum(np.abs(xv), axis=1) / xv.shape[1]
    err = np.abs(g - want)
    assert np.all(err <= SUM_TOL * scale), f"{where}: row-mean err {float(np.max(err)):.3e}"
    return float(np.max(err / np.maximum(scale, 1e-300)))


def check_softmax_cols(got: np.ndarray, x: np.ndarray, where: str = "", log: bool = False):
    """Column softmax: the row checks on the transposes."""
    g = np.ascontiguousarray(np.asarray(got).T)
    xt = np.ascontiguousarray(np.asarray(x).T)
    return check_log_softmax(g, xt, where) if log else check_softmax(g, xt, where)


def check_gelu(got: np.ndarray, x: np.ndarray, where: str = "") -> float:
    xv = np.asarray(x, dtype=np.float64).ravel()
    g = np.asarray(got, dtype=np.float64).ravel()
    with np.errstate(invalid="ignore", over="ignore"):
        want = oracle.gelu(xv)
        a = oracle.GELU_C * (xv + oracle.GELU_K * xv ** 3)
    nan = np.isnan(want)
    assert np.all(np.isnan(g[nan])), f"{where}: NaN expected"
    inf = np.isinf(want) & ~nan
    assert np.all(g[inf] == want[inf]), f"{where}: inf expected"
    fin = ~nan & ~inf
    err = np.abs(g[fin] - want[fin])
    with np.errstate(over="ignore"):
        bound = (1e-6 * (2.0 + np.abs(a[fin])) * np.abs(want[fin]) + 2.0 ** -50 * np.abs(xv[fin])
                 + 1e-36)
    assert np.all(err <= bound), f"{where}: gelu err {float(np.max(err)):.3e}"
    return float(np.max(err)) if err.size else 0.0


def attention_reference(qf, kf, vf, causal: bool, scale=None):
    """The oracle's (O, LSE) and, per element, the bound |O - O_oracle| may reach.

    O = P V / l with l = sum_j p_j.  Per output element (i, c), with
    A_ic = sum_j P_ij |v_jc| (the oracle's attention with |V| for V, taken in
    the same call as O by stacking V and |V| side by side):
      * p_j enters the second product rounded to bf16 (8 significant bits,
        so a relative error <= 2^-8 each), while l sums p in fp32: at most
        2^-8 A_ic;
      * a score is an fp32 sum of d exact bf16 products: absolute error <=
        d 2^-24 scale sum_k |q_ik k_jk| =: e_i (bounded by the componentwise
        max of |k| over keys), a relative error of about e_i in p_j, which
        moves O by at most e_i (A_ic + |O_ic|);
      * the fp32 sums over S keys of p v and of p: at most S 2^-24 (A_ic + |O_ic|);
      * 1e-6 for results near zero.
    A wrong V tile or a misplaced key block moves O by the weight of whole
    tiles, far above this bound."""
    d = qf.shape[-1]
    S = kf.shape[-2]
    sc = (1.0 / np.sqrt(d)) if not scale else scale
    both, lse = oracle.attention(qf, kf, np.concatenate([vf, np.abs(vf)], axis=-1), causal=causal,
                                 scale=scale or None)
    o, a = both[..., :d], both[..., d:]
    kmax = np.max(np.abs(kf), axis=-2)                               # (..., d)
    e = d * 2.0 ** -24 * sc * np.einsum("...ik,...k->...i", np.abs(qf), kmax)[..., None]
    with np.errstate(invalid="ignore"):
        bound = 2.0 ** -8 * a + (e + S * 2.0 ** -24) * (a + np.abs(o)) + 1e-6
    return o, lse, bound


def row_blocks(M: int, N: int, elements: int = 1 << 24):
    """Consecutive row ranges [r0, r1) of about ``elements`` entries each."""
    step = max(1, elements // max(N, 1))
    for r0 in range(0, M, step):
        yield r0, min(M, r0 + step)


def check_every_row(check, y_dev, x_host: np.ndarray, where: str = "") -> dict:
    """Apply a row check (check_softmax, check_log_softmax, ...) to every row of
    a device result against the oracle, one block of rows at a time; returns
    the largest of each error the check reports."""
    M, N = x_host.shape[0], x_host.shape[1]
    worst: dict = {}
    for r0, r1 in row_blocks(M, N):
        res = check(y_dev[r0:r1].cpu().numpy(), x_host[r0:r1], f"{where} rows {r0}-{r1}")
        if isinstance(res, dict):
            for k, v in res.items():
                worst[k] = max(worst.get(k, 0.0), v)
        elif res is not None:
            worst["max"] = max(worst.get("max", 0.0), float(res))
    return worst
