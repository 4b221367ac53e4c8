"""Plant plausible mistakes in copies of the oracle and check that a pin catches each.

Each mutant below is the oracle with one slip a reader could make when
restating the pages: a dropped max subtraction, the wrong axis, a missing
exp, a flipped sign, masked lanes loaded as 0 instead of -inf, a dropped
tail tile, a merge that forgets to rescale.  A pin suite that lets one of
these through would not be trusted to check the CUDA path.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from test_oracle_pins import (ATTENTION_CHECKS, GELU_CHECKS, LOG_SOFTMAX_CHECKS, MERGE_CHECKS, ROW_MAX_CHECKS, ROW_MEAN_CHECKS,
                              ROW_SUM_CHECKS, SOFTMAX_CHECKS, SOFTMAX_COLS_CHECKS)


def _rows(x):
    a = np.asarray(x, dtype=np.float64)
    return a[None, :] if a.ndim == 1 else a


def sm_no_max_shift(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a)
        return e / e.sum(axis=1, keepdims=True)


def sm_wrong_axis(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a - a.max(axis=0, keepdims=True))
        return e / e.sum(axis=0, keepdims=True)


def sm_min_shift(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a - a.min(axis=1, keepdims=True))
        return e / e.sum(axis=1, keepdims=True)


def sm_no_exp(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = a - a.max(axis=1, keepdims=True)
        return e / e.sum(axis=1, keepdims=True)


def sm_flipped_sign(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a.max(axis=1, keepdims=True) - a)
        return e / e.sum(axis=1, keepdims=True)


def sm_divide_by_max(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a - a.max(axis=1, keepdims=True))
        return e / e.max(axis=1, keepdims=True)


def sm_global_sum(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        e = np.exp(a - a.max(axis=1, keepdims=True))
        return e / e.sum()


def sm_mask_as_zero(x):
    a = np.where(np.isneginf(_rows(x)), 0.0, _rows(x))
    return oracle.softmax_rows(a)


def sm_drop_last_column(x):
    a = _rows(x)
    y = oracle.softmax_rows(a[:, :-1]) if a.shape[1] > 1 else oracle.softmax_rows(a)
    out = np.zeros_like(a)
    out[:, :y.shape[1]] = y
    return out


SOFTMAX_MUTANTS = [sm_no_max_shift, sm_wrong_axis, sm_min_shift, sm_no_exp, sm_flipped_sign,
                   sm_divide_by_max, sm_global_sum, sm_mask_as_zero, sm_drop_last_column]


def rst_drop_tail(row, block):
    r = np.asarray(row, dtype=np.float64).ravel()
    acc = np.zeros(block)
    trace = []
    for start in range(0, r.size - block + 1, block):   # forgets the ragged tile
        acc = acc + r[start:start + block]
        trace.append(acc.copy())
    return trace, float(acc.sum())


def rst_wraparound(row, block):
    r = np.asarray(row, dtype=np.float64).ravel()
    acc = np.zeros(block)
    trace = []
    for start in range(0, r.size, block):
        tile = np.resize(r[start:], block)                  # masked lanes not zero
        acc = acc + tile
        trace.append(acc.copy())
    return trace, float(acc.sum())


def rs_mean(x):
    return np.mean(_rows(x), axis=1) if _rows(x).shape[1] else np.zeros(_rows(x).shape[0])


def rs_float32(x):
    return np.sum(_rows(x).astype(np.float32), axis=1, dtype=np.float32).astype(np.float64)


ROW_SUM_MUTANTS = [(oracle.row_sum, rst_drop_tail), (oracle.row_sum, rst_wraparound),
                   (rs_mean, oracle.row_sum_tiles), (rs_float32, oracle.row_sum_tiles)]


def mg_no_rescale(a, b):
    return (max(a[0], b[0]), a[1] + b[1])


def mg_min(a, b):
    m = min(a[0], b[0]) if min(a[0], b[0]) != -np.inf else max(a[0], b[0])
    with np.errstate(all="ignore"):
        ta = 0.0 if a[0] == -np.inf else a[1] * float(np.exp(a[0] - m))
        tb = 0.0 if b[0] == -np.inf else b[1] * float(np.exp(b[0] - m))
    return (m, ta + tb)


def mg_flipped(a, b):
    m = max(a[0], b[0])
    if m == -np.inf:
        return (-np.inf, 0.0)
    ta = 0.0 if a[0] == -np.inf else a[1] * float(np.exp(m - a[0]))
    tb = 0.0 if b[0] == -np.inf else b[1] * float(np.exp(m - b[0]))
    return (m, ta + tb)


def mg_unguarded(a, b):
    m = max(a[0], b[0])
    with np.errstate(all="ignore"):
        return (m, a[1] * float(np.exp(a[0] - m)) + b[1] * float(np.exp(b[0] - m)))


MERGE_MUTANTS = [mg_no_rescale, mg_min, mg_flipped, mg_unguarded]


def _caught(fn, *args) -> bool:
    try:
        fn(*args)
    except (AssertionError, ValueError, FloatingPointError, IndexError):
        return True
    return False


@pytest.mark.parametrize("mutant", SOFTMAX_MUTANTS, ids=lambda m: m.__name__)
def test_softmax_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in SOFTMAX_CHECKS)


@pytest.mark.parametrize("pair", ROW_SUM_MUTANTS, ids=lambda p: p[0].__name__ + "+" + p[1].__name__)
def test_row_sum_mutant_is_caught(pair):
    assert any(_caught(check, *pair) for check in ROW_SUM_CHECKS)


@pytest.mark.parametrize("mutant", MERGE_MUTANTS, ids=lambda m: m.__name__)
def test_merge_mutant_is_caught(mutant):
    assert any(_caught(check, oracle.partial, mutant) for check in MERGE_CHECKS)



def lsm_no_log(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        z = a - a.max(axis=1, keepdims=True)
        return z - np.exp(z).sum(axis=1, keepdims=True)      # forgot the log


def lsm_flipped(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        z = a.max(axis=1, keepdims=True) - a
        return z - np.log(np.exp(-z).sum(axis=1, keepdims=True))


def lsm_unshifted_log(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        z = a - a.max(axis=1, keepdims=True)
        return a - np.log(np.exp(z).sum(axis=1, keepdims=True))   # m dropped from the output


def lsm_log_of_softmax_max(x):
    a = _rows(x)
    with np.errstate(all="ignore"):
        z = a - a.max(axis=1, keepdims=True)
        return z - np.log(np.exp(z).max(axis=1, keepdims=True))


LOG_SOFTMAX_MUTANTS = [lsm_no_log, lsm_flipped, lsm_unshifted_log, lsm_log_of_softmax_max]


def rmax_min(x):
    a = _rows(x)
    return np.min(a, axis=1) if a.shape[1] else np.full(a.shape[0], -np.inf)


def rmax_nan_ignoring(x):
    a = _rows(x)
    return np.nanmax(a, axis=1) if a.shape[1] else np.full(a.shape[0], -np.inf)


def rmax_empty_zero(x):
    a = _rows(x)
    return np.max(a, axis=1) if a.shape[1] else np.zeros(a.shape[0])


ROW_MAX_MUTANTS = [rmax_min, rmax_nan_ignoring, rmax_empty_zero]


def rmean_n_minus_one(x):
    a = _rows(x)
    return a.sum(axis=1) / max(a.shape[1] - 1, 1) if a.shape[1] else np.full(a.shape[0], np.nan)


def rmean_sum(x):
    a = _rows(x)
    return a.sum(axis=1) if a.shape[1] else np.full(a.shape[0], np.nan)


def rmean_empty_zero(x):
    a = _rows(x)
    return a.sum(axis=1) / a.shape[1] if a.shape[1] else np.zeros(a.shape[0])


ROW_MEAN_MUTANTS = [rmean_n_minus_one, rmean_sum, rmean_empty_zero]


def scols_wrong_axis(x):
    return oracle.softmax_rows(np.asarray(x, dtype=np.float64))


def scols_no_shift(x):
    a = np.asarray(x, dtype=np.float64)
    with np.errstate(all="ignore"):
        e = np.exp(a)
        return e / e.sum(axis=0, keepdims=True)


def scols_row_max_shift(x):
    a = np.asarray(x, dtype=np.float64)
    with np.errstate(all="ignore"):
        e = np.exp(a - a.max(axis=1, keepdims=True))
        return e / e.sum(axis=0, keepdims=True)


SOFTMAX_COLS_MUTANTS = [scols_wrong_axis, scols_no_shift, scols_row_max_shift]


@pytest.mark.parametrize("mutant", LOG_SOFTMAX_MUTANTS, ids=lambda m: m.__name__)
def test_log_softmax_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in LOG_SOFTMAX_CHECKS)


@pytest.mark.parametrize("mutant", ROW_MAX_MUTANTS, ids=lambda m: m.__name__)
def test_row_max_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in ROW_MAX_CHECKS)


@pytest.mark.parametrize("mutant", ROW_MEAN_MUTANTS, ids=lambda m: m.__name__)
def test_row_mean_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in ROW_MEAN_CHECKS)


@pytest.mark.parametrize("mutant", SOFTMAX_COLS_MUTANTS, ids=lambda m: m.__name__)
def test_softmax_cols_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in SOFTMAX_COLS_CHECKS)



def gelu_no_half(x):
    a = np.asarray(x, dtype=np.float64)
    return a * (1.0 + np.tanh(0.79788456 * (a + 0.044715 * a ** 3)))


def gelu_square_term(x):
    a = np.asarray(x, dtype=np.float64)
    return 0.5 * a * (1.0 + np.tanh(0.79788456 * (a + 0.044715 * a ** 2)))


def gelu_minus_tanh(x):
    a = np.asarray(x, dtype=np.float64)
    return 0.5 * a * (1.0 - np.tanh(0.79788456 * (a + 0.044715 * a ** 3)))


def gelu_sigmoid_form(x):                     # x * sigmoid(1.702 x): a different approximation
    a = np.asarray(x, dtype=np.float64)
    return a / (1.0 + np.exp(-1.702 * a))


GELU_MUTANTS = [gelu_no_half, gelu_square_term, gelu_minus_tanh, gelu_sigmoid_form]


@pytest.mark.parametrize("mutant", GELU_MUTANTS, ids=lambda m: m.__name__)
def test_gelu_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in GELU_CHECKS)



def _att(q, k, v, causal=False, scale=None, *, flip=False, noscale=False, colsm=False, mask_diag=False):
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    L, d, S = q.shape[-2], q.shape[-1], k.shape[-2]
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    s = np.matmul(q, np.swapaxes(k, -1, -2)) * (1.0 if noscale else sc)
    if causal:
        i = np.arange(L)[:, None]
        j = np.arange(S)[None, :]
        s = np.where((j >= i + (S - L)) if mask_diag else (j > i + (S - L)), -np.inf, s)
    with np.errstate(all="ignore"):
        if colsm:
            e = np.exp(s - s.max(axis=-2, keepdims=True))
            p = e / e.sum(axis=-2, keepdims=True)
        else:
            e = np.exp(s - s.max(axis=-1, keepdims=True))
            p = e / e.sum(axis=-1, keepdims=True)
        m = s.max(axis=-1)
        lse = m + np.log(np.exp(s - m[..., None]).sum(axis=-1))
    o = np.matmul(p, v if not flip else v[..., ::-1, :])
    return o, lse


def att_no_scale(q, k, v, causal=False, scale=None):
    return _att(q, k, v, causal, scale, noscale=True)


def att_softmax_over_queries(q, k, v, causal=False, scale=None):
    return _att(q, k, v, causal, scale, colsm=True)


def att_mask_diagonal(q, k, v, causal=False, scale=None):
    return _att(q, k, v, causal, scale, mask_diag=True)


def att_reversed_values(q, k, v, causal=False, scale=None):
    return _att(q, k, v, causal, scale, flip=True)


ATTENTION_MUTANTS = [att_no_scale, att_softmax_over_queries, att_mask_diagonal, att_reversed_values]


@pytest.mark.parametrize("mutant", ATTENTION_MUTANTS, ids=lambda m: m.__name__)
def test_attention_mutant_is_caught(mutant):
    assert any(_caught(check, mutant) for check in ATTENTION_CHECKS)
