"""Pins for the float64 oracle: values the pages print and facts the mathematics fixes.

None of these retypes the oracle's own formula.  The softmax is pinned by
closed forms (uniform row, two-element sigmoid, one-hot limit), invariants
(rows sum to one, shift invariance), brute force along a different route
(un-shifted exp over an exactly rounded sum, in pure Python) and library
routines (torch / scipy softmax in float64).  The row sum is pinned by the
lecture's worked example (3,1,4,1 | 5,9,2,6 | 5,3 -> 39), Gauss's closed form
and an exactly rounded sum.  ``test_oracle_mutants.py`` plants plausible
mistakes in copies of these functions and checks that a pin here fails.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fixtures ----

def load_worked_example():
    rec = {}
    with open(os.path.join(GOLDEN, "row_sum_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            rec[key.strip()] = [float(v) for v in val.split()]
    return rec


def small_cases():
    """Small matrices in each workload's value recipe (ragged shapes included)."""
    out = []
    for name, (M, N) in {"c1": (7, 256), "c2": (5, 1000), "c3": (3, 4097),
                         "c4": (6, 333), "c5": (2, 5003)}.items():
        w = workloads.WORKLOADS[name].with_shape(M, N)
        out.append((name, workloads.matrix(w).astype(np.float64)))
    return out


# ------------------------------------------------------- softmax pin checks ----

def check_rows_sum_to_one(sm):
    for name, x in small_cases():
        y = sm(x)
        assert y.shape == x.shape, name
        assert np.all(np.isfinite(y)), name
        assert np.max(np.abs(np.sum(y, axis=1) - 1.0)) <= 1e-12, name


def check_shift_invariance(sm):
    rng = np.random.default_rng(11)
    x = rng.normal(0.0, 3.0, size=(4, 37))
    base = sm(x)
    for c in (-100.0, 1000.0):
        shifted = sm(x + c)
        assert np.all(np.isfinite(shifted)), c
        assert np.max(np.abs(shifted - base)) <= 1e-12, c


def check_constant_row(sm):
    for N in (1, 2, 3, 7, 256, 1000):
        for v in (-5.0, 0.0, 42.0):
            y = sm(np.full((2, N), v))
            assert np.all(y == 1.0 / N), (N, v)


def check_two_element_sigmoid(sm):
    rng = np.random.default_rng(12)
    for _ in range(200):
        x0, x1 = rng.uniform(-30, 30, size=2)
        y = sm(np.array([[x0, x1]]))[0]
        s0 = 1.0 / (1.0 + math.exp(x1 - x0))
        s1 = 1.0 / (1.0 + math.exp(x0 - x1))
        assert abs(y[0] - s0) <= 1e-14 * max(s0, 1e-300) + 1e-300
        assert abs(y[1] - s1) <= 1e-14 * max(s1, 1e-300) + 1e-300


def check_brute_force(sm):
    """Un-shifted exp over an exactly rounded sum, element by element, in pure Python."""
    rng = np.random.default_rng(13)
    for M, N in ((3, 5), (5, 3), (1, 8), (4, 1), (2, 7)):
        x = rng.uniform(-20, 20, size=(M, N))
        y = sm(x)
        for i in range(M):
            den = math.fsum(math.exp(v) for v in x[i])
            for j in range(N):
                want = math.exp(x[i, j]) / den
                assert abs(y[i, j] - want) <= 1e-14 * want, (M, N, i, j)


def check_library(sm):
    torch = pytest.importorskip("torch")
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(14)
    x = rng.normal(0, 4, size=(9, 50))
    y = sm(x)
    t = torch.softmax(torch.from_numpy(x), dim=1).numpy()
    s = scipy_special.softmax(x, axis=1)
    assert np.max(np.abs(y - t)) <= 1e-15
    assert np.max(np.abs(y - s)) <= 1e-15


def check_one_hot_limit(sm):
    x = np.zeros((3, 10))
    for i, j in enumerate((0, 4, 9)):
        x[i, j] = 1e4
    y = sm(x)
    for i, j in enumerate((0, 4, 9)):
        want = np.zeros(10)
        want[j] = 1.0
        assert np.array_equal(y[i], want)


def check_masked_entries(sm):
    w = workloads.WORKLOADS["c4"].with_shape(4, 4096)
    x = workloads.matrix(w).astype(np.float64)
    y = sm(x)
    neg = np.isneginf(x)
    assert neg.sum() == 4 * 41
    assert np.all(y[neg] == 0.0)
    for i in range(4):
        spikes = x[i] == 50.0
        assert spikes.sum() == 205
        vals = y[i][spikes]
        assert np.all(vals == vals[0])      # ties share the mass exactly
        # the spikes dominate: all other entries are below e^(max normal - 50)
        assert vals.sum() > 1.0 - 1e-9


def check_all_masked_row_is_nan(sm):
    x = np.array([[-np.inf, -np.inf, -np.inf], [0.0, -np.inf, 0.0]])
    y = sm(x)
    assert np.all(np.isnan(y[0]))
    assert y[1, 0] == 0.5 and y[1, 1] == 0.0 and y[1, 2] == 0.5


SOFTMAX_CHECKS = [
    check_rows_sum_to_one, check_shift_invariance, check_constant_row,
    check_two_element_sigmoid, check_brute_force, check_library,
    check_one_hot_limit, check_masked_entries, check_all_masked_row_is_nan,
]


# ------------------------------------------------------- row-sum pin checks ----

def check_worked_example(rs, rst):
    g = load_worked_example()
    row = np.array(g["row"])
    block = int(g["block"][0])
    trace, total = rst(row, block)
    assert len(trace) == 3
    for k in range(3):
        assert list(trace[k]) == g[f"acc_after_tile_{k}"]
    assert total == g["total"][0] == 39.0
    assert rs(row[None, :])[0] == 39.0


def check_gauss(rs, rst):
    for N in (1, 2, 10, 999, 4096, 32768):
        x = np.arange(1, N + 1, dtype=np.float64)[None, :]
        assert rs(x)[0] == N * (N + 1) // 2
        assert rst(x[0], 1024)[1] == N * (N + 1) // 2


def check_exact_sum(rs, rst):
    for name, x in small_cases():
        x = np.where(np.isfinite(x), x, 0.0)
        got = rs(x)
        for i in range(x.shape[0]):
            want = math.fsum(x[i])
            scale = math.fsum(abs(v) for v in x[i])
            assert abs(got[i] - want) <= 1e-13 * scale, name
            assert abs(rst(x[i], 128)[1] - want) <= 1e-13 * scale, name


def check_empty_rows(rs, rst):
    assert np.array_equal(rs(np.zeros((3, 0))), np.zeros(3))
    assert rst(np.zeros(0), 4) == ([], 0.0)


ROW_SUM_CHECKS = [check_worked_example, check_gauss, check_exact_sum, check_empty_rows]


# --------------------------------------------------------- merge pin checks ----

def check_merge_equals_unsplit(part, mg):
    rng = np.random.default_rng(15)
    for trial in range(50):
        N = int(rng.integers(2, 400))
        x = rng.normal(0, 5, size=N)
        if trial % 5 == 0:
            x[rng.choice(N, size=N // 3, replace=False)] = -np.inf
        whole_m = float(np.max(x))
        whole_s = math.fsum(math.exp(v - whole_m) for v in x)
        k = int(rng.integers(1, min(N, 9)))
        cuts = sorted(rng.choice(np.arange(1, N), size=k, replace=False).tolist())
        bounds = [0] + cuts + [N]
        parts = [part(x[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        order = rng.permutation(len(parts))
        acc = (-np.inf, 0.0)
        for idx in order:
            acc = mg(acc, parts[idx])
        assert acc[0] == whole_m
        assert abs(acc[1] - whole_s) <= 1e-13 * whole_s


def check_merge_identity_and_masked(part, mg):
    p = (1.5, 3.25)
    assert mg((-np.inf, 0.0), p) == p
    assert mg(p, (-np.inf, 0.0)) == p
    masked = part(np.array([-np.inf, -np.inf]))
    assert masked == (-np.inf, 0.0)
    got = mg(masked, part(np.array([0.0, 0.0])))
    assert got == (0.0, 2.0)
    assert mg(masked, masked) == (-np.inf, 0.0)


MERGE_CHECKS = [check_merge_equals_unsplit, check_merge_identity_and_masked]


# ------------------------------------------------------------------- tests ----

@pytest.mark.parametrize("check", SOFTMAX_CHECKS, ids=lambda c: c.__name__)
def test_softmax_pins(check):
    check(oracle.softmax_rows)


@pytest.mark.parametrize("check", ROW_SUM_CHECKS, ids=lambda c: c.__name__)
def test_row_sum_pins(check):
    check(oracle.row_sum, oracle.row_sum_tiles)


@pytest.mark.parametrize("check", MERGE_CHECKS, ids=lambda c: c.__name__)
def test_merge_pins(check):
    check(oracle.partial, oracle.merge)


def test_split_softmax_matches_definition():
    rng = np.random.default_rng(16)
    x = rng.normal(0, 3, size=(6, 1000))
    x[2, ::7] = -np.inf
    for cuts in ([500], [1, 999], [10, 250, 251, 700]):
        assert np.max(np.abs(oracle.softmax_rows_split(x, cuts) - oracle.softmax_rows(x))) <= 1e-15
    for check in (check_rows_sum_to_one, check_brute_force, check_masked_entries,
                  check_one_hot_limit, check_shift_invariance):
        check(lambda a: oracle.softmax_rows_split(a, [1] if np.asarray(a).shape[1] > 1 else []))


def test_empty_columns():
    assert oracle.softmax_rows(np.zeros((4, 0))).shape == (4, 0)


# ------------------------------------------------- log-softmax pin checks ----

def check_log_exp_is_softmax(lsm):
    """exp of the log-softmax is the (independently pinned) softmax."""
    for name, x in small_cases():
        got = np.exp(lsm(x))
        want = oracle.softmax_rows(x)
        assert np.max(np.abs(got - want)) <= 1e-13, name


def check_log_two_element(lsm):
    rng = np.random.default_rng(21)
    for _ in range(200):
        x0, x1 = rng.uniform(-30, 30, size=2)
        y = lsm(np.array([[x0, x1]]))[0]
        want0 = -math.log1p(math.exp(x1 - x0))     # log sigma(x0 - x1)
        want1 = -math.log1p(math.exp(x0 - x1))
        assert abs(y[0] - want0) <= 1e-13 * max(1.0, abs(want0))
        assert abs(y[1] - want1) <= 1e-13 * max(1.0, abs(want1))


def check_log_brute_force(lsm):
    """x_j - log(sum_k exp(x_k)) with an exactly rounded sum (no max shift)."""
    rng = np.random.default_rng(22)
    for M, N in ((3, 5), (5, 3), (1, 8), (2, 7)):
        x = rng.uniform(-20, 20, size=(M, N))
        y = lsm(x)
        for i in range(M):
            lse = math.log(math.fsum(math.exp(v) for v in x[i]))
            for j in range(N):
                assert abs(y[i, j] - (x[i, j] - lse)) <= 1e-13 * max(1.0, abs(y[i, j]))


def check_log_library(lsm):
    torch = pytest.importorskip("torch")
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(23)
    x = rng.normal(0, 4, size=(9, 50))
    y = lsm(x)
    assert np.max(np.abs(y - torch.log_softmax(torch.from_numpy(x), dim=1).numpy())) <= 1e-13
    assert np.max(np.abs(y - scipy_special.log_softmax(x, axis=1))) <= 1e-13


def check_log_special_rows(lsm):
    for N in (1, 2, 7, 1000):
        y = lsm(np.full((1, N), 3.5))[0]
        assert np.max(np.abs(y + math.log(N))) <= 1e-15 * max(1.0, math.log(N))
    y = lsm(np.array([[0.0, -np.inf, 0.0], [-np.inf, -np.inf, -np.inf]]))
    assert y[0, 1] == -np.inf and abs(y[0, 0] + math.log(2)) <= 1e-16
    assert np.all(np.isnan(y[1]))
    rng = np.random.default_rng(24)
    x = rng.normal(0, 3, size=(3, 40))
    for c in (-100.0, 1000.0):                        # shift invariance
        assert np.max(np.abs(lsm(x + c) - lsm(x))) <= 1e-11


LOG_SOFTMAX_CHECKS = [check_log_exp_is_softmax, check_log_two_element, check_log_brute_force,
                      check_log_library, check_log_special_rows]


# ------------------------------------------------- row max / mean pin checks ----

def check_max_worked_example(rmax):
    g = load_worked_example()
    assert rmax(np.array(g["row"])[None, :])[0] == 9.0      # 3 1 4 1 5 9 2 6 5 3


def check_max_brute_force(rmax):
    for name, x in small_cases():
        got = rmax(x)
        for i in range(x.shape[0]):
            assert got[i] == max(x[i].tolist()), name   # Python's max, element by element


def check_max_special(rmax):
    x = np.array([[1.0, np.nan, 3.0], [-np.inf, -np.inf, -np.inf], [-np.inf, -7.0, -np.inf]])
    got = rmax(x)
    assert math.isnan(got[0]) and got[1] == -np.inf and got[2] == -7.0
    assert np.all(rmax(np.zeros((2, 0))) == -np.inf)


def check_mean_worked_example(rmean):
    g = load_worked_example()
    assert rmean(np.array(g["row"])[None, :])[0] == 39.0 / 10.0


def check_mean_gauss(rmean):
    for N in (1, 2, 10, 999, 4096):
        x = np.arange(1, N + 1, dtype=np.float64)[None, :]
        assert rmean(x)[0] == (N + 1) / 2


def check_mean_exact(rmean):
    for name, x in small_cases():
        x = np.where(np.isfinite(x), x, 0.0)
        got = rmean(x)
        for i in range(x.shape[0]):
            want = math.fsum(x[i]) / x.shape[1]
            scale = math.fsum(abs(v) for v in x[i]) / x.shape[1]
            assert abs(got[i] - want) <= 1e-13 * scale, name
    assert np.all(np.isnan(rmean(np.zeros((2, 0)))))


ROW_MAX_CHECKS = [check_max_worked_example, check_max_brute_force, check_max_special]
ROW_MEAN_CHECKS = [check_mean_worked_example, check_mean_gauss, check_mean_exact]


# ------------------------------------------------- column softmax pin checks ----

def check_cols_transposed_rows(scols):
    """A column softmax is the (independently pinned) row softmax of the transpose."""
    for name, x in small_cases():
        xt = np.ascontiguousarray(x.T)                # N x M: columns of length M
        assert np.max(np.abs(scols(xt) - oracle.softmax_rows(x).T)) <= 1e-15, name


def check_cols_sum_to_one(scols):
    rng = np.random.default_rng(25)
    x = rng.normal(0, 3, size=(300, 17))
    assert np.max(np.abs(scols(x).sum(axis=0) - 1.0)) <= 1e-12


def check_cols_two_rows(scols):
    rng = np.random.default_rng(26)
    x = rng.uniform(-30, 30, size=(2, 50))
    y = scols(x)
    for j in range(50):
        want = 1.0 / (1.0 + math.exp(x[1, j] - x[0, j]))
        assert abs(y[0, j] - want) <= 1e-14 * max(want, 1e-300) + 1e-300


def check_cols_library_and_shift(scols):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(27)
    x = rng.normal(0, 4, size=(60, 9))
    y = scols(x)
    assert np.max(np.abs(y - torch.softmax(torch.from_numpy(x), dim=0).numpy())) <= 1e-15
    assert np.max(np.abs(scols(x + 1000.0) - y)) <= 1e-12
    z = np.array([[-np.inf, 0.0], [-np.inf, -np.inf]])
    got = scols(z)
    assert np.all(np.isnan(got[:, 0])) and got[0, 1] == 1.0 and got[1, 1] == 0.0


SOFTMAX_COLS_CHECKS = [check_cols_transposed_rows, check_cols_sum_to_one, check_cols_two_rows,
                       check_cols_library_and_shift]


@pytest.mark.parametrize("check", LOG_SOFTMAX_CHECKS, ids=lambda c: c.__name__)
def test_log_softmax_pins(check):
    check(oracle.log_softmax_rows)


@pytest.mark.parametrize("check", ROW_MAX_CHECKS, ids=lambda c: c.__name__)
def test_row_max_pins(check):
    check(oracle.row_max)


@pytest.mark.parametrize("check", ROW_MEAN_CHECKS, ids=lambda c: c.__name__)
def test_row_mean_pins(check):
    check(oracle.row_mean)


@pytest.mark.parametrize("check", SOFTMAX_COLS_CHECKS, ids=lambda c: c.__name__)
def test_softmax_cols_pins(check):
    check(oracle.softmax_cols)



# ------------------------------------------------------------- GeLU pin checks ----

def check_gelu_closed_values(g):
    assert g(np.array([0.0]))[0] == 0.0
    want1 = 0.5 * (1.0 + math.tanh(0.79788456 * (1.0 + 0.044715)))   # x = 1, the pages' check value
    assert abs(g(np.array([1.0]))[0] - want1) <= 1e-16
    assert abs(want1 - 0.8411919906) <= 1e-9                          # the number itself
    big = np.array([10.0, 30.0, 1e3])
    assert np.all(g(big) == big)                                      # tanh saturates to 1
    assert np.all(g(-big) == 0.0)


def check_gelu_reflection(g):
    """gelu(x) - gelu(-x) = x: the tanh terms cancel (tanh is odd)."""
    x = np.random.default_rng(41).normal(0, 3, size=1000)
    assert np.max(np.abs(g(x) - g(-x) - x)) <= 1e-14 * max(1.0, float(np.max(np.abs(x))))


def check_gelu_library(g):
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(42).normal(0, 3, size=(64, 64))
    t = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    # torch uses sqrt(2/pi) = 0.7978845608...; the pages round it to 0.79788456
    assert np.max(np.abs(g(x) - t)) <= 1e-8


def check_gelu_derivative_at_zero(g):
    """d/dx gelu at 0 is 1/2 (central difference), and gelu is smooth there."""
    h = 1e-6
    d = (g(np.array([h]))[0] - g(np.array([-h]))[0]) / (2 * h)
    assert abs(d - 0.5) <= 1e-9


GELU_CHECKS = [check_gelu_closed_values, check_gelu_reflection, check_gelu_library,
               check_gelu_derivative_at_zero]


@pytest.mark.parametrize("check", GELU_CHECKS, ids=lambda c: c.__name__)
def test_gelu_pins(check):
    check(oracle.gelu)



# -------------------------------------------------------- attention pin checks ----

def check_attn_uniform_scores(att):
    """q = 0: every score is 0, so every output row is the mean of v's rows."""
    rng = np.random.default_rng(51)
    k = rng.normal(size=(2, 7, 16)); v = rng.normal(size=(2, 7, 16))
    o, lse = att(np.zeros((2, 5, 16)), k, v)
    assert np.max(np.abs(o - v.mean(axis=1, keepdims=True))) <= 1e-14
    assert np.max(np.abs(lse - math.log(7))) <= 1e-14


def check_attn_one_hot(att):
    """A query far more aligned with one key than the rest returns that key's value row."""
    d = 8
    k = np.eye(d)[:6] * 1.0
    v = np.arange(6 * d, dtype=np.float64).reshape(6, d)
    q = np.zeros((3, d))
    for i, j in enumerate((0, 3, 5)):
        q[i, j] = 1e4
    o, _ = att(q, k, v, scale=1.0)
    for i, j in enumerate((0, 3, 5)):
        assert np.array_equal(o[i], v[j])


def check_attn_causal_first_row(att):
    """Causal: query 0 sees key 0 only, so O[0] = v[0] and LSE[0] = score[0, 0]."""
    rng = np.random.default_rng(52)
    q = rng.normal(size=(4, 8)); k = rng.normal(size=(4, 8)); v = rng.normal(size=(4, 8))
    o, lse = att(q, k, v, causal=True)
    assert np.max(np.abs(o[0] - v[0])) <= 1e-15
    assert abs(lse[0] - float(q[0] @ k[0]) / math.sqrt(8)) <= 1e-14
    o2, _ = att(q[:1], k[:1], v[:1])                   # prefix = non-causal on the prefix
    assert np.max(np.abs(o[:1] - o2)) <= 1e-15


def check_attn_brute_force(att):
    """Pure-Python loops with an exactly rounded normaliser."""
    rng = np.random.default_rng(53)
    for causal in (False, True):
        q = rng.normal(size=(5, 3)); k = rng.normal(size=(5, 3)); v = rng.normal(size=(5, 4))
        o, lse = att(q, k, v, causal=causal, scale=0.7)
        for i in range(5):
            js = [j for j in range(5) if not (causal and j > i)]
            sc = [0.7 * sum(q[i, t] * k[j, t] for t in range(3)) for j in js]
            den = math.fsum(math.exp(x) for x in sc)
            assert abs(lse[i] - math.log(den)) <= 1e-13
            for c in range(4):
                num = math.fsum(math.exp(x) * v[j, c] for x, j in zip(sc, js))
                assert abs(o[i, c] - num / den) <= 1e-13 * max(1.0, abs(num / den))


def check_attn_library(att):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(54)
    q = rng.normal(size=(2, 3, 17, 32)); k = rng.normal(size=(2, 3, 23, 32)); v = rng.normal(size=(2, 3, 23, 32))
    for causal in (False, True):
        o, _ = att(q, k, v, causal=causal)
        tq, tk, tv = (torch.from_numpy(a) for a in (q, k, v))
        if causal:   # torch's is_causal aligns to the top-left; build the bottom-right mask
            L, S = 17, 23
            mask = torch.ones(L, S, dtype=torch.bool).tril(diagonal=S - L)
            t = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
        else:
            t = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
        assert np.max(np.abs(o - t.numpy())) <= 1e-12


ATTENTION_CHECKS = [check_attn_uniform_scores, check_attn_one_hot, check_attn_causal_first_row,
                    check_attn_brute_force, check_attn_library]


@pytest.mark.parametrize("check", ATTENTION_CHECKS, ids=lambda c: c.__name__)
def test_attention_pins(check):
    check(oracle.attention)
