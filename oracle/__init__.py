"""Float64 CPU oracle for the row-wise softmax, the row sum and their variants.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` do.  It shares no code with the
CUDA path; the only thing both sides take from a common place is their seeded
input (``workloads``), which holds none of this arithmetic.

Everything here is plain numpy in float64, written to be checked against the
lecture pages by eye, with no blocking, fusion or reordering beyond what the
pages state.  Sources (page title, then section):

* "Kernels, Triton, XLA" (CS336 lecture 06 notes), section "Reductions and
  tiling: softmax, row sum, matmul": the naive softmax is max per row,
  subtract, exponentiate, sum, divide; masked lanes load -inf, the softmax
  equivalent of zero; the row sum sweeps tiles into a per-thread accumulator
  vector and reduces it to a scalar at the end (masked lanes load 0).
* "Chapter 7: GPU High-Performance Programming", section 7.5.1 "Triton
  Implementation of Softmax" and "Triton Implementation of Row Sum".
* The lecture transcript (English captions, 01:06:17-01:08:46): the worked
  row-sum trace 3,1,4,1 | 5,9,2,6 | 5,3 with four per-thread accumulators.

Where the pages are silent the oracle takes these readings:

* A row that is entirely -inf has no finite maximum; the naive steps give
  (-inf) - (-inf) = NaN, so the whole output row is NaN.  The same holds for
  rows holding +inf or NaN.
* The split-row merge of partial (max, sum) pairs is not on the pages; it is
  derived from the definition s = sum_j exp(x_j - m): for disjoint segments a,
  b with partials (m_a, s_a), (m_b, s_b), m = max(m_a, m_b) and
  s = s_a exp(m_a - m) + s_b exp(m_b - m), identity (-inf, 0), and a segment
  whose max is -inf contributes 0 (never exp(-inf - -inf)).
* The log-softmax is not on the pages.  It is read as the logarithm of their
  softmax: log(exp(x - m) / s) = (x - m) - log(s).  -inf entries give -inf;
  the rows that give NaN in the softmax give NaN.
* The row max is the first of the naive softmax's five steps; the row mean is
  the row sum divided by N.  An empty row has max -inf (the max's identity)
  and mean NaN (0 / 0).
* The column softmax (a softmax down each column, over the rows) is the
  pages' softmax with rows and columns exchanged; the lecture transcript's
  question after the softmax kernel asks for it, and the answer is the same
  computation with the strides swapped (transcript, the softmax kernel's
  Q&A).

* GeLU is the tanh approximation the pages implement three ways ("Kernels,
  Triton, XLA", section "GeLU three ways: the case for fusion"; "GPU
  High-Performance Programming", section 7.4.1), with the constants as
  printed there: 0.5 x (1 + tanh(0.79788456 (x + 0.044715 x^3))).

* Attention is named, not defined, by the pages: the ingredients above
  (elementwise, row-wise reduction, tiled reduction, tiled matmul) are what a
  FlashAttention kernel fuses ("Kernels, Triton, XLA", end of "Reductions
  and tiling"; "CS336 2026 Lecture 6: Kernels, Triton", the assignment
  paragraph and the summary).  The reading taken is scaled dot-product
  attention per head, O = softmax(Q K^T * scale) V with the row softmax
  above over the keys, optionally causal (key j > query i masked with -inf,
  the softmax's zero), and LSE = m + log(s) per query row.

Pins (see ``tests/test_oracle_pins.py``): every function here is checked
against values the pages print or the mathematics fixes, never against itself.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "softmax_rows",
    "row_sum",
    "row_sum_tiles",
    "partial",
    "merge",
    "softmax_rows_split",
    "log_softmax_rows",
    "row_max",
    "row_mean",
    "softmax_cols",
    "gelu",
    "attention",
]


def _as_rows(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    if a.ndim == 1:
        a = a[None, :]
    if a.ndim != 2:
        raise ValueError("expected an M x N matrix")
    return a


def softmax_rows(x) -> np.ndarray:
    """Row-wise softmax of an M x N matrix, in float64.

    The five steps of the naive version on "Kernels, Triton, XLA", section
    "Reductions and tiling" (and section 7.5.1 of "GPU High-Performance
    Programming"): (1) max of each row, (2) subtract it, (3) exponentiate,
    (4) sum each row, (5) divide.  exp(-inf - m) is exactly 0, which is why
    the pages load masked lanes as -inf.
    """
    a = _as_rows(x)
    if a.shape[1] == 0:
        return a.copy()
    with np.errstate(invalid="ignore", over="ignore"):
        m = np.max(a, axis=1, keepdims=True)          # (1) row max
        z = a - m                                       # (2) subtract
        numerator = np.exp(z)                           # (3) exponentiate
        denominator = np.sum(numerator, axis=1, keepdims=True)  # (4) row sum
        return numerator / denominator                  # (5) divide


def row_sum(x) -> np.ndarray:
    """Sum of each row of an M x N matrix, in float64 (the built-in row sum).

    "Kernels, Triton, XLA", section "Reductions and tiling", paragraph "Row
    sum, when the row doesn't fit": out[i] = sum_j x[i, j].  An empty row
    sums to 0, the value masked lanes load.
    """
    a = _as_rows(x)
    return np.sum(a, axis=1)


def row_sum_tiles(row, block: int):
    """The pages' tiled row sum, step by step, for one row.

    A vector of ``block`` per-thread accumulators starts at zero; each tile of
    ``block`` consecutive columns is loaded with lanes past the end of the row
    set to 0.0 and added element-wise; after the last tile the accumulators
    are summed to a scalar ("Kernels, Triton, XLA", section "Reductions and
    tiling"; the transcript's worked example at 01:07:32).

    Returns ``(trace, total)`` where ``trace[k]`` is the accumulator vector
    after tile ``k``.
    """
    r = np.asarray(row, dtype=np.float64).ravel()
    if block <= 0:
        raise ValueError("block must be positive")
    acc = np.zeros(block, dtype=np.float64)
    trace = []
    for start in range(0, r.size, block):
        tile = np.zeros(block, dtype=np.float64)        # masked lanes: 0.0
        chunk = r[start:start + block]
        tile[:chunk.size] = chunk
        acc = acc + tile
        trace.append(acc.copy())
    return trace, float(np.sum(acc))


def partial(segment) -> tuple[float, float]:
    """(max, sum of exp(x - max)) of one row segment; (-inf, 0) if empty or all -inf."""
    s = np.asarray(segment, dtype=np.float64).ravel()
    if s.size == 0:
        return (-np.inf, 0.0)
    m = float(np.max(s))
    if m == -np.inf:
        return (-np.inf, 0.0)
    with np.errstate(invalid="ignore"):
        return (m, float(np.sum(np.exp(s - m))))


def merge(a: tuple[float, float], b: tuple[float, float]) -> tuple[float, float]:
    """Merge two partials of disjoint segments (derived from the definition)."""
    m_a, s_a = a
    m_b, s_b = b
    m = max(m_a, m_b)
    if m == -np.inf:
        return (-np.inf, 0.0)
    t_a = 0.0 if m_a == -np.inf else s_a * float(np.exp(m_a - m))
    t_b = 0.0 if m_b == -np.inf else s_b * float(np.exp(m_b - m))
    return (m, t_a + t_b)


def softmax_rows_split(x, cuts) -> np.ndarray:
    """Softmax of each row computed from the partials of the segments ``cuts`` defines.

    ``cuts`` are interior column indices; each row is split there, every
    segment's partial is taken, the partials are merged left to right, and the
    row is normalised with the merged (max, sum).  It reaches the same result
    as :func:`softmax_rows` (up to rounding order); it exists to state the
    split-row rule in one place for the tests.
    """
    a = _as_rows(x)
    bounds = [0] + sorted(int(c) for c in cuts) + [a.shape[1]]
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        acc = (-np.inf, 0.0)
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            acc = merge(acc, partial(a[i, lo:hi]))
        m, s = acc
        with np.errstate(invalid="ignore", divide="ignore"):
            out[i] = np.exp(a[i] - m) / s if m != -np.inf else np.nan
    return out


def log_softmax_rows(x) -> np.ndarray:
    """Row-wise log-softmax of an M x N matrix, in float64.

    The logarithm of the pages' softmax ("Kernels, Triton, XLA", section
    "Reductions and tiling"), which the pages do not show: (1) max of each
    row, (2) subtract it, (3) exponentiate, (4) sum each row, (5) take the log
    of the sum, (6) subtract it from the shifted row: (x - m) - log(s).
    """
    a = _as_rows(x)
    if a.shape[1] == 0:
        return a.copy()
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        m = np.max(a, axis=1, keepdims=True)          # (1) row max
        z = a - m                                       # (2) subtract
        e = np.exp(z)                                   # (3) exponentiate
        s = np.sum(e, axis=1, keepdims=True)            # (4) row sum
        return z - np.log(s)                            # (5), (6)


def row_max(x) -> np.ndarray:
    """Max of each row, in float64: step (1) of the naive softmax on "Kernels,
    Triton, XLA", section "Reductions and tiling".  A row holding a NaN gives
    NaN; an empty row gives -inf."""
    a = _as_rows(x)
    if a.shape[1] == 0:
        return np.full(a.shape[0], -np.inf)
    return np.max(a, axis=1)


def row_mean(x) -> np.ndarray:
    """Mean of each row, in float64: the row sum ("Kernels, Triton, XLA",
    paragraph "Row sum, when the row doesn't fit") divided by N.  An empty row
    gives NaN."""
    a = _as_rows(x)
    if a.shape[1] == 0:
        return np.full(a.shape[0], np.nan)
    return np.sum(a, axis=1) / a.shape[1]


def softmax_cols(x) -> np.ndarray:
    """Softmax down each column of an M x N matrix (over the rows), in float64.

    The five naive steps with the reduction taken over i for every column j:
    (1) m_j = max_i x[i, j], (2) subtract, (3) exponentiate, (4) s_j = sum_i,
    (5) divide.  A column that is all -inf, or holds +inf or NaN, is NaN.
    """
    a = np.asarray(x, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("expected an M x N matrix")
    if a.shape[0] == 0:
        return a.copy()
    with np.errstate(invalid="ignore", over="ignore"):
        m = np.max(a, axis=0, keepdims=True)          # (1) column max
        z = a - m                                       # (2) subtract
        numerator = np.exp(z)                           # (3) exponentiate
        denominator = np.sum(numerator, axis=0, keepdims=True)  # (4) column sum
        return numerator / denominator                  # (5) divide


GELU_C = 0.79788456      # the pages' constant (sqrt(2 / pi) to 8 digits)
GELU_K = 0.044715


def gelu(x) -> np.ndarray:
    """GeLU, tanh approximation, elementwise in float64, as the pages write it
    ("Kernels, Triton, XLA", section "GeLU three ways"): the inner polynomial
    a = 0.79788456 (x + 0.044715 x^3), then 0.5 x (1 + tanh(a))."""
    a = np.asarray(x, dtype=np.float64)
    inner = GELU_C * (a + GELU_K * a * a * a)
    return 0.5 * a * (1.0 + np.tanh(inner))


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Scaled dot-product attention of one or more heads, in float64.

    q: (..., L, d), k and v: (..., S, d).  Steps: (1) scores = q k^T * scale
    (a library matmul), (2) causal: scores[i, j] = -inf for j > i + (S - L)
    (queries aligned to the last keys), (3) P = softmax_rows(scores), the
    pinned row softmax, (4) O = P v.  Returns (O, LSE) with LSE the log of
    the row sum of exp(scores) (m + log s), -inf for an all-masked row.
    scale defaults to 1 / sqrt(d).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, d = q.shape[-2], q.shape[-1]
    S = k.shape[-2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    scores = np.matmul(q, np.swapaxes(k, -1, -2)) * scale          # (1)
    if causal:                                                        # (2)
        i = np.arange(L)[:, None]
        j = np.arange(S)[None, :]
        scores = np.where(j > i + (S - L), -np.inf, scores)
    flat = scores.reshape(-1, S)
    p = softmax_rows(flat).reshape(scores.shape)                      # (3)
    out = np.matmul(p, v)                                             # (4)
    with np.errstate(divide="ignore", invalid="ignore"):
        m = np.max(flat, axis=1)
        lse = m + np.log(np.sum(np.exp(flat - m[:, None]), axis=1))
    return out, lse.reshape(scores.shape[:-1])
