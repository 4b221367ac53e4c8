"""Seeded synthetic inputs shaped like the lecture pages' softmax / row-sum workloads.

This module only draws random numbers.  It holds none of the softmax or
row-sum arithmetic, so it can feed both the float64 oracle (``oracle/``) and
the CUDA path (``row_reduction_softmax_gb300``) without coupling them: the two
sides see bit-identical fp32 inputs because they are generated here, once.

Every row is drawn from its own stream, keyed by ``(seed, row)`` through
numpy's ``SeedSequence`` -> ``PCG64``.  A single row of a full-size matrix can
therefore be regenerated on its own, which is how full-size parity tests
compare sampled rows against the oracle without rebuilding the whole matrix.

The five named workloads follow the configurations the pages' methods are
measured on (fp32, contiguous row-major, ``ld == N``):

=====  ===============  ===========================================================
name   M x N            values
=====  ===============  ===========================================================
c1     128 x 256        Normal(0, 1)
c2     8192 x 1024      Normal(0, 2^2)                 (row fits one block)
c3     4096 x 32768     Uniform(-8, 8)                 (row overflows one block)
c4     16384 x 4096     Normal(0, 3^2); per row round(0.05 N) positions = +50 and
                        round(0.01 N) other positions = -inf (never a whole row)
c5     32 x 1048576     Normal(0, 1)                   (fewer rows than SMs)
=====  ===============  ===========================================================
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "VARIANT_WORKLOADS", "AttentionWorkload", "ATTENTION_WORKLOADS",
           "row_values", "matrix", "spike_mask_counts", "to_bf16_bits", "attention_inputs"]


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    dist: str  # "normal" | "uniform" | "logits"
    seed: int
    sigma: float = 1.0
    lo: float = 0.0
    hi: float = 0.0
    spike: float = 50.0
    spike_frac: float = 0.0
    mask_frac: float = 0.0
    ops: tuple = field(default=("softmax",))

    def with_shape(self, M: int, N: int) -> "Workload":
        """Same value recipe and seed at another shape (small parity cases)."""
        return Workload(self.name, M, N, self.dist, self.seed, self.sigma, self.lo,
                        self.hi, self.spike, self.spike_frac, self.mask_frac, self.ops)

    @property
    def elements(self) -> int:
        return self.M * self.N


WORKLOADS = {
    "c1": Workload("c1", 128, 256, "normal", seed=0, sigma=1.0),
    "c2": Workload("c2", 8192, 1024, "normal", seed=1, sigma=2.0),
    "c3": Workload("c3", 4096, 32768, "uniform", seed=2, lo=-8.0, hi=8.0,
                   ops=("softmax", "row_sum")),
    "c4": Workload("c4", 16384, 4096, "logits", seed=3, sigma=3.0, spike=50.0,
                   spike_frac=0.05, mask_frac=0.01),
    "c5": Workload("c5", 32, 1048576, "normal", seed=4, sigma=1.0),
}


# Workloads of the variants built on the same skeleton (the pages give no
# sizes for them; these reuse the recipes above at shapes of the same size):
# the column softmax on c2's and c4's values with the long axis down the
# columns, and the elementwise GeLU on a 16384 x 16384 Normal(0, 1) matrix,
# the "16,384-dim" input of the pages' GeLU benchmark.
VARIANT_WORKLOADS = {
    "cols_c2": Workload("cols_c2", 1024, 8192, "normal", seed=1, sigma=2.0, ops=("softmax_cols",)),
    "cols_c4": Workload("cols_c4", 4096, 16384, "logits", seed=3, sigma=3.0, spike=50.0,
                        spike_frac=0.05, mask_frac=0.01, ops=("softmax_cols",)),
    "gelu_16k": Workload("gelu_16k", 16384, 16384, "normal", seed=6, sigma=1.0, ops=("gelu",)),
}


def _rng(seed: int, row: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(row)])))


def spike_mask_counts(N: int, spike_frac: float, mask_frac: float) -> tuple[int, int]:
    """Per-row counts of +spike and -inf positions; at least one entry stays finite."""
    k_spike = int(round(spike_frac * N))
    k_mask = int(round(mask_frac * N))
    k_spike = min(k_spike, N)
    k_mask = min(k_mask, max(N - 1, 0))          # never mask a whole row
    if k_spike + k_mask > N:
        k_spike = N - k_mask
    return k_spike, k_mask


def row_values(w: Workload, row: int) -> np.ndarray:
    """fp32 values of row ``row`` of workload ``w`` (length ``w.N``)."""
    g = _rng(w.seed, row)
    N = w.N
    if w.dist == "normal":
        v = g.standard_normal(N, dtype=np.float32) * np.float32(w.sigma)
    elif w.dist == "uniform":
        v = g.random(N, dtype=np.float32) * np.float32(w.hi - w.lo) + np.float32(w.lo)
    elif w.dist == "logits":
        v = g.standard_normal(N, dtype=np.float32) * np.float32(w.sigma)
        k_spike, k_mask = spike_mask_counts(N, w.spike_frac, w.mask_frac)
        if k_spike + k_mask:
            pos = g.choice(N, size=k_spike + k_mask, replace=False)
            v[pos[:k_spike]] = np.float32(w.spike)
            v[pos[k_spike:]] = -np.inf
    else:
        raise ValueError(f"unknown distribution {w.dist!r}")
    return v.astype(np.float32, copy=False)


def matrix(w: Workload, ld: int | None = None, rows=None, pad_value=np.nan,
           out: np.ndarray | None = None) -> np.ndarray:
    """Rows of ``w`` as a ``(len(rows), ld)`` fp32 array.

    Columns ``[N, ld)`` (the leading-dimension gap) are filled with
    ``pad_value`` (NaN by default) so that a kernel that reads past ``N``
    poisons its row instead of passing silently.
    """
    ld = w.N if ld is None else int(ld)
    if ld < w.N:
        raise ValueError("ld < N")
    rows = range(w.M) if rows is None else rows
    rows = list(rows)
    if out is None:
        out = np.empty((len(rows), ld), dtype=np.float32)
    if ld > w.N:
        out[:, w.N:] = pad_value
    for i, r in enumerate(rows):
        out[i, :w.N] = row_values(w, r)
    return out



# ------------------------------------------------------------- attention ----

@dataclass(frozen=True)
class AttentionWorkload:
    """Q, K, V of B x H heads: [B*H, L, d] and [B*H, S, d], Normal(0, 1), bf16."""
    name: str
    B: int
    H: int
    L: int
    S: int
    d: int
    causal: bool
    seed: int

    @property
    def BH(self) -> int:
        return self.B * self.H

    def with_shape(self, BH: int, L: int, S: int, d: int, causal: bool) -> "AttentionWorkload":
        return AttentionWorkload(self.name, 1, BH, L, S, d, causal, self.seed)


# The pages give no attention sizes; this is a common training shape for a
# 128-wide head (B = 4 sequences of 4096 tokens, 16 heads), both unmasked and
# causal.
ATTENTION_WORKLOADS = {
    "attn": AttentionWorkload("attn", 4, 16, 4096, 4096, 128, False, 7),
    "attn_causal": AttentionWorkload("attn_causal", 4, 16, 4096, 4096, 128, True, 8),
}


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounding to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(a, dtype=np.float32))
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def attention_inputs(w: AttentionWorkload, heads=None):
    """(q, k, v) as bf16 bit patterns (uint16 arrays) for the heads listed
    (all by default).  Each head is drawn from its own stream keyed by
    (seed, head, tensor), so one head can be regenerated alone."""
    hs = range(w.BH) if heads is None else heads
    out = []
    for t, n in enumerate((w.L, w.S, w.S)):
        arr = np.empty((len(hs), n, w.d), dtype=np.uint16)
        for i, h in enumerate(hs):
            g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, int(h), t])))
            arr[i] = to_bf16_bits(g.standard_normal((n, w.d), dtype=np.float32))
        out.append(arr)
    return tuple(out)
