"""The attention parity bound is tight enough to catch tile-sized mistakes (CPU only).

``gpu_helpers.attention_reference`` bounds |O - O_oracle| per element from the
kernel's arithmetic.  Here the kernel's rounding steps are emulated in numpy
(fp32 scores, p rounded to bf16 for the second product, l summed in fp32),
which must stay inside the bound, and mistakes the size of one key tile are
planted in copies of the oracle's inputs -- one V tile shifted by a key, the
last 64 columns of a V tile reversed (a swizzle slip), one K tile dropped --
each of which must leave it.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import attention_reference


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even), returned as fp32."""
    u = a.astype(np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


@pytest.fixture(scope="module", params=[False, True], ids=["unmasked", "causal"])
def case(request):
    causal = request.param
    w = workloads.ATTENTION_WORKLOADS["attn"].with_shape(2, 256, 640, 128, causal)
    q, k, v = (_f64(a) for a in workloads.attention_inputs(w))
    o, lse, bound = attention_reference(q, k, v, causal)
    return q, k, v, causal, o, bound


def test_emulated_kernel_rounding_stays_inside(case):
    q, k, v, causal, o, bound = case
    L, S, d = q.shape[1], k.shape[1], q.shape[2]
    s = (q.astype(np.float32) @ k.astype(np.float32).transpose(0, 2, 1)) * np.float32(1 / np.sqrt(d))
    if causal:
        s = np.where(np.arange(S)[None, :] > np.arange(L)[:, None] + (S - L), -np.inf, s)
    p = np.exp((s - s.max(-1, keepdims=True)).astype(np.float64)).astype(np.float32)
    l = p.sum(-1, keepdims=True, dtype=np.float32)
    o_kernel = (_bf16_round(p) @ v.astype(np.float32)) / l
    assert np.all(np.abs(o_kernel - o) <= bound)


@pytest.mark.parametrize("slip", ["v_tile_shift", "v_swizzle", "k_tile_dropped"])
def test_tile_mistakes_leave_the_bound(case, slip):
    q, k, v, causal, o, bound = case
    t = slice(384, 512)                                   # the fourth key tile of 128
    k2, v2 = k.copy(), v.copy()
    if slip == "v_tile_shift":
        v2[:, t] = np.roll(v[:, t], 1, axis=1)
    elif slip == "v_swizzle":
        v2[:, t, 64:] = v[:, t, 64:][:, :, ::-1]
    else:
        k2[:, t] = -1e4                                   # that tile's keys get no weight
    bad, _ = oracle.attention(q, k2, v2, causal=causal)
    ok = ~np.isnan(o).any(axis=-1)
    assert np.max((np.abs(bad - o) / bound)[ok]) > 10.0
