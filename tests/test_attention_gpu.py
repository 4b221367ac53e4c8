"""GPU parity of the fused attention forward against the float64 oracle.

Inputs are bf16 (the generator rounds Normal(0, 1) draws to bf16, and the
oracle takes the same bf16 values in float64).  Tolerances, derived from the
kernel's arithmetic (``gpu_helpers.attention_reference``): per element,
|O - O_ref| <= 2^-8 sum_j p_j |v_jc| (p rounded to bf16, 8 significant
bits, for the second product; l summed in fp32) plus the fp32 error of the scores and of the two
sums over keys, plus 1e-6.  LSE is m + log l in fp32: |LSE - LSE_ref| <=
1e-5 * max(1, |LSE_ref|) + 1e-5.
"""
from __future__ import annotations


import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import attention_reference

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LSE_TOL = 1e-5


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_dev(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def check(o, lse, q, k, v, causal, where, heads=None, rows=None, scale=None):
    qf, kf, vf = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    want_o, want_lse, bound = attention_reference(qf, kf, vf, causal, scale)
    if rows is not None:
        want_o, want_lse, bound = want_o[:, rows], want_lse[:, rows], bound[:, rows]
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    nan_rows = np.isnan(want_o).any(axis=-1)
    assert np.all(np.isnan(o[nan_rows])), f"{where}: rows that see no key must be NaN"
    assert np.all(np.isneginf(lse[nan_rows])), f"{where}: their LSE must be -inf"
    ok = ~nan_rows
    err = np.abs(o - want_o)
    assert np.all(err[ok] <= bound[ok]), \
        f"{where}: max |dO| {float(np.max(err[ok])):.3e}, max |dO| / bound {float(np.max(err[ok] / bound[ok])):.3f}"
    lerr = np.abs(lse[ok] - want_lse[ok])
    assert np.all(lerr <= LSE_TOL * np.maximum(1.0, np.abs(want_lse[ok])) + LSE_TOL), \
        f"{where}: max |dLSE| {float(np.max(lerr)):.3e}"
    return float(np.max(err[ok])) if ok.any() else 0.0


SHAPES = [  # (BH, L, S, d, causal)
    (1, 128, 128, 64, False), (1, 128, 128, 128, False), (2, 128, 256, 128, False),
    (3, 256, 128, 64, False), (1, 200, 300, 64, False), (2, 131, 77, 128, False),
    (1, 1, 1, 64, False), (2, 5, 1000, 128, False), (1, 128, 128, 64, True),
    (3, 256, 256, 128, True), (2, 300, 300, 64, True), (1, 5, 1000, 128, True),
    (1, 1000, 5, 64, True), (4, 512, 512, 128, False), (2, 384, 640, 128, True),
]


@pytest.mark.parametrize("BH,L,S,d,causal", SHAPES)
def test_attention_parity(lib, BH, L, S, d, causal):
    w = workloads.ATTENTION_WORKLOADS["attn"].with_shape(BH, L, S, d, causal)
    q, k, v = workloads.attention_inputs(w)
    o, lse = rrs.attention(to_dev(q), to_dev(k), to_dev(v), causal=causal)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check(o.cpu().numpy(), lse.cpu().numpy(), q, k, v, causal, f"{BH}x{L}x{S}x{d} causal={causal}")


def test_attention_scale_and_repeat(lib):
    w = workloads.ATTENTION_WORKLOADS["attn"].with_shape(2, 256, 384, 64, False)
    q, k, v = workloads.attention_inputs(w)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    o1, l1 = rrs.attention(tq, tk, tv, scale=0.05)
    o2, l2 = rrs.attention(tq, tk, tv, scale=0.05)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)          # deterministic
    check(o1.cpu().numpy(), l1.cpu().numpy(), q, k, v, False, "scale 0.05", scale=0.05)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_scores_rising_across_key_tiles(lib, causal):
    """Scores that grow by hundreds (log2 units) from one key tile to the
    next: p against the first tile's reference would overflow, so every later
    tile must move the reference and rescale O -- the same softmax."""
    BH, L, S, d = 2, 256, 640, 64
    rng = np.random.default_rng(41)
    q = np.ones((BH, L, d), dtype=np.float32) * rng.uniform(0.5, 1.0, size=(BH, L, 1)).astype(np.float32)
    ramp = (np.arange(S, dtype=np.float32) / S * 40.0)[None, :, None]   # up to 40 per component:
    # the max score rises by about 90 log2 units per key tile
    k = np.broadcast_to(ramp, (BH, S, d)) + rng.normal(0, 0.05, size=(BH, S, d)).astype(np.float32)
    v = rng.normal(0, 1, size=(BH, S, d)).astype(np.float32)
    qb, kb, vb = (workloads.to_bf16_bits(a) for a in (q, k, v))
    o, lse = rrs.attention(to_dev(qb), to_dev(kb), to_dev(vb), causal=causal)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check(o.cpu().numpy(), lse.cpu().numpy(), qb, kb, vb, causal, f"rising scores causal={causal}")


def test_attention_rejects_bad_arguments(lib):
    q = torch.zeros(1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rrs.RRSError) as e:
        rrs.attention(q, q, q)                                     # d = 96
    assert e.value.status == 1
    q = torch.zeros(1, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(1, 128, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(rrs.RRSError) as e:                         # o overlaps q
        rrs.attention_ptr(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 0, 1, 128, 128, 64)
    assert e.value.status == 2
    rrs.attention_ptr(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 0, 128, 128, 64)


@pytest.mark.parametrize("name", ["attn", "attn_causal"])
def test_full_size_attention_sampled(lib, name):
    w = workloads.ATTENTION_WORKLOADS[name]
    q, k, v = workloads.attention_inputs(w)
    o, lse = rrs.attention(to_dev(q), to_dev(k), to_dev(v), causal=w.causal)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    rng = np.random.default_rng(w.seed)
    heads = sorted({0, w.BH - 1, *rng.choice(w.BH, size=4, replace=False).tolist()})
    rows = sorted({0, w.L - 1, w.L // 2, *rng.choice(w.L, size=12, replace=False).tolist()})
    got_o = o[heads][:, rows].cpu().numpy()
    got_l = lse[heads][:, rows].cpu().numpy()
    check(got_o, got_l, q[heads], k[heads], v[heads], w.causal, f"{name} sampled", rows=rows)
    assert bool(torch.isfinite(o).all())
    del o, lse
    torch.cuda.empty_cache()
