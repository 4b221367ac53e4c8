"""The committed ncu summaries against the traffic formula.

The fused kernels read each element of x once and write each element of y
once: a capture's DRAM reads must be the bytes of x (4 M N), not the naive
five-step algorithm's several passes.  Writes are checked on the
steady-state captures (back-to-back launches, caches not flushed, so each
launch pays the write-back its predecessor left in the L2): the L2 write
sectors must be exactly the bytes of y and the DRAM writes nearly so.  An
isolated launch (the full section sets) leaves part of y dirty in the L2,
so its DRAM writes are not checked.  The figures come from the text
summaries under profiles/ (the commands inside), so this runs on CPU.
"""
from __future__ import annotations

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# summary file, bytes of x, the reads allowed above them (fraction)
CASES = [
    ("softmax_row_regs_c2.md", 4 * 8192 * 1024, 0.01),
    ("softmax_row_regs_c4.md", 4 * 16384 * 4096, 0.01),
    ("softmax_cluster_c3.md", 4 * 4096 * 32768, 0.01),
    ("softmax_staged_grid_c5.md", 4 * 32 * 1048576, 0.01),
    ("row_reduce_rows_c3.md", 4 * 4096 * 32768, 0.01),
    ("gelu_kernel_gelu_16k.md", 4 * 16384 * 16384, 0.01),
    # the column kernels read x twice, the second time mostly from the L2
    ("softmax_cols_two_pass_cols_c4.md", 4 * 4096 * 16384, 0.15),
    ("softmax_cols_band_cols_c2.md", 4 * 1024 * 8192, 0.15),
]


def dram_read_bytes(name: str) -> float:
    with open(os.path.join(ROOT, "profiles", name)) as f:
        text = f.read()
    m = re.search(r"\| dram__bytes_read\.sum \| ([0-9.]+) MB \|", text)
    assert m, f"{name}: no dram__bytes_read line"
    return float(m.group(1)) * 1e6


@pytest.mark.parametrize("name,x_bytes,slack", CASES)
def test_each_element_of_x_is_read_once(name, x_bytes, slack):
    got = dram_read_bytes(name)
    assert x_bytes * (1 - 0.01) <= got <= x_bytes * (1 + slack), \
        f"{name}: {got / 1e6:.2f} MB read from DRAM for {x_bytes / 1e6:.2f} MB of x"



def steady(name: str) -> dict:
    with open(os.path.join(ROOT, "profiles", name)) as f:
        text = f.read()
    out = {}
    for key, pat in [("read", r"\| steady dram__bytes_read\.sum \| ([0-9.]+) MB \|"),
                     ("write", r"\| steady dram__bytes_write\.sum \| ([0-9.]+) MB \|"),
                     ("l2_write", r"\| steady L2 write sectors x 32 B[^|]*\| ([0-9.]+) MB \|")]:
        m = re.search(pat, text)
        assert m, f"{name}: no steady {key} line"
        out[key] = float(m.group(1)) * 1e6
    # optional: the global-store sectors leaving the SMs (no local-memory spill stores)
    m = re.search(r"\| steady global store sectors x 32 B[^|]*\| ([0-9.]+) MB \|", text)
    if m:
        out["global_st"] = float(m.group(1)) * 1e6
    return out


# summary file, bytes of x, bytes of y written (the softmax writes M N floats,
# the row sum M), the DRAM writes expected at least (fraction of y: 32 MiB of
# y partly stay dirty in the L2 between the bench's launches), the reads
# allowed above the bytes of x (fraction: the column and row two-pass kernels
# re-read x, the second time mostly from the L2), and the L2 write sectors allowed above the
# bytes of y (fraction: a kernel that spills registers sends its
# local-memory stores to the L2 too; where a summary gives the global-store
# sectors, those are checked to be exactly y)
STEADY = [
    ("softmax_cluster_c3.md", 4 * 4096 * 32768, 4 * 4096 * 32768, 0.99, 0.01, 0.001),
    ("softmax_row_regs_c2.md", 4 * 8192 * 1024, 4 * 8192 * 1024, 0.9, 0.01, 0.001),
    ("softmax_row_regs_c4.md", 4 * 16384 * 4096, 4 * 16384 * 4096, 0.97, 0.01, 0.001),
    ("softmax_staged_grid_c5.md", 4 * 32 * 1048576, 4 * 32 * 1048576, 0.95, 0.01, 0.001),
    ("row_reduce_rows_c3.md", 4 * 4096 * 32768, 4 * 4096, 0.0, 0.01, 0.001),
    ("softmax_cols_two_pass_cols_c4.md", 4 * 4096 * 16384, 4 * 4096 * 16384, 0.97, 0.10, 0.01),
    ("softmax_cols_band_cols_c2.md", 4 * 1024 * 8192, 4 * 1024 * 8192, 0.85, 0.10, 0.001),
    ("softmax_rows_two_pass_c5.md", 4 * 32 * 1048576, 4 * 32 * 1048576, 0.97, 0.15, 0.001),
    ("gelu_kernel_gelu_16k.md", 4 * 16384 * 16384, 4 * 16384 * 16384, 0.99, 0.01, 0.001),
]


@pytest.mark.parametrize("name,x_bytes,y_bytes,min_write,read_slack,l2_extra", STEADY)
def test_steady_state_reads_x_once_and_writes_y_once(name, x_bytes, y_bytes, min_write, read_slack, l2_extra):
    st = steady(name)
    assert 0.98 * x_bytes <= st["read"] <= (1 + read_slack) * x_bytes, f"{name}: {st['read'] / 1e6:.2f} MB read"
    # every store lands in the L2 once: the sectors written are the bytes of y
    # (plus, where allowed, register spill stores)
    assert y_bytes - max(0.001 * y_bytes, 0.2e6) <= st["l2_write"] <= y_bytes + max(l2_extra * y_bytes, 0.2e6), \
        f"{name}: {st['l2_write'] / 1e6:.2f} MB"
    if "global_st" in st:
        assert abs(st["global_st"] - y_bytes) <= max(0.001 * y_bytes, 0.2e6), f"{name}: {st['global_st'] / 1e6:.2f} MB"
    assert min_write * y_bytes <= st["write"] <= 1.01 * y_bytes + 2e6, f"{name}: {st['write'] / 1e6:.2f} MB"


def test_two_phase_reads_x_at_most_twice():
    """The fallback split path re-reads x; the capture shows how much of the
    re-read the L2 serves: between 8 and 12 bytes per element per call."""
    with open(os.path.join(ROOT, "profiles", "softmax_two_phase_c5.md")) as f:
        text = f.read()
    rd = float(re.search(r"\| steady dram__bytes_read\.sum \| [0-9.]+ MB \| [0-9.]+ MB \| ([0-9.]+) MB \|", text).group(1))
    wr = float(re.search(r"\| steady dram__bytes_write\.sum \| [0-9.]+ MB \| [0-9.]+ MB \| ([0-9.]+) MB \|", text).group(1))
    per_element = (rd + wr) * 1e6 / (32 * 1048576)
    assert 8.0 <= per_element <= 12.5, per_element


def test_every_profiled_kernel_has_its_sources_listed():
    """Each kernel with a committed traffic figure is keyed to its own
    sources (the bench falls back to hashing all of csrc/ otherwise, which
    would drop every figure on any change), and those files exist."""
    import bench
    csrc = os.path.join(ROOT, "row_reduction_softmax_gb300", "csrc")
    for names in bench.KERNEL_SOURCES.values():
        for n in names + bench.COMMON_SOURCES:
            assert os.path.exists(os.path.join(csrc, n)), n
    pat = re.compile(r"traffic:\s+kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=(\d+)\s+source=(\w+)")
    seen = 0
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                m = pat.search(line)
                if m:
                    seen += 1
                    assert m.group(1) in bench.KERNEL_SOURCES, f"{name}: {m.group(1)} has no source list"
    assert seen >= 6


def test_every_traffic_figure_is_for_the_current_sources(lib):
    """Each committed traffic line is keyed to its kernel's sources, the
    shared device headers and the launch plan of its workload on a GB300
    (152 SMs, 227 KB of shared memory per CTA): a kernel changed since its
    counters were taken fails here until they are taken again."""
    import bench
    import row_reduction_softmax_gb300 as rrs
    import workloads
    pat = re.compile(r"traffic:\s+kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=(\d+)\s+source=(\w+)")
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                m = pat.search(line)
                if not m:
                    continue
                kernel, wl, _, source = m.groups()
                plan = None
                if wl in workloads.WORKLOADS:
                    w = workloads.WORKLOADS[wl]
                    planner = rrs.plan_row_sum if kernel == "row_reduce_rows_kernel" else rrs.plan_softmax
                    plan = planner(w.M, w.N, w.N, True, 152, 232448)
                elif kernel.startswith("softmax_cols_"):
                    w = workloads.VARIANT_WORKLOADS[wl]
                    plan = rrs.plan_softmax_cols(w.M, w.N, w.N, True, 152, 232448)
                assert bench.source_hash(kernel, plan) == source, f"{name}: {kernel} changed since its capture"
