"""The committed ncu summaries against the traffic formula.

The fused kernels read each element of x once: a capture's DRAM reads must
be the bytes of x (4 M N), not the naive five-step algorithm's several
passes.  Writes are not checked: an isolated launch leaves part of y dirty
in the L2 when it ends.  The figures come from the text summaries under
profiles/ (one ncu capture each, the command inside), so this runs on CPU.
"""
from __future__ import annotations

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# summary file, bytes of x, the reads allowed above them (fraction)
CASES = [
    ("softmax_row_regs_c2.md", 4 * 8192 * 1024, 0.01),
    ("softmax_cluster_c3.md", 4 * 4096 * 32768, 0.01),
    ("softmax_staged_grid_c5.md", 4 * 32 * 1048576, 0.01),
    ("row_reduce_rows_c3.md", 4 * 4096 * 32768, 0.01),
    ("gelu_kernel_gelu_16k.md", 4 * 16384 * 16384, 0.01),
    # the column band kernel reads x twice, the second time mostly from the L2
    ("softmax_cols_band_cols_c4.md", 4 * 4096 * 16384, 0.15),
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
