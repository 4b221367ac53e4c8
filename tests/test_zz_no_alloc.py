"""softmax_rows_noalloc: the entry point for callers that cannot allocate device memory.

Callers such as an inference engine's plugin execute hook (the engine owns all
device memory) or a latency-critical loop (an allocation could synchronise the
device or fail mid-step) may not call cudaMalloc.  softmax_rows_noalloc keeps
its partials in a fixed array inside the library instead.  These tests call it
through the C ABI twice in a row -- on different inputs, so a stale scratch
would show -- and check each result against softmax_rows on the same input,
with the tolerances every softmax test here uses.  This file is collected
last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import ABS_TOL, ROW_SUM_TOL, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

INVALID = 1


def _call_noalloc(lib, x, y, M, N, ld):
    return lib.softmax_rows_noalloc(x.data_ptr(), y.data_ptr(), M, N, ld,
                                    torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,M,N", [("c5", 32, 1 << 20), ("c4", 300, 4096), ("c3", 7, 40003)])
def test_noalloc_matches_softmax_rows_twice(lib, name, M, N):
    rrs.force_path("auto", "auto")
    w = workloads.WORKLOADS[name].with_shape(M, N)
    inputs = [workloads.matrix(w)]
    inputs.append(np.flip(inputs[0], axis=0).copy() * np.float32(0.5))   # a different second input
    for x_host in inputs:                                                  # two calls in a row
        x = torch.from_numpy(x_host).cuda()
        y_ref = torch.empty_like(x)
        y = torch.full_like(x, float("nan"))
        lib_status = lib.softmax_rows(x.data_ptr(), y_ref.data_ptr(), M, N, N,
                                      torch.cuda.current_stream().cuda_stream)
        assert lib_status == 0
        assert _call_noalloc(lib, x, y, M, N, N) == 0
        torch.cuda.synchronize()
        diff = (y.double() - y_ref.double()).abs().max().item()
        assert diff <= ABS_TOL, diff
        assert (y.double().sum(dim=1) - 1.0).abs().max().item() <= ROW_SUM_TOL
        rows = [0, M // 2, M - 1]
        check_softmax(y[rows].cpu().numpy(), x_host[rows], f"noalloc {name}")


def test_noalloc_rejects_too_many_rows_without_launching(lib):
    x = torch.zeros(131073, 4, device="cuda")
    y = torch.empty_like(x)
    assert _call_noalloc(lib, x, y, 131073, 4, 4) == INVALID
    assert _call_noalloc(lib, x, y, 0, 4, 4) == 0                       # nothing to do
    assert _call_noalloc(lib, x, x, 4, 4, 4) == 2                       # x and y overlap
