"""Failure detection on the GPU, without faulting it.

The split-row GRID path waits for the partials of other CTAs.  Every such
wait is bounded (about a second): when it runs out, the kernel records the
failure in a device error word and returns, and the host reads the status.
Here the failure is made on purpose from the host -- rrs_inject_fault makes
one CTA skip publishing a partial, a flag nothing else sets -- and the test
checks the reported status and that the context is still usable.
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIMEOUT = 4


def test_grid_wait_runs_out_and_is_reported(lib):
    path = "grid"
    M, N = 4, 65536
    x_host = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(M, N))
    x = torch.from_numpy(x_host).cuda()
    y = torch.empty_like(x)
    try:
        rrs.force_path(path)
        assert rrs.device_error() == 0
        assert lib.rrs_inject_fault(1) == 0
        rrs.softmax_rows(x, y)                      # the launch itself succeeds
        assert rrs.device_error() == TIMEOUT         # ... and its waits ran out
        assert rrs.device_error() == 0               # the word was cleared
    finally:
        lib.rrs_inject_fault(0)
        rrs.force_path("auto", "auto")
    # the context is still usable and results are right again
    rrs.force_path(path)
    try:
        rrs.softmax_rows(x, y)
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax(y.cpu().numpy(), x_host, "after an injected timeout")
    finally:
        rrs.force_path("auto", "auto")
