"""CUDA graphs: the hot-path calls captured once and replayed.

A caller that captures softmax_rows or row_sum in a CUDA graph replays the
same kernel arguments every time.  The split-row grid path draws a fresh
ticket for every launch on the device, so a replay never takes a (max, sum)
partial left by the previous replay for one of its own; to show it, x changes
between replays (a stale partial would then give a wrong row).  Each path's
first call runs before the capture: it allocates the path's workspace (and
the grid path's host error word), which a capture may not do.
"""
from __future__ import annotations

import numpy as np
import pytest

import row_reduction_softmax_gb300 as rrs
import workloads
from gpu_helpers import check_every_row, check_row_sum, check_softmax

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_path(lib):
    rrs.force_path("auto", "auto")
    yield
    rrs.force_path("auto", "auto")


def _plan_path(M, N):
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return rrs.plan_softmax(M, N, N, True, props.multi_processor_count,
                            props.shared_memory_per_block_optin)["path_name"]


@pytest.mark.parametrize("name,M,N,path", [("c1", 128, 256, "row_regs"), ("c3", 8, 32768, "cluster"),
                                           ("c5", 32, 1 << 20, "grid"), ("c5", 6, 300001, "two_phase"),
                                           ("c5", 6, 300001, "two_pass")])
def test_softmax_replayed_from_a_graph(name, M, N, path):
    x1 = workloads.matrix(workloads.WORKLOADS[name].with_shape(M, N))
    x2 = np.flip(x1, axis=1).copy() * np.float32(-0.5)          # other values, other row maxima
    if path == "two_phase":
        rrs.force_path("two_phase")
    else:
        assert _plan_path(M, N) == path
    x = torch.from_numpy(x1).cuda()
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rrs.softmax_rows(x, y)                                   # allocations happen here, eagerly
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rrs.softmax_rows(x, y)
    for k, xh in enumerate([x1, x2, x1, x2, x2]):
        x.copy_(torch.from_numpy(xh))
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_every_row(check_softmax, y, xh, f"{path} {M}x{N} replay {k}")
    del g


def test_row_sum_replayed_from_a_graph():
    M, N = 4096, 32768
    x1 = workloads.matrix(workloads.WORKLOADS["c3"])
    x = torch.from_numpy(x1).cuda()
    out = torch.empty(M, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rrs.row_sum(x, out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rrs.row_sum(x, out)
    for k, scale in enumerate([1.0, -0.5]):
        xh = x1 * np.float32(scale)
        x.copy_(torch.from_numpy(xh))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        check_row_sum(out.cpu().numpy(), xh, f"row sum replay {k}")
    del g


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")   # the refused call captured nothing
def test_capture_refuses_to_allocate_and_keeps_captured_workspaces():
    """A captured call that would need a larger workspace is refused (nothing
    is enqueued); a workspace a graph captured stays valid when a later eager
    call on the same stream grows it."""
    small = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(2, 1 << 18))
    big = workloads.matrix(workloads.WORKLOADS["c5"].with_shape(64, 1 << 20))   # slots past 64 KiB
    assert _plan_path(2, 1 << 18) == "grid" and _plan_path(64, 1 << 20) == "grid"
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    ws = [rrs.plan_softmax(M, N, N, True, props.multi_processor_count,
                           props.shared_memory_per_block_optin)["workspace_bytes"]
          for M, N in ((2, 1 << 18), (64, 1 << 20))]
    assert ws[0] <= 65536 < ws[1]                       # the smallest workspace is 64 KiB
    xs, xb = torch.from_numpy(small).cuda(), torch.from_numpy(big).cuda()
    ys, yb = torch.empty_like(xs), torch.empty_like(xb)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rrs.softmax_rows(xs, ys)                        # this stream's grid workspace: small
    torch.cuda.synchronize()
    g_bad = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_bad, stream=s):
        with pytest.raises(rrs.RRSError) as e:
            rrs.softmax_rows(xb, yb)                    # would grow the workspace inside the capture
    assert e.value.status == 6
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rrs.softmax_rows(xs, ys)                        # captured: uses the small workspace
    with torch.cuda.stream(s):
        rrs.softmax_rows(xb, yb)                        # eager: grows the workspace (the old one is kept)
    torch.cuda.synchronize()
    assert rrs.device_error() == 0
    check_every_row(check_softmax, yb, big, "eager call after growth")
    for k, xh in enumerate([small, np.flip(small, axis=1).copy()]):
        xs.copy_(torch.from_numpy(xh))
        ys.fill_(float("nan"))
        g.replay()                                      # still replays into the kept workspace
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_every_row(check_softmax, ys, xh, f"replay {k} after growth")
    del g, g_bad


def test_softmax_cols_two_pass_replayed_from_a_graph():
    """The two-pass column path draws its ticket on the device too: a replay
    never takes a column partial of the previous replay (x changes between
    replays, and every column is checked)."""
    from gpu_helpers import check_softmax_cols
    M, N = 4096, 8192
    x1 = workloads.matrix(workloads.WORKLOADS["c4"].with_shape(M, N))
    x2 = np.flip(x1, axis=0).copy() * np.float32(-0.5)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    assert rrs.plan_softmax_cols(M, N, N, True, sms)["path_name"] == "two_pass"
    x = torch.from_numpy(x1).cuda()
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rrs.softmax_cols(x, y)                                   # allocations happen here, eagerly
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rrs.softmax_cols(x, y)
    for k, xh in enumerate([x2, x1, x2]):
        x.copy_(torch.from_numpy(xh))
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert rrs.device_error() == 0
        check_softmax_cols(y.cpu().numpy(), xh, f"cols two-pass replay {k}")
    del g
