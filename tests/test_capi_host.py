"""Host-side tests of the C ABI (no GPU): exports, argument checks, the planner.

Only calls that return before anything touches CUDA are made here: argument
errors, the pure planner and the occupancy / wave arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rrs.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

OK, INVALID, ALIAS, CUDA, TIMEOUT, NOMEM, UNSUPPORTED = range(7)


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"RRS_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_two_entry_points(lib):
    names = declared_symbols()
    assert "softmax_rows" in names and "row_sum" in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["RRS_OK", "RRS_ERR_INVALID_ARG", "RRS_ERR_ALIAS", "RRS_ERR_CUDA",
                                 "RRS_ERR_TIMEOUT", "RRS_ERR_NOMEM", "RRS_ERR_UNSUPPORTED"]):
        assert lib.rrs_status_string(code).decode() == name
    assert lib.rrs_status_string(99).decode() == "RRS_ERR_UNKNOWN"


@pytest.mark.parametrize("fn", ["softmax_rows", "row_sum"])
def test_argument_errors_before_any_launch(lib, fn):
    f = getattr(lib, fn)
    a, b = 0x10000, 0x900000
    assert f(a, b, -1, 4, 4, None) == INVALID            # M < 0
    assert f(a, b, 4, -1, 4, None) == INVALID            # N < 0
    assert f(a, b, 4, 8, 7, None) == INVALID             # ld < N
    assert f(a, b, 4, 0, 0, None) == INVALID             # ld < 1
    assert f(a, b, 0, 8, 8, None) == OK                  # no rows: no work
    assert f(None, None, 0, 8, 8, None) == OK
    assert f(None, b, 4, 8, 8, None) == INVALID          # null x
    assert f(a, None, 4, 8, 8, None) == INVALID          # null y / out
    assert f(a + 2, b, 4, 8, 8, None) == INVALID         # not 4-byte aligned
    assert f(a, a + 16, 4, 8, 8, None) == ALIAS          # overlapping ranges
    assert f(a, b, 1 << 62, 1 << 20, 1 << 20, None) == INVALID  # extent overflow


def test_softmax_no_columns_is_a_no_op(lib):
    assert lib.softmax_rows(0x10000, 0x900000, 4, 0, 1, None) == OK


def test_inject_fault_rejects_unknown(lib):
    assert lib.rrs_inject_fault(7) == INVALID
    assert lib.rrs_inject_fault(0) == OK


def test_occupy_rejects_bad_arguments_before_any_gpu_call(lib):
    """The SM-holding test kernel is bounded: at most 0.2 s, at least one CTA,
    no negative sizes -- refused before the library touches a device."""
    for ctas, smem, ns in [(0, 0, 1000), (-1, 0, 1000), (70000, 0, 1000), (1, -1, 1000),
                           (1, 0, -1), (1, 0, 200_000_001)]:
        assert lib.rrs_test_occupy(ctas, smem, ns, None) == INVALID, (ctas, smem, ns)


def test_force_path_rejects_unknown(lib):
    assert lib.rrs_force_path(99, -1) == INVALID
    assert lib.rrs_force_path(-1, 99) == INVALID
    assert lib.rrs_force_path(-1, -1) == OK


# ----------------------------------------------------------------- planner ----

def plan(M, N, ld=None, vector_ok=True, sms=152):
    import row_reduction_softmax_gb300 as rrs
    return rrs.plan_softmax(M, N, ld, vector_ok, sms)


def test_planner_on_the_five_workloads(lib):
    p1 = plan(128, 256)
    assert p1["path_name"] == "row_regs" and p1["warps_per_row"] == 1 and p1["vec"] == 2
    p2 = plan(8192, 1024)
    assert p2["path_name"] == "row_regs" and p2["warps_per_row"] == 1 and p2["vec"] == 8
    p3 = plan(4096, 32768)
    assert p3["path_name"] == "cluster" and p3["cluster"] == 4 and p3["grid"] == 4096 * 4
    p4 = plan(16384, 4096)
    assert p4["path_name"] == "row_regs" and p4["warps_per_row"] == 4
    p5 = plan(32, 1 << 20)
    assert p5["path_name"] == "grid"


def test_grid_plan_for_the_longest_rows(lib):
    import row_reduction_softmax_gb300 as rrs
    try:
        rrs.force_path("grid")
        p5 = plan(32, 1 << 20)
        assert p5["path_name"] == "grid" and p5["threads"] == 512
        # 76 segments of 13800 floats (one 55 KB stage each) per row, 2 rows per round
        assert (p5["ctas_per_row"], p5["rows_per_cta"], p5["grid"], p5["rounds"]) == (76, 2, 152, 16)
        assert p5["stages"] == 4 and p5["tile"] >= p5["chunk"] and p5["vec"] == 8
    finally:
        rrs.force_path("auto", "auto")


def test_planner_unaligned_takes_scalar_path(lib):
    p = plan(100, 1000, ld=1001, vector_ok=False)         # short rows: scalar warp-per-row
    assert p["path_name"] == "row_regs" and p["vector_io"] == 0
    assert p["vec"] * 32 * p["warps_per_row"] * 4 >= 1000
    p = plan(100, 20000, ld=20001, vector_ok=False)       # long rows: scalar cluster split
    assert p["path_name"] == "cluster" and p["vector_io"] == 0
    p = plan(100, 131075, ld=131075, vector_ok=False)     # beyond 16 CTAs' registers: scalar two-pass
    assert p["path_name"] == "two_pass" and p["vector_io"] == 0
    p = plan(4, 1 << 24)                                    # past the grid, 2048 chunks a row: two-phase
    assert p["path_name"] == "two_phase"
    p = plan(32, 1048575, ld=1048576)                       # ragged past the cluster: scalar two-pass
    assert p["path_name"] == "two_pass" and p["vector_io"] == 0
    p = plan(100, 50257, ld=50260)                          # aligned rows, N % 4 != 0: cluster with a tail
    assert p["path_name"] == "cluster" and p["vector_io"] == 1


@pytest.mark.parametrize("N", [16385, 20001, 32767, 50257, 65537, 100001, 131072])
def test_scalar_cluster_plans_cover_the_row(lib, N):
    p = plan(5, N, ld=N + 1, vector_ok=False)
    assert p["path_name"] == "cluster" and p["vector_io"] == 0
    cs = p["cluster"]
    assert 1 <= cs <= 16 and p["grid"] == 5 * cs
    assert -(-N // cs) <= 4 * p["vec"] * p["threads"]     # each CTA's scalar segment fits its slots


def row_slots(q):
    """Floats one row's register slots hold under a plan."""
    if q["path_name"] == "cluster":
        return 4 * q["vec"] * q["threads"] * q["cluster"]
    return 4 * q["vec"] * 32 * q["warps_per_row"]


def forced_plan(path, M, N, ld, vector_ok):
    import row_reduction_softmax_gb300 as rrs
    rrs.force_path(path)
    try:
        return plan(M, N, ld=ld, vector_ok=vector_ok)
    finally:
        rrs.force_path("auto", "auto")


@pytest.mark.parametrize("vector_ok", [False, True])
@pytest.mark.parametrize("N", [1, 3, 5, 127, 129, 1023, 1025, 4095, 4096, 4097, 6144, 8191, 8192,
                               12287, 12288, 16383, 16384])
@pytest.mark.parametrize("M", [7, 152, 153, 1024, 4096])
def test_row_plans_cover_the_row(lib, M, N, vector_ok):
    """Up to 4096 floats the register kernel; up to 16384 the register
    kernel or the cluster split, whichever holds the row in no more register
    slots (the cluster split when they tie), the cluster split only for more
    rows than SMs and, for rows of up to 8192 floats, 2^23 floats or more."""
    ld = N if vector_ok else N + 1
    p = plan(M, N, ld=ld, vector_ok=vector_ok)
    if not vector_ok:
        assert p["vector_io"] == 0
    if N <= 4096:
        assert p["path_name"] == "row_regs"
    assert p["path_name"] in ("row_regs", "cluster")
    # a slot holds 4 scalars, or one float4 with the N % 4 tail beside the slots
    need = N // 4 if p["vector_io"] == 1 else -(-N // 4)
    if p["path_name"] == "row_regs":
        assert p["vec"] * 32 * p["warps_per_row"] >= need
    else:
        assert -(-need // p["cluster"]) <= p["vec"] * p["threads"]
    if 4096 < N:
        r = forced_plan("row_regs", M, N, ld, vector_ok)
        c = forced_plan("cluster", M, N, ld, vector_ok)
        assert r["path_name"] == "row_regs" and c["path_name"] == "cluster"
        many_rows = M > 152 and (N > 8192 or M * N >= 1 << 23)
        want = "cluster" if many_rows and row_slots(c) <= row_slots(r) else "row_regs"
        assert p["path_name"] == want, (row_slots(c), row_slots(r))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 31, 127, 128, 129, 255, 256, 257, 1000, 1024, 2047,
                               2048, 2049, 4095, 4096, 4097, 8191, 16384, 16385, 32767, 32768,
                               65536, 131072, 131073, 1 << 20, (1 << 20) + 3])
@pytest.mark.parametrize("M", [1, 7, 152, 4096])
def test_planner_covers_every_column(lib, M, N):
    p = plan(M, N)
    assert 32 <= p["threads"] <= 1024 and p["threads"] % 32 == 0
    assert p["grid"] >= 1
    n4 = N // 4
    if p["path_name"] == "row_regs":
        gt = 32 * p["warps_per_row"]
        assert p["vec"] * gt >= n4 and (N % 4) <= gt
        assert p["rows_per_cta"] * gt == p["threads"]
    elif p["path_name"] == "cluster":
        cs = p["cluster"]
        assert 1 <= cs <= 16 and p["grid"] % cs == 0
        seg4 = -(-n4 // cs)
        assert seg4 <= p["vec"] * p["threads"]
    elif p["path_name"] == "two_phase":
        C, chunk = p["ctas_per_row"], p["chunk"]
        assert chunk % 1024 == 0 and C * chunk >= N > (C - 1) * chunk
        assert p["workspace_bytes"] == M * C * 8
    elif p["path_name"] == "row_staged":
        assert N % 4 == 0 and p["threads"] == 544 and p["grid"] == min(M, 152)
        assert p["smem_bytes"] == 2048 + p["stages"] * p["tile"] * 4 <= 232448
        if p["vec"] > 0:                                    # whole rows in registers
            assert p["vec"] * 32 * p["warps_per_row"] * 4 >= N and p["tile"] >= N
            groups = 16 // p["warps_per_row"]
            assert p["stages"] % groups == 0 and groups <= p["stages"] <= 64
        else:                                               # a row staged as <= 4 sub-tiles
            assert p["tile"] % 4 == 0 and -(-N // p["tile"]) <= 4 < p["stages"]
    elif p["path_name"] == "grid":
        C, seg = p["ctas_per_row"], p["chunk"]
        assert N % 4 == 0 and seg % 4 == 0 and C * seg >= N > (C - 1) * seg
        R = p["rows_per_cta"]
        assert p["threads"] == 512 and p["grid"] == R * C <= 152 and R <= M and C <= 160
        assert p["tile"] >= seg and p["tile"] % 32 == 0 and 2 <= p["stages"] <= 64
        assert -(-seg // 4) <= p["vec"] * 448 and p["vec"] in (2, 4, 8)
        assert p["smem_bytes"] == 2048 + p["stages"] * p["tile"] * 4 <= 232448
        assert p["rounds"] == -(-M // R) and p["workspace_bytes"] == 128 + M * C * 16


def test_forced_paths(lib):
    import row_reduction_softmax_gb300 as rrs
    try:
        rrs.force_path("cluster")
        assert plan(64, 1024)["path_name"] == "cluster"
        rrs.force_path("two_phase")
        assert plan(64, 1024)["path_name"] == "two_phase"
        rrs.force_path("grid")
        assert plan(64, 1024)["path_name"] == "grid"
        rrs.force_path("row_staged")
        assert plan(64, 30000)["path_name"] == "row_staged"
        assert plan(64, 1024)["path_name"] == "row_staged"
        with pytest.raises(rrs.RRSError):
            plan(64, 1022)                                  # N % 4 != 0
        rrs.force_path("row_regs")
        with pytest.raises(rrs.RRSError) as e:
            plan(4, 65536)
        assert e.value.status == UNSUPPORTED
        assert plan(4, 1024, vector_ok=False)["vector_io"] == 0   # the scalar variant
    finally:
        rrs.force_path("auto", "auto")


def test_row_sum_planner(lib):
    import row_reduction_softmax_gb300 as rrs
    p = rrs.plan_row_sum(4096, 32768)
    assert p["path_name"] == "row" and p["threads"] == 256 and p["warps_per_row"] == 8
    p = rrs.plan_row_sum(32, 1 << 20)
    assert p["path_name"] == "split" and p["ctas_per_row"] * p["chunk"] >= 1 << 20
    p = rrs.plan_row_sum(10, 10)
    assert p["path_name"] == "row" and p["warps_per_row"] == 1


# ------------------------------------------- occupancy and wave arithmetic ----

def load_hardware_problems():
    rows = []
    with open(os.path.join(GOLDEN, "hardware_problems.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, rest = line.split(":", 1)
            lhs, rhs = rest.split("->")
            args = dict(kv.split("=") for kv in lhs.split())
            want = dict(kv.split("=") for kv in rhs.split())
            rows.append((kind.strip(), args, want))
    return rows


def test_occupancy_and_waves_match_the_lecture_problems(lib):
    import row_reduction_softmax_gb300 as rrs
    seen = set()
    for kind, a, want in load_hardware_problems():
        seen.add(kind)
        if kind == "occupancy":
            blocks, warps, pct = rrs.occupancy(int(a["threads"]), int(a["regs"]), int(a["sm_regs"]),
                                               int(a["max_warps"]))
            assert (blocks, warps) == (int(want["blocks"]), int(want["warps"]))
            assert pct == float(want["percent"])
        elif kind == "waves":
            n, last, idle = rrs.waves(int(a["blocks"]), int(a["sms"]))
            assert (n, last, idle) == (int(want["waves"]), int(want["last"]), int(want["idle"]))
    assert seen == {"occupancy", "waves"}


# ------------------------------------------------------------ column softmax ---

@pytest.mark.parametrize("N", [1, 3, 4, 127, 128, 129, 8192, 16384])
@pytest.mark.parametrize("M", [1, 2, 7, 64, 100, 1024, 2048, 2049, 4096, 8192, 8193])
def test_cols_planner(lib, M, N):
    import row_reduction_softmax_gb300 as rrs
    p = rrs.plan_softmax_cols(M, N)
    bands = -(-N // 32)
    assert p["threads"] == 256
    q = rrs.plan_softmax_cols(M, N, vector_ok=False)
    # unaligned: the two-pass path's scalar form up to 8 slices a band, else the two-phase pair
    assert q["path_name"] == ("two_pass" if -(-M // 512) <= 8 else "two_phase") and q["vector_io"] == 0
    # aligned input with items enough to interleave (slices of 512 rows x
    # bands at least twice the lag of 3 x 152 items) and at most 8 slices
    # per band: the two-pass path
    if -(-M // 512) * bands >= 2 * 3 * 152 and -(-M // 512) <= 8:
        assert p["path_name"] == "two_pass" and p["stages"] == 3 * 152
        return
    # otherwise the band path, the fewest CTAs per band (a power of two, at
    # most 8) that keep a CTA at most 512 rows (M < 2048) or 1024 rows
    assert p["path_name"] == "band" and p["workspace_bytes"] == 0
    cs, rows = p["cluster"], p["rows_per_cta"]
    cap = 512 if M < 2048 else 1024
    assert cs in (1, 2, 4, 8) and rows == -(-M // cs)
    assert rows <= cap or cs == 8
    assert cs == 1 or -(-M // (cs // 2)) > cap                # no smaller cluster would do
    assert p["grid"] == bands * cs
    # registers budgeted for four CTAs per SM
    assert p["vec"] == 4


def test_cols_forced_paths(lib):
    import row_reduction_softmax_gb300 as rrs
    try:
        rrs.force_cols_path("two_phase")
        assert rrs.plan_softmax_cols(64, 1024)["path_name"] == "two_phase"
        p = rrs.plan_softmax_cols(4096, 1024)
        chunks, chunk = p["ctas_per_row"], p["chunk"]
        assert chunks * chunk >= 4096 > (chunks - 1) * chunk
        assert p["grid"] == 32 * chunks and p["workspace_bytes"] == chunks * 1024 * 8
        rrs.force_cols_path("band")
        assert rrs.plan_softmax_cols(64, 1024)["path_name"] == "band"
        with pytest.raises(rrs.RRSError) as e:
            rrs.plan_softmax_cols(64, 1024, vector_ok=False)
        assert e.value.status == UNSUPPORTED
        rrs.force_cols_path("cluster")
        p = rrs.plan_softmax_cols(8192, 1024)            # forced: up to 16 CTAs per band
        assert p["path_name"] == "cluster" and p["cluster"] == 16 and p["vec"] == 16
        with pytest.raises(rrs.RRSError) as e:
            rrs.plan_softmax_cols(8193, 1024)
        assert e.value.status == UNSUPPORTED
    finally:
        rrs.force_cols_path("auto")
    assert lib.rrs_force_cols_path(7) == 1


def test_new_entry_points_check_arguments(lib):
    import ctypes
    # host-side checks run before any device call
    assert lib.softmax_rows_ex(None, 4, None, 4, 0, 4, 0, None) == 0        # empty: no work
    assert lib.softmax_rows_ex(None, 4, None, 4, 2, 4, 2, None) == 1        # unknown flag bit
    assert lib.softmax_rows_ex(None, 3, None, 4, 2, 4, 0, None) == 1        # ldx < N
    assert lib.softmax_cols(None, 4, None, 2, 2, 4, 0, None) == 1           # ldy < N
    assert lib.softmax_cols(None, 4, None, 4, 2, 4, 0, None) == 1           # null pointers
    assert lib.log_softmax_rows(None, None, -1, 4, 4, None) == 1            # M < 0
    assert lib.row_max(None, None, 0, 4, 4, None) == 0
    assert lib.row_mean(None, None, 2, 4, 3, None) == 1                     # ld < N
    buf = (ctypes.c_float * 64)()
    a = ctypes.addressof(buf)
    # overlap that is not exact in-place: rejected before the pointers are examined
    assert lib.softmax_rows_ex(a, 8, a + 16, 8, 2, 8, 0, None) == 2
    assert lib.softmax_rows_ex(a, 8, a, 4, 2, 4, 0, None) == 2               # same base, other stride
    assert lib.softmax_cols(a, 8, a + 4, 8, 2, 8, 0, None) == 2


def two_pass_item(lib, t, Q, D):
    pass_, k = ctypes.c_int(), ctypes.c_int64()
    assert lib.rrs_cols_two_pass_item(t, Q, D, ctypes.byref(pass_), ctypes.byref(k)) == OK
    return pass_.value, k.value


@pytest.mark.parametrize("bands,S,D", [(1, 1, 1), (3, 1, 1), (3, 1, 3), (5, 4, 4), (5, 4, 7), (5, 4, 20),
                                       (512, 8, 304), (256, 2, 304), (7, 3, 3)])
def test_cols_two_pass_sequence(lib, bands, S, D):
    """COLS_TWO_PASS deals every item once to each pass, and the first pass of
    every slice of a band comes before any second pass of that band (so a
    second pass waits only on CTAs that drew earlier, hence are running)."""
    Q = bands * S
    seen = {1: {}, 2: {}}
    for t in range(2 * Q):
        p, k = two_pass_item(lib, t, Q, D)
        assert p in (1, 2) and 0 <= k < Q and k not in seen[p]
        seen[p][k] = t
    assert len(seen[1]) == Q and len(seen[2]) == Q
    for k, t2 in seen[2].items():
        b = k // S
        assert max(seen[1][b * S + r] for r in range(S)) < t2
    if D < Q:   # the second pass of an item trails its first by 2 D + 1 arrivals in the interleaved stretch
        k = D
        if k < Q - D:
            assert seen[2][k] - seen[1][k] == 2 * D + 1


def test_cols_two_pass_item_rejects_bad_arguments(lib):
    p, k = ctypes.c_int(), ctypes.c_int64()
    assert lib.rrs_cols_two_pass_item(0, 4, 0, ctypes.byref(p), ctypes.byref(k)) == INVALID
    assert lib.rrs_cols_two_pass_item(0, 4, 5, ctypes.byref(p), ctypes.byref(k)) == INVALID
    assert lib.rrs_cols_two_pass_item(8, 4, 2, ctypes.byref(p), ctypes.byref(k)) == INVALID
    assert lib.rrs_cols_two_pass_item(-1, 4, 2, ctypes.byref(p), ctypes.byref(k)) == INVALID
    assert lib.rrs_cols_two_pass_item(0, 4, 2, None, ctypes.byref(k)) == INVALID


@pytest.mark.parametrize("M,N", [(1, 1), (5, 33), (512, 64), (513, 64), (4096, 16384), (1024, 8192), (70000, 40)])
def test_cols_two_pass_plan(lib, M, N):
    import row_reduction_softmax_gb300 as rrs
    rrs.force_cols_path("two_pass")
    try:
        p = rrs.plan_softmax_cols(M, N, N, True, 152)
    finally:
        rrs.force_cols_path("auto")
    assert p["path_name"] == "two_pass"
    bands = -(-N // 32)
    R, S, D = p["chunk"], p["ctas_per_row"], p["stages"]
    assert S == -(-M // R) and S <= D <= bands * S and p["grid"] == 2 * bands * S
    assert p["workspace_bytes"] == 128 + bands * S * 32 * 16


@pytest.mark.parametrize("M,N,ld,vec", [(1, 1, 1, False), (3, 8192, 8192, True), (3, 8193, 8196, True),
                                        (32, 1 << 20, 1 << 20, True), (4, 300001, 300003, False),
                                        (2, 5_000_000, 5_000_000, True)])
def test_row_two_pass_plan(lib, M, N, ld, vec):
    import row_reduction_softmax_gb300 as rrs
    rrs.force_path("two_pass")
    try:
        p = plan(M, N, ld=ld, vector_ok=vec)
    finally:
        rrs.force_path("auto", "auto")
    assert p["path_name"] == "two_pass" and p["threads"] == 256 and p["chunk"] == 8192
    S = -(-N // 8192)
    assert p["ctas_per_row"] == S and S <= p["stages"] <= M * S and p["grid"] == 2 * M * S
    assert p["stages"] == min(M * S, max(S, 4 * 152))             # the lag: 4 x SMs, clamped
    assert p["workspace_bytes"] == 128 + M * S * 16
    assert p["vector_io"] == (1 if vec and N % 4 == 0 else 0)   # float4 only for whole float4 rows


@pytest.mark.parametrize("N,path", [(2_097_152, "two_pass"), (2_097_153, "two_phase")])
def test_unaligned_long_rows_between_two_pass_and_two_phase(lib, N, path):
    """Rows the grid split cannot align take the two-pass split up to 256
    chunks of 8192 floats a row, the two-phase pair past that."""
    p = plan(8, N, ld=N + 1, vector_ok=False)
    assert p["path_name"] == path and p["vector_io"] == 0
    if path == "two_pass":
        assert p["ctas_per_row"] == 256
