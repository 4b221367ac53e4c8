#!/usr/bin/env python3
"""Benchmark of the fused row softmax (and row sum) on GB300, one JSON line.

A step is one ``softmax_rows`` call over the headline workload (default
``c3``: 4096 x 32768 fp32, Uniform(-8, 8), seed 2 -- the largest of the five
workloads, whose rows overflow one block and are split over a thread-block
cluster), inputs resident in HBM.  Consecutive steps rotate over enough x/y
buffer pairs that the working set is at least four times the L2 (or use one
pair larger than it), so every step reads x from HBM.  Every x and y buffer
is written once before the timed region, so no step pays a first touch.
Timed with CUDA events on the launching stream, warm-up first, barrier +
synchronize on both sides, max over ranks.

The line carries, besides the contract's keys:
  roofline      the dominant kernel's algorithmic bytes (8 per element: one
                fp32 read, one fp32 write) / its average launch time, against
                the measured HBM copy peak; ncu DRAM traffic per launch when a
                committed profile matches the current kernel sources
  e2e           the same metric through the public API with pinned host
                buffers: H2D of x, the call, D2H of y, all in the timed region
  cpu_baseline  the float64 oracle timed on this host (test infrastructure,
                timed here only as a baseline): one process, and in
                `all_cores` one process per host core over blocks of rows
  suite         every other row of the hot path -- the split-row softmax
                (cluster / grid / two-phase), the single-pass softmax on the
                masked-logit rows, the row sum -- each timed on its workload
                with its roofline fraction and a sampled-row parity check
  variants      the operations built on the same skeleton -- log-softmax, in
                place, row max / mean, column softmax, GeLU -- timed and checked
                the same way, and the fused attention forward (TFLOP/s against
                the measured bf16 tensor peak)
  clocks        SM clock and clock-event reasons sampled during the timed region
  summary       last, one short entry per suite / variant row (time per call,
                fraction of the peak and, for the softmax rows, the time of a
                plain device copy of the same bytes), so that a reader of only
                the end of the line still sees every row

``--impl reference`` times the oracle instead, on the same metric and config.
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

ROOFLINE_GBS = 8000.0          # the 8 TB/s HBM figure the metric is stated against
FALLBACK_HBM_GBS = 6800.0
METRIC = "softmax rows/s and achieved HBM GB/s as fraction of 8 TB/s roofline (1×GB300)"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-suite", action="store_true", help="skip the per-row suite")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the variants (log-softmax, in place, row max/mean, columns, GeLU)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget")
    ap.add_argument("--suite-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--path", default="auto", help="force a softmax path (auto, row_regs, cluster, ...)")
    ap.add_argument("--only", default=None,
                    help="run only the suite / variant entries named here, as workload:op, comma-separated "
                         "(for example c3:softmax,cols_c4:softmax_cols,attn:attention_fwd)")
    ap.add_argument("--json-out", default=None, help="also write the JSON line to this file")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers ---

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank gets the max over all ranks."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(M: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: rows of all replicas over the slowest rank's time."""
    return world * M * steps / (max_ms / 1e3)


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed on its own: the burst figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured"
    except Exception:
        return 1900.0, "fallback"


# The sources each timed kernel is built from, beyond the device headers
# every kernel shares.  A committed ncu figure is keyed to a hash of these
# files and of the launch plan the planner makes for the workload, so it
# stands while neither the kernel nor its launch changes.
KERNEL_SOURCES = {
    "softmax_row_regs_kernel": ["softmax_row.cu"],
    "softmax_cluster_kernel": ["softmax_split.cu"],
    "softmax_staged_grid_kernel": ["softmax_staged.cu", "sm100_async.cuh"],
    "row_reduce_rows_kernel": ["row_sum.cu"],
    "softmax_cols_band_kernel": ["softmax_cols.cu", "sm100_async.cuh", "two_pass_common.cuh"],
    "softmax_cols_two_pass_kernel": ["softmax_cols.cu", "sm100_async.cuh", "two_pass_common.cuh"],
    "softmax_rows_two_pass_kernel": ["softmax_rows_two_pass.cu", "sm100_async.cuh", "two_pass_common.cuh"],
    "attention_fwd_kernel": ["attention.cu", "sm100_async.cuh", "sm100_tcgen05.cuh"],
    "gelu_kernel": ["gelu.cu"],
}
COMMON_SOURCES = ["device_common.cuh", "launch_util.h"]


def source_hash(kernel: str | None = None, plan: dict | None = None) -> str:
    """Hash of the sources a kernel is built from (all of csrc/ for an unknown
    or no kernel) and of its launch plan: a committed ncu figure stands only
    while it matches."""
    csrc = os.path.join(ROOT, "row_reduction_softmax_gb300", "csrc")
    if kernel in KERNEL_SOURCES:
        paths = [os.path.join(csrc, n) for n in sorted(COMMON_SOURCES + KERNEL_SOURCES[kernel])]
    else:
        paths = sorted(glob.glob(os.path.join(csrc, "*")))
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    if plan is not None:
        h.update(json.dumps({k: plan[k] for k in sorted(plan) if k != "path_name"}, sort_keys=True).encode())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, workload: str, plan: dict | None = None):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    kernel's current sources and launch plan."""
    want = source_hash(kernel, plan)
    pat = re.compile(r"traffic:\s+kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=(\d+)\s+source=(\w+)")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == want:
                    return int(m.group(3))
    return None


class ClockSampler:
    """Samples the SM clock and clock-event reasons through NVML (read only)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle", 0x10: "sync_boost"}

    def __init__(self, pci_bus_id: str | None, period_s: float = 0.01):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            rc = 1
            if pci_bus_id:
                rc = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.handle))
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.handle))
            if rc != 0:
                return
            v = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(v)) == 0:
                self.max_mhz = v.value
            try:
                self._reason_fn = self.nvml.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self._reason_fn = self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            self.ok = False

    def _sample(self):
        v = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(v)) == 0:
            self.samples.append(v.value)
        if self._reason_fn(self.handle, ctypes.byref(r)) == 0:
            self.reasons |= r.value

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            self._stop.wait(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self.ok and self._thread:
            self._stop.set()
            self._thread.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        names = [n for bit, n in sorted(self.REASONS.items()) if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples), "source": "nvml"}


def pci_bus_id(torch, dev: int):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


def sampled_rows(M: int, k: int, seed: int):
    rng = np.random.default_rng(seed + 2024)
    return sorted({0, M - 1, *rng.choice(M, size=min(M, k), replace=False).tolist()})


def oracle_parity_softmax(y_dev, w, rows):
    """Max errors of sampled output rows against the float64 oracle (test infrastructure)."""
    import oracle
    x = workloads.matrix(w, rows=rows).astype(np.float64)
    want = oracle.softmax_rows(x)
    got = y_dev[rows].cpu().numpy().astype(np.float64)
    ok = ~np.isnan(want).any(axis=1)
    big = want[ok] >= 1e-30
    return {"rows_checked": len(rows),
            "max_abs": float(np.max(np.abs(got[ok] - want[ok]))),
            "max_rel": float(np.max(np.abs(got[ok][big] - want[ok][big]) / want[ok][big])),
            "row_sum": float(np.max(np.abs(got[ok].sum(axis=1) - 1.0)))}


def oracle_parity_row_sum(out_dev, w, rows):
    import oracle
    x = workloads.matrix(w, rows=rows).astype(np.float64)
    want = oracle.row_sum(x)
    got = out_dev[rows].cpu().numpy().astype(np.float64)
    scale = np.abs(x).sum(axis=1)
    return {"rows_checked": len(rows), "max_abs": float(np.max(np.abs(got - want))),
            "max_normwise": float(np.max(np.abs(got - want) / scale))}


def kernel_of(plan: dict) -> str:
    """Name of the kernel a plan launches (the two-phase path launches two)."""
    name = plan["path_name"]
    if name == "row_staged":
        return "softmax_staged_rows_kernel" if plan["vec"] > 0 else "softmax_staged_long_kernel"
    return {"row_regs": "softmax_row_regs_kernel", "cluster": "softmax_cluster_kernel",
            "two_phase": "softmax_partials_kernel+softmax_finalize_kernel",
            "grid": "softmax_staged_grid_kernel", "two_pass": "softmax_rows_two_pass_kernel",
            "row": "row_reduce_rows_kernel",
            "split": "row_reduce_partials_kernel+row_reduce_finalize_kernel"}.get(name, name)


def touch(bufs) -> None:
    """Write every output buffer once (zeros), so that no timed call is the
    first to touch its pages; the caller synchronizes before timing."""
    for b in bufs:
        b.zero_()


def l2_pairs(torch, pair_bytes: int) -> int:
    l2 = getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0) \
        or 129 * 10**6
    return int(max(1, min(8, -(-4 * l2 // pair_bytes))))


# --------------------------------------------------------------- our arm ---

def run_ours(args):
    import torch
    import row_reduction_softmax_gb300 as rrs

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    rrs.load_library()
    rrs.force_path(args.path, "auto")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    w = workloads.WORKLOADS[args.workload]
    M, N = w.M, w.N
    x_host = workloads.matrix(w)
    pair_bytes = 2 * M * N * 4
    npairs = l2_pairs(torch, pair_bytes)
    xs = [torch.from_numpy(x_host).to(dev) for _ in range(npairs)]
    ys = [torch.empty_like(xs[0]) for _ in range(npairs)]
    touch(ys)
    plan = rrs.plan_softmax(M, N, N, True, torch.cuda.get_device_properties(dev).multi_processor_count,
                            torch.cuda.get_device_properties(dev).shared_memory_per_block_optin)
    launches_per_call = 2 if plan["path_name"] == "two_phase" else 1

    def step(k):
        r = k % npairs
        rrs.softmax_rows_ptr(xs[r].data_ptr(), ys[r].data_ptr(), M, N, N, sh)

    for k in range(max(args.warmup, 3)):
        step(k)
    torch.cuda.synchronize()

    sampler = ClockSampler(pci_bus_id(torch, dev.index))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    ev0.record(stream)
    for k in range(args.steps):
        step(k)
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    if rrs.device_error() != 0:
        raise SystemExit("device error word set during the timed region")

    # The same call timed one at a time (an event pair around each of 50
    # calls, after the timed region): the distribution behind the average.
    trial_us = []
    if rank == 0:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
        for k, (a, b) in enumerate(pairs):
            a.record(stream)
            step(k)
            b.record(stream)
        torch.cuda.synchronize()
        trial_us = sorted(a.elapsed_time(b) * 1e3 for a, b in pairs)

    ms_per_step = ms / args.steps
    rows_per_s = job_rows_per_s(M, args.steps, world, ms)
    alg_bytes = 8 * M * N
    achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    kernel_name = kernel_of(plan)
    parity = oracle_parity_softmax(ys[(args.steps - 1) % npairs], w, sampled_rows(M, 16, w.seed)) \
        if rank == 0 else None

    out = {
        "metric": METRIC,
        "value": rows_per_s,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: softmax_rows fp32 {M}x{N} {w.dist} seed {w.seed}",
                   "M": M, "N": N, "ld": N, "path": plan["path_name"],
                   "l2": f"rotating {npairs} x/y pairs ({npairs * pair_bytes >> 20} MiB, >= 4x L2)",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs": achieved,
        "frac_of_8tbs": achieved / ROOFLINE_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"of {peak_kind}",
                     "kernel": kernel_name, "algorithmic_bytes_per_launch": alg_bytes,
                     "traffic": ncu_traffic(kernel_name, w.name, plan),
                     "source": source_hash(kernel_name, plan)},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": sampler.summary(),
        "parity": parity,
    }
    if trial_us:
        out["trials"] = {"n": len(trial_us), "median_us": statistics.median(trial_us),
                         "p95_us": trial_us[int(0.95 * (len(trial_us) - 1))],
                         "how": "one call between a CUDA event pair, 50 calls, after the timed loop"}

    if not args.no_e2e:
        out["e2e"] = run_e2e(args, torch, rrs, dev, x_host, w)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        out["cpu_baseline"]["all_cores"] = cpu_baseline_all_cores(w, args.cpu_seconds / 2)
    if not args.no_suite:
        out["suite"] = run_suite(args, torch, rrs, dev, rank)
    if not args.no_variants:
        out["variants"] = run_variants(args, torch, rrs, dev, rank)
    out["summary"] = summary(out)
    del xs, ys
    if rank == 0:
        line = json.dumps(out)
        print(line, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(line + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, torch, rrs, dev, x_host, w):
    """H2D of x from pinned memory, the call, D2H of y -- two slots, three streams, overlapped."""
    M, N = w.M, w.N
    xp = torch.from_numpy(x_host).pin_memory()
    yp = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    xd = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(2)]
    yd = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_run + ev_out:
        e.record(s_run)

    def step(k):
        j = k % 2
        s_in.wait_event(ev_run[j])          # x slot free: its last call has read it
        with torch.cuda.stream(s_in):
            xd[j].copy_(xp, non_blocking=True)
        ev_in[j].record(s_in)
        s_run.wait_event(ev_in[j])
        s_run.wait_event(ev_out[j])         # y slot free: its last copy-out is done
        rrs.softmax_rows_ptr(xd[j].data_ptr(), yd[j].data_ptr(), M, N, N, s_run.cuda_stream)
        ev_run[j].record(s_run)
        s_out.wait_event(ev_run[j])
        with torch.cuda.stream(s_out):
            yp[j].copy_(yd[j], non_blocking=True)
        ev_out[j].record(s_out)

    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    steps = args.e2e_steps
    t0 = time.perf_counter()
    for k in range(steps):
        step(k)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    # the last result read back must be the softmax of x
    import oracle
    rows = sampled_rows(M, 4, w.seed)
    want = oracle.softmax_rows(x_host[rows].astype(np.float64))
    got = yp[(steps - 1) % 2][rows].numpy().astype(np.float64)
    return {"value": M * steps / dt, "unit": "rows/s", "h2d_bytes_per_step": M * N * 4,
            "d2h_bytes_per_step": M * N * 4, "steps": steps,
            "ms_per_step": dt / steps * 1e3, "max_abs_err_readback": float(np.max(np.abs(got - want))),
            "how": "pinned host x -> device, softmax_rows, device -> pinned host y; 2 slots, 3 streams"}


def _oracle_block_worker(task):
    """One host process of the all-cores CPU baseline: the oracle, as it
    stands, over its block of the workload's rows from a common start
    instant until the budget is spent."""
    name, r0, r1, start_at, budget_s = task
    import oracle
    w = workloads.WORKLOADS[name]
    x = workloads.matrix(w, rows=range(r0, r1))
    while time.time() < start_at:
        time.sleep(0.001)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.softmax_rows(x)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return (r1 - r0) * reps, time.perf_counter() - t0


def cpu_baseline_all_cores(w, budget_s: float, start_delay_s: float = 5.0):
    """The oracle on every host core: the rows split into one block per
    core, one spawned process each (no CUDA in them), timed together."""
    import multiprocessing as mp
    n = max(1, min(os.cpu_count() or 1, w.M))
    bounds = [(w.M * i // n, w.M * (i + 1) // n) for i in range(n)]
    start_at = time.time() + start_delay_s   # after every process has imported and built its block
    tasks = [(w.name, a, b, start_at, budget_s) for a, b in bounds if b > a]
    with mp.get_context("spawn").Pool(len(tasks)) as pool:
        res = pool.map(_oracle_block_worker, tasks)
    rows = sum(r for r, _ in res)
    dt = max(t for _, t in res)
    return {"value": rows / dt, "unit": "rows/s", "cores": len(tasks), "kind": "oracle",
            "sample": f"{len(tasks)} processes, each the float64 numpy oracle over a block of "
                      f"{w.M // len(tasks)}-{-(-w.M // len(tasks))} rows of the {w.M}x{w.N} matrix, "
                      f"{dt:.1f} s together",
            "gbs": 8 * w.N * rows / dt / 1e9}


def cpu_baseline(w, budget_s: float):
    """The float64 oracle, as it stands, on this host: whole-matrix passes until the budget is spent."""
    import oracle
    x = workloads.matrix(w)
    reps = 0
    cpu0 = time.process_time()
    t0 = time.perf_counter()
    while True:
        oracle.softmax_rows(x)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cpu = time.process_time() - cpu0
    return {"value": w.M * reps / dt, "unit": "rows/s", "cores": max(1, round(cpu / dt)),
            "kind": "oracle",
            "sample": f"{reps} pass(es) over the whole {w.M}x{w.N} matrix, float64 numpy, {dt:.1f} s",
            "gbs": 8 * w.M * w.N * reps / dt / 1e9, "host_cpus": os.cpu_count()}


def run_suite(args, torch, rrs, dev, rank):
    """Every other row of the hot path on its workload: kernel time, roofline fraction, parity."""
    peak, peak_kind = measured_hbm_peak()
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    entries = []
    for name, op in [("c1", "softmax"), ("c2", "softmax"), ("c3", "softmax"), ("c3", "row_sum"),
                     ("c4", "softmax"), ("c5", "softmax")]:
        if not selected(args, name, op):
            continue
        w = workloads.WORKLOADS[name]
        M, N = w.M, w.N
        x_host = workloads.matrix(w)
        if op == "softmax":
            pair_bytes = 2 * M * N * 4
            plan = rrs.plan_softmax(M, N, N, True, props.multi_processor_count,
                                    props.shared_memory_per_block_optin)
            alg = 8 * M * N
        else:
            pair_bytes = M * N * 4 + M * 4
            plan = rrs.plan_row_sum(M, N, N, True, props.multi_processor_count,
                                    props.shared_memory_per_block_optin)
            alg = 4 * M * N + 4 * M
        npairs = l2_pairs(torch, pair_bytes) if name != "c1" else 1
        xs = [torch.from_numpy(x_host).to(dev) for _ in range(npairs)]
        del x_host
        ys = [torch.empty_like(xs[0]) if op == "softmax" else
              torch.empty(M, dtype=torch.float32, device=dev) for _ in range(npairs)]
        touch(ys)
        fn = rrs.softmax_rows_ptr if op == "softmax" else rrs.row_sum_ptr

        def call(k):
            r = k % npairs
            fn(xs[r].data_ptr(), ys[r].data_ptr(), M, N, N, sh)

        for k in range(3):
            call(k)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for k in range(args.suite_steps):
            call(k)
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / args.suite_steps
        gbs = alg / (ms / 1e3) / 1e9
        copy_ms = None
        if op == "softmax":
            # context: torch's device copy of the same bytes (y <- x) over the same
            # rotating buffers, outside the timed region above
            for k in range(3):
                ys[k % npairs].copy_(xs[k % npairs])
            torch.cuda.synchronize()
            ev0.record(stream)
            for k in range(args.suite_steps):
                ys[k % npairs].copy_(xs[k % npairs])
            ev1.record(stream)
            torch.cuda.synchronize()
            copy_ms = ev0.elapsed_time(ev1) / args.suite_steps
        entry = {"workload": name, "op": op, "M": M, "N": N, "path": plan["path_name"],
                 "kernel": kernel_of(plan),
                 "grid": plan["grid"], "threads": plan["threads"], "cluster": plan["cluster"],
                 "ms_per_call": ms, "rows_per_s": M / (ms / 1e3), "hbm_gbs": gbs,
                 "frac_of_8tbs": gbs / ROOFLINE_GBS, "frac_of_peak": gbs / peak,
                 "peak_kind": f"of {peak_kind}", "calls_timed": args.suite_steps,
                 "l2": f"{npairs} rotating pair(s)"}
        if copy_ms is not None:
            entry["copy_us"] = copy_ms * 1e3
            entry["vs_copy"] = copy_ms / ms
        if rank == 0:
            # parity of the softmax's own output: one more call on pair 0
            if copy_ms is not None:
                fn(xs[0].data_ptr(), ys[0].data_ptr(), M, N, N, sh)
                torch.cuda.synchronize()
            rows = sampled_rows(M, 6, w.seed)
            last = ys[0] if copy_ms is not None else ys[(args.suite_steps - 1) % npairs]
            entry["parity"] = (oracle_parity_softmax(last, w, rows) if op == "softmax"
                               else oracle_parity_row_sum(last, w, rows))
        entries.append(entry)
        del xs, ys
        torch.cuda.empty_cache()
    return entries


def run_variants(args, torch, rrs, dev, rank):
    """The variants on the softmax skeleton, each on its workload: log-softmax, in place,
    row max / mean, column softmax and GeLU -- kernel time, roofline fraction, parity."""
    import oracle
    peak, peak_kind = measured_hbm_peak()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    W = dict(workloads.WORKLOADS)
    W.update(workloads.VARIANT_WORKLOADS)
    cases = [("c2", "log_softmax"), ("c3", "log_softmax"), ("c5", "log_softmax"),
             ("c3", "softmax_in_place"), ("c5", "softmax_unaligned"), ("c3", "row_max"), ("c3", "row_mean"),
             ("cols_c2", "softmax_cols"), ("cols_c4", "softmax_cols"), ("gelu_16k", "gelu")]
    entries = []
    for name, op in cases:
        if not selected(args, name, op):
            continue
        w = W[name]
        M, N = w.M, w.N
        x_host = workloads.matrix(w)
        reduce = op in ("row_max", "row_mean")
        alg = 4 * M * N + 4 * M if reduce else 8 * M * N
        npairs = l2_pairs(torch, alg)
        if op == "softmax_unaligned":
            # rows one float past a 16-byte boundary, stride N + 1: no float4
            # access, and x and y misaligned differently, so the planner's
            # scalar paths (the two-pass split for rows this long)
            ld_u = N + 1
            xs, ys = [], []
            for _ in range(npairs):
                xb = torch.zeros(M * ld_u + 4, dtype=torch.float32, device=dev)
                xv = xb[1:1 + M * ld_u].view(M, ld_u)
                xv[:, :N].copy_(torch.from_numpy(x_host))
                xs.append(xv)
                yb = torch.zeros(M * ld_u + 4, dtype=torch.float32, device=dev)
                ys.append(yb[2:2 + M * ld_u].view(M, ld_u))
        else:
            xs = [torch.from_numpy(x_host).to(dev) for _ in range(npairs)]
            ys = [torch.empty(M, dtype=torch.float32, device=dev) if reduce else
                  (xs[r] if op == "softmax_in_place" else torch.empty_like(xs[0]))
                  for r in range(npairs)]
        if op not in ("softmax_in_place", "softmax_unaligned"):
            touch(ys)

        def call(k, op=op, M=M, N=N):
            r = k % npairs
            x, y = xs[r].data_ptr(), ys[r].data_ptr()
            if op == "log_softmax":
                rrs.softmax_rows_ex_ptr(x, N, y, N, M, N, rrs.LOG_SOFTMAX, sh)
            elif op == "softmax_in_place":
                rrs.softmax_rows_ex_ptr(x, N, x, N, M, N, 0, sh)
            elif op == "softmax_unaligned":
                rrs.softmax_rows_ex_ptr(x, N + 1, y, N + 1, M, N, 0, sh)
            elif op == "row_max":
                rrs.row_max_ptr(x, y, M, N, N, sh)
            elif op == "row_mean":
                rrs.row_mean_ptr(x, y, M, N, N, sh)
            elif op == "softmax_cols":
                rrs.softmax_cols_ptr(x, N, y, N, M, N, 0, sh)
            else:
                rrs.gelu_ptr(x, y, M * N, sh)

        for k in range(3):
            call(k)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for k in range(args.suite_steps):
            call(k)
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / args.suite_steps
        gbs = alg / (ms / 1e3) / 1e9
        entry = {"workload": name, "op": op, "M": M, "N": N, "ms_per_call": ms, "hbm_gbs": gbs,
                 "frac_of_8tbs": gbs / ROOFLINE_GBS, "frac_of_peak": gbs / peak,
                 "peak_kind": f"of {peak_kind}", "calls_timed": args.suite_steps,
                 "l2": f"{npairs} rotating pair(s)"}
        if op == "softmax_cols":
            entry["path"] = rrs.plan_softmax_cols(M, N)["path_name"]
        if op == "softmax_unaligned":
            entry["path"] = rrs.plan_softmax(M, N, N + 1, False)["path_name"]
            entry["ld"] = N + 1
        if rank == 0:
            # one fresh call on the original x, compared with the oracle on a sample
            if op == "softmax_unaligned":
                xs[0][:, :N].copy_(torch.from_numpy(x_host))
            else:
                xs[0].copy_(torch.from_numpy(x_host))
            call(0)
            torch.cuda.synchronize()
            rows = sampled_rows(M, 6, w.seed)
            if op == "softmax_unaligned":
                got = ys[0][rows, :N].cpu().numpy().astype(np.float64)
                want = oracle.softmax_rows(x_host[rows].astype(np.float64))
                entry["parity"] = {"rows_checked": len(rows), "max_abs": float(np.max(np.abs(got - want)))}
            elif op in ("log_softmax", "softmax_in_place"):
                got = ys[0][rows].cpu().numpy().astype(np.float64)
                want = (oracle.log_softmax_rows if op == "log_softmax" else oracle.softmax_rows)(
                    x_host[rows].astype(np.float64))
                fin = np.isfinite(want)
                entry["parity"] = {"rows_checked": len(rows),
                                   "max_abs": float(np.max(np.abs(got[fin] - want[fin])))}
            elif reduce:
                got = ys[0][rows].cpu().numpy().astype(np.float64)
                want = (oracle.row_max if op == "row_max" else oracle.row_mean)(
                    x_host[rows].astype(np.float64))
                entry["parity"] = {"rows_checked": len(rows),
                                   "max_abs": float(np.max(np.abs(got - want)))}
            elif op == "softmax_cols":
                cols = sampled_rows(N, 6, w.seed + 1)
                got = ys[0][:, cols].cpu().numpy().astype(np.float64)
                want = oracle.softmax_cols(x_host[:, cols].astype(np.float64))
                entry["parity"] = {"cols_checked": len(cols),
                                   "max_abs": float(np.max(np.abs(got - want)))}
            else:
                rng = np.random.default_rng(w.seed)
                idx = rng.integers(0, M * N, size=100000)
                got = ys[0].view(-1)[torch.from_numpy(idx).to(dev)].cpu().numpy().astype(np.float64)
                want = oracle.gelu(x_host.reshape(-1)[idx].astype(np.float64))
                entry["parity"] = {"elements_checked": int(idx.size),
                                   "max_rel": float(np.max(np.abs(got - want) /
                                                           np.maximum(np.abs(want), 1e-30)))}
        entries.append(entry)
        del xs, ys, x_host
        torch.cuda.empty_cache()
    entries.extend(run_attention(args, torch, rrs, dev, rank))
    return entries


def summary(out: dict) -> dict:
    """One short entry per timed row: "workload:op" -> [microseconds per call,
    fraction of the measured peak (HBM, or bf16 tensor for attention)]."""
    rows = {f"headline {out['config']['workload'].split(':')[0]}:softmax":
            [round(out["ms_per_step"] * 1e3, 2), round(out["roofline"]["frac"], 3)]}
    for e in out.get("suite", []) + out.get("variants", []):
        frac = e["roofline"]["frac"] if "roofline" in e else e["frac_of_peak"]
        rows[f"{e['workload']}:{e['op']}"] = [round(e["ms_per_call"] * 1e3, 2), round(frac, 3)]
        if "copy_us" in e:
            rows[f"{e['workload']}:{e['op']}"].append(round(e["copy_us"], 2))
    return rows


def selected(args, name: str, op: str) -> bool:
    """Whether --only lets the suite / variant entry workload:op run."""
    if not args.only:
        return True
    return f"{name}:{op}" in {t.strip() for t in args.only.split(",")}


def attention_flops(L: int, S: int, d: int, causal: bool) -> int:
    """FLOPs of one head: 2 d per (query, visible key) pair for Q K^T and as many for P V."""
    if not causal:
        pairs = L * S
    else:  # key j visible to query i when j <= i + S - L
        pairs = sum(max(0, min(S, i + S - L + 1)) for i in range(L))
    return 4 * d * pairs


def run_attention(args, torch, rrs, dev, rank):
    """Fused attention forward (softmax inside the two products) on its workloads:
    kernel time, tensor-core roofline fraction against the measured bf16 peak, and
    parity of sampled heads and rows against the oracle."""
    import oracle
    peak, peak_kind = measured_bf16_peak()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    entries = []
    for name, w in workloads.ATTENTION_WORKLOADS.items():
        if not selected(args, name, "attention_fwd"):
            continue
        q, k, v = workloads.attention_inputs(w)
        dq, dk, dv = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) for a in (q, k, v))
        o = torch.empty(w.BH, w.L, w.d, dtype=torch.float32, device=dev)
        lse = torch.empty(w.BH, w.L, dtype=torch.float32, device=dev)

        def call():
            rrs.attention_ptr(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              w.BH, w.L, w.S, w.d, w.causal, 0.0, sh)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        steps = max(3, min(args.suite_steps, 20))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            call()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        flops = w.BH * attention_flops(w.L, w.S, w.d, w.causal)
        tflops = flops / (ms / 1e3) / 1e12
        entry = {"workload": name, "op": "attention_fwd", "B": w.B, "H": w.H, "L": w.L, "S": w.S,
                 "d": w.d, "causal": w.causal, "dtype": "bf16 in, fp32 accumulate and out",
                 "ms_per_call": ms, "tflops": tflops,
                 "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                              "frac": tflops / peak, "peak_kind": f"of {peak_kind}",
                              "flops_per_launch": flops},
                 "calls_timed": steps, "inputs": "resident (K/V of one head: 2 MiB, L2-resident)"}
        if rank == 0:
            h = w.BH // 2
            rows = sampled_rows(w.L, 6, w.seed)
            f64 = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            want_o, want_l = oracle.attention(f64(q[h]), f64(k[h]), f64(v[h]), causal=w.causal)
            got_o = o[h][rows].cpu().numpy().astype(np.float64)
            got_l = lse[h][rows].cpu().numpy().astype(np.float64)
            entry["parity"] = {"head": h, "rows_checked": len(rows),
                               "max_abs_o": float(np.max(np.abs(got_o - want_o[rows]))),
                               "max_abs_lse": float(np.max(np.abs(got_l - want_l[rows])))}
        entries.append(entry)
        del dq, dk, dv, o, lse
        torch.cuda.empty_cache()
    return entries


# --------------------------------------------------------- reference arm ---

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    # size each step's sample so the whole run takes about a minute for any --steps
    probe = workloads.matrix(w, rows=range(min(w.M, 64)))
    t0 = time.perf_counter()
    oracle.softmax_rows(probe)
    per_row = (time.perf_counter() - t0) / probe.shape[0]
    total_steps = args.steps + max(args.warmup, 3)
    sample_rows = int(max(1, min(w.M, 60.0 / (total_steps * per_row))))
    x = workloads.matrix(w, rows=range(sample_rows))
    for _ in range(max(args.warmup, 3)):
        oracle.softmax_rows(x)
    cpu0 = time.process_time()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.softmax_rows(x)
    dt = time.perf_counter() - t0
    cpu = time.process_time() - cpu0
    value = sample_rows * args.steps / dt
    cores = max(1, round(cpu / dt))
    sample = f"{sample_rows} of {w.M} rows of {w.name} ({w.M}x{w.N}) per step, float64 numpy oracle"
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: softmax_rows fp32 {w.M}x{w.N} {w.dist} seed {w.seed}",
                   "M": w.M, "N": w.N, "ld": w.N, "path": "oracle (CPU)"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    line = json.dumps(out)
    print(line, flush=True)
    if args.json_out:
        with open(args.json_out, "w") as f:
            f.write(line + "\n")


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
