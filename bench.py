"""Benchmark: NVFP4 block-scaled batched GEMV on GB300, through the C ABI.

Headline workload: M=16384, K=8192, L=16 (1.21 GB per call, plain scales), the
largest of the five workloads.  One step is one ``nvfp4_gemv`` call, the whole
hot path.

Timed region (``value``): K back-to-back calls replayed from a CUDA graph,
bracketed by CUDA events on the launching stream; that K-call window is
repeated R times (until the windows add up to at least 0.5 s) and ``value``
is the median over the windows of elapsed / K, in microseconds per call.
Consecutive calls rotate over resident copies of the inputs (at least 2, and
together at least 32x the 129 MB L2), so every call reads its operands from
HBM (cold L2): the kernel streams A with an L2 evict_first policy, and such
lines outlive a rotation of only 2x L2 (ncu: 25.5 of 33.1 MB per call read
from DRAM there, 33.08 MB over 4 GB of sets).  Consecutive calls do overlap: each call is launched with
programmatic stream serialization, so its CTAs start (and prefetch their first
lines of A into L2) while the previous call's last CTAs finish.  Each line
therefore also carries ``single_call_l2_flushed_us``: one event-bracketed call
after writing a buffer of twice the L2 size, nothing overlapping it.

Before the headline line, one line per (workload, scale layout) of the other
workloads (the pages' three timed shapes, the small parity shape, and the
headline shape with pre-permuted scales) gives the same two figures
(``--no-extra`` skips them).

``e2e``: the same call through the C ABI with host buffers: each step copies
a, b, sfa, sfb from pinned host memory, runs the GEMV and copies c back.

``cpu_baseline`` and ``--impl reference``: the CPU oracle on the host cores
(every core, one thread per core over disjoint rows) on a bounded sample of
the same workload, scaled to a whole call; the one-core figure is given beside
it.

``--all-configs`` also times the scale repack, the extended entry point and
the small-N GEMM (extra JSON lines after the headline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_block_scaled_gemv_gb300 import synthetic  # noqa: E402

METRIC = "us/call (cold L2) and achieved HBM GB/s as % of GB300 peak, NVFP4 GEMV"
UNIT = "us/call"
WORKLOAD = synthetic.WORKLOADS[4]  # ("M16384_K8192_L16", 16384, 8192, 16)
# Rotation for cold-L2 timing.  The GEMV streams A with an L2 evict_first
# policy; measured with ncu on GB300 (dram__bytes_read.sum per call, graph of
# back-to-back calls, no cache flush between them), M7168_K2048_L4 rotating
# over 8 sets (265 MB, 2x L2) read 25.5 of its 33.1 MB per call from DRAM
# (evict_first lines outlive the rotation), over 120 sets (4 GB) 33.08 MB.
COLD_L2_MULTIPLE = 32
MAX_SETS = 1024
MIN_WINDOW_S = 0.5  # the timed K-call windows add up to at least this
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_NAMES = ("direct", "pipelined", "tensor", "blockdot", "blockwise")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20,
                    help="calls per timed window (each window is timed on its own)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--layout", choices=["plain", "permuted"], default="plain")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload lines printed before the headline")
    ap.add_argument("--all-configs", action="store_true",
                    help="also time the scale repack, the extended entry point and the "
                         "small-N GEMM (lines after the headline)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workload", default=WORKLOAD[0],
                    help="one of " + ", ".join(w[0] for w in synthetic.WORKLOADS) +
                         ", or any M<m>_K<k>_L<l>")
    ap.add_argument("--ncu", action="store_true",
                    help="only run warmup+steps calls of --workload (for profiler captures)")
    ap.add_argument("--schedule", default=None,
                    help="with --ncu: KERNEL,LANES_PER_ROW,K_SPLIT,CTAS for nvfp4_gemv_explicit "
                         "instead of the chosen schedule")
    ap.add_argument("--rotate", type=int, default=0,
                    help="with --ncu: calls rotate over this many input sets (default 2)")
    ap.add_argument("--graph", action="store_true",
                    help="with --ncu: replay the --steps calls from one CUDA graph")
    ap.add_argument("--gemm-workload", default=None,
                    help="with --ncu: run nvfp4_gemm_small_n on this decode-batch workload "
                         "(e.g. M7168_N8_K2048_L4) instead of the GEMV")
    ap.add_argument("--repack", action="store_true",
                    help="with --ncu: run the scale repack of --workload's sfa instead of the GEMV")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# ranks (replicas only: each rank runs the whole workload on its own GPU)
# ---------------------------------------------------------------------------

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float) -> float:
    """Largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_id: str, interval_ms: int = 50):
        self.samples = []
        self.proc = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        # only samples taken inside the timed region count
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(p[1]) for p in inside if p[1].replace(".", "", 1).isdigit()]
        smax = [float(p[2]) for p in inside if p[2].replace(".", "", 1).isdigit()]
        reasons = set()
        for p in inside:
            for name, val in zip(REASON_NAMES, p[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index].strip()
    return str(dev_index)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

# The sources each GEMV kernel is compiled from (the host planner's choice is
# checked through the recorded schedule instead).
_COMMON_SOURCES = ("internal.h", "ptx.cuh", "epilogue.cuh")
KERNEL_SOURCES = {
    "direct": _COMMON_SOURCES + ("gemv_kernel.cuh", "gemv_plain.cu", "gemv_permuted.cu"),
    "pipelined": _COMMON_SOURCES + ("gemv_kernel.cuh", "gemv_async.cuh", "gemv_async_plain.cu",
                                    "gemv_async_permuted.cu"),
    "tensor": _COMMON_SOURCES + ("tc_ptx.cuh", "gemv_tc.cu"),
    "blockdot": _COMMON_SOURCES + ("tc_ptx.cuh", "gemv_blockdot.cu"),
    "blockwise": _COMMON_SOURCES + ("gemv_kernel.cuh", "gemv_blockwise.cu"),
}
_SCHEDULE_KEYS = ("kernel", "lanes_per_row", "k_split", "ctas")


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources one GEMV kernel (a KERNEL_NAMES entry) is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_gemv_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(workload: str, layout: str, schedule: dict):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernels'
    sources are unchanged since it was captured and the launch runs the
    schedule that was captured (a launch's traffic depends on both)."""
    path = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(f"{workload}/{layout}")
    kernel = KERNEL_NAMES[schedule["kernel"]]
    if not entry or entry.get("kernel") != kernel or \
            entry.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    captured = entry.get("schedule") or {}
    if any(captured.get(k) != schedule.get(k) for k in _SCHEDULE_KEYS):
        return None
    return entry.get("dram_bytes_per_launch")


class DeviceProblem:
    """`sets` resident copies of one problem's inputs and outputs."""

    def __init__(self, torch, nv, p, M, K, L, layout, dev, sets):
        self.M, self.K, self.L, self.layout = M, K, L, layout
        a = torch.from_numpy(p["a"]).to(dev)
        b = torch.from_numpy(p["b"]).to(dev)
        sfa = torch.from_numpy(p["sfa"]).to(dev)
        sfb = torch.from_numpy(p["sfb"]).to(dev)
        if layout == nv.SF_PERMUTED_128x4:
            sfa = nv.repack_scales(sfa)
            sfb = nv.repack_scales(sfb.view(L, 1, K // 16))
        self.sets = []
        for i in range(sets):
            self.sets.append({
                "a": a.clone(), "b": b.clone(), "sfa": sfa.clone(), "sfb": sfb.clone(),
                "c": torch.empty((L, M), dtype=torch.float16, device=dev)})
        del a, b, sfa, sfb

    def call(self, nv, i, stream_handle):
        s = self.sets[i % len(self.sets)]
        nv.nvfp4_gemv(s["a"].data_ptr(), s["b"].data_ptr(), s["sfa"].data_ptr(),
                      s["sfb"].data_ptr(), s["c"].data_ptr(), self.M, self.K, self.L,
                      self.layout, stream_handle)


class ExtProblem(DeviceProblem):
    """DeviceProblem called through nvfp4_gemv_ex: an output scale, an fp16
    [L][M] bias, and b as row 0 of an [L][pad_rows][K/2] buffer."""

    def __init__(self, torch, nv, p, M, K, L, layout, dev, sets, pad_rows=8, alpha=0.5):
        super().__init__(torch, nv, p, M, K, L, layout, dev, sets)
        self.alpha = alpha
        self.b_stride = pad_rows * (K // 2)
        gen = torch.Generator().manual_seed(0)
        for s in self.sets:
            padded = torch.zeros((L, pad_rows, K // 2), dtype=torch.uint8, device=dev)
            padded[:, 0, :] = s["b"].view(L, K // 2)
            s["b"] = padded
            s["bias"] = (torch.randn((L, M), generator=gen) * 4).to(torch.float16).to(dev)

    def call(self, nv, i, stream_handle):
        s = self.sets[i % len(self.sets)]
        nv.nvfp4_gemv_ex(s["a"].data_ptr(), s["b"].data_ptr(), s["sfa"].data_ptr(),
                         s["sfb"].data_ptr(), s["c"].data_ptr(), self.M, self.K, self.L,
                         self.layout, alpha=self.alpha, bias=s["bias"].data_ptr(),
                         b_batch_stride=self.b_stride, stream=stream_handle)


def time_graph(torch, nv, prob, steps, warmup, stream, min_window_s=MIN_WINDOW_S, period=None):
    """Microseconds per call over windows of `steps` back-to-back calls.

    Call i uses input set i % period (period = len(prob.sets) by default).
    The calls are captured into CUDA graphs of g calls each (g the largest
    divisor of `steps` up to 64), graph j holding calls j*g .. j*g+g-1, as
    many graphs as one full turn of the rotation takes; a window replays
    steps/g of them in turn, continuing the rotation from the previous window.
    Each window is bracketed by its own pair of CUDA events on the launching
    stream; windows follow one another until they add up to min_window_s.
    Returns (median us per call over the windows, (t0, t1) host monotonic
    bounds of the timed region, calls timed, windows)."""
    handle = stream.cuda_stream
    period = period or len(prob.sets)
    g_size = max(d for d in range(1, min(64, steps) + 1) if steps % d == 0)
    n_graphs = period // math.gcd(period, g_size)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            prob.call(nv, i, handle)
    stream.synchronize()
    graphs = []
    for j in range(n_graphs):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(j * g_size, (j + 1) * g_size):
                prob.call(nv, i, handle)
        graphs.append(graph)
    turn = [0]

    def replay_window():
        for _ in range(steps // g_size):
            graphs[turn[0]].replay()
            turn[0] = (turn[0] + 1) % n_graphs

    # warm every graph and estimate one window's length
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for graph in graphs:
            graph.replay()
        e0.record(stream)
        replay_window()
        e1.record(stream)
    stream.synchronize()
    est_s = max(e0.elapsed_time(e1) * 1e-3, 1e-6)
    windows = max(1, min(100000, int(min_window_s / est_s) + 1))
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(windows)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    with torch.cuda.stream(stream):
        for s0, s1 in events:
            s0.record(stream)
            replay_window()
            s1.record(stream)
    stream.synchronize()
    t1 = time.monotonic()
    torch.cuda.synchronize()
    barrier()
    per_call = [s0.elapsed_time(s1) * 1e3 / steps for s0, s1 in events]
    return statistics.median(per_call), (t0, t1), steps * windows, windows


def l2_bytes(torch, dev) -> int:
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)


def time_single_flushed(torch, nv, prob, reps, stream):
    """Median and min microseconds of one event-bracketed call, each after
    writing a buffer of twice the L2 size (nothing else runs in the bracket)."""
    dev = prob.sets[0]["a"].device
    flush = torch.empty(2 * l2_bytes(torch, dev), dtype=torch.uint8, device=dev)
    handle = stream.cuda_stream
    times = []
    with torch.cuda.stream(stream):
        for i in range(reps):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            prob.call(nv, i, handle)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
    del flush
    return statistics.median(times), min(times)


def time_e2e(torch, nv, p, M, K, L, dev, steps, stream):
    """End-to-end per-step microseconds with host buffers (pinned)."""
    host = {k: torch.from_numpy(v).pin_memory() for k, v in p.items()}
    d = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    c = torch.empty((L, M), dtype=torch.float16, device=dev)
    c_host = torch.empty((L, M), dtype=torch.float16).pin_memory()
    handle = stream.cuda_stream

    def step():
        for k in ("a", "b", "sfa", "sfb"):
            d[k].copy_(host[k], non_blocking=True)
        nv.nvfp4_gemv(d["a"].data_ptr(), d["b"].data_ptr(), d["sfa"].data_ptr(),
                      d["sfb"].data_ptr(), c.data_ptr(), M, K, L, nv.SF_PLAIN, handle)
        c_host.copy_(c, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    stream.synchronize()
    h2d = sum(v.numel() * v.element_size() for k, v in host.items())
    d2h = c_host.numel() * c_host.element_size()
    del host, d, c, c_host
    return e0.elapsed_time(e1) * 1e3 / steps, h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_us_per_call(p, M, K, L, budget_s: float, threads: int = 1):
    """The oracle on `threads` host cores over a bounded sample of outputs,
    scaled to a full call.  Each thread evaluates its own random outputs (the
    oracle's C routine runs without the interpreter lock); the oracle itself
    is unchanged.  Returns (us_per_call, sample description)."""
    import concurrent.futures

    import oracle

    oracle.build()
    rows = L * M
    rng = np.random.default_rng(0)
    n = 64
    spent, done = 0.0, 0

    def work(idx):
        li, mi = idx
        oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)

    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        while True:
            chunks = [(rng.integers(0, L, n), rng.integers(0, M, n)) for _ in range(threads)]
            t0 = time.perf_counter()
            list(pool.map(work, chunks))
            spent += time.perf_counter() - t0
            done += n * threads
            if spent >= budget_s:
                break
            n = min(8192, n * 2)
    us = spent / done * rows * 1e6
    return us, (f"{done} random outputs (full K each) of the {rows}-output call in {spent:.2f} s "
                f"of wall time on {threads} host core(s), scaled to the whole call")


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    name, M, K, L = workload_by_name(args.workload)
    p = synthetic.make_problem(M, K, L, seed=0)
    cores = host_cores()
    # every step is one bounded sample; the whole run stays within about a minute
    per_step_budget = max(0.02, min(10.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_us_per_call(p, M, K, L, per_step_budget / 4, cores)
    vals, samples = [], []
    for _ in range(args.steps):
        us, sample = oracle_us_per_call(p, M, K, L, per_step_budget, cores)
        vals.append(us)
        samples.append(sample)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "M": M, "K": K, "L": L, "scale_layout": "plain"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": samples[-1]},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def rotating_sets(nbytes: int, steps: int, l2: int) -> int:
    """Input copies to rotate over: together at least COLD_L2_MULTIPLE x the L2
    (at least 2, at most MAX_SETS), and a divisor of `steps` or a multiple of it
    (so that a window of `steps` calls takes whole turns or whole fractions of
    the rotation)."""
    need = max(2, min(MAX_SETS, -(-COLD_L2_MULTIPLE * l2 // nbytes)))
    if need <= steps:
        return next(d for d in range(need, steps + 1) if steps % d == 0)
    return -(-need // steps) * steps


def l2_state(nbytes: int, sets: int, l2: int) -> str:
    if sets * nbytes >= COLD_L2_MULTIPLE * l2:
        return (f"{sets} rotating input sets, {sets * nbytes / 1e9:.2f} GB >= "
                f"{COLD_L2_MULTIPLE}x L2 (cold L2 every call)")
    return (f"{sets} rotating input sets, {sets * nbytes / 1e6:.1f} MB: less than "
            f"{COLD_L2_MULTIPLE}x L2, inputs partly L2-resident")


def kernel_name(nv, torch, dev, M, K, L, layout) -> str:
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = nv.nvfp4_gemv_plan(M, K, L, layout, sms)
    return KERNEL_NAMES[plan["kernel"]]


def config_line(torch, nv, dev, stream, peaks, wname, wM, wK, wL, lay_name, steps, warmup):
    """One (workload, layout): graph-replayed back-to-back calls and single
    L2-flushed calls, as a compact JSON line."""
    lay = nv.SF_PLAIN if lay_name == "plain" else nv.SF_PERMUTED_128x4
    wp = synthetic.make_problem(wM, wK, wL, seed=0)
    wbytes = synthetic.algorithmic_bytes(wM, wK, wL)
    wsteps = max(steps, 64)
    sets = rotating_sets(wbytes, wsteps, l2_bytes(torch, dev))
    wprob = DeviceProblem(torch, nv, wp, wM, wK, wL, lay, dev, sets)
    wus, _, calls, windows = time_graph(torch, nv, wprob, wsteps, max(warmup, 16), stream,
                                        min_window_s=0.25)
    smed, smin = time_single_flushed(torch, nv, wprob, 20, stream)
    gbs = wbytes / (wus * 1e-6) / 1e9
    sgbs = wbytes / (smed * 1e-6) / 1e9
    del wprob
    torch.cuda.empty_cache()
    return {"kind": "per_workload", "workload": wname, "scale_layout": lay_name,
            "kernel": kernel_name(nv, torch, dev, wM, wK, wL, lay),
            "bytes_per_call": wbytes, "us_per_call": round(wus, 3), "gb_per_s": round(gbs, 1),
            "pct_of_hbm_peak": round(100 * gbs / peaks["hbm_gbs"], 2),
            "single_call_l2_flushed_us": round(smed, 3),
            "single_call_l2_flushed_min_us": round(smin, 3),
            "single_call_pct_of_hbm_peak": round(100 * sgbs / peaks["hbm_gbs"], 2),
            "rotating_sets": sets, "l2": l2_state(wbytes, sets, l2_bytes(torch, dev)),
            "calls": calls, "windows": windows}


def run_native(args):
    import torch

    import nvfp4_block_scaled_gemv_gb300 as nv
    from nvfp4_block_scaled_gemv_gb300 import build as libbuild

    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    libbuild.build()
    nv.library()
    stream = torch.cuda.Stream(device=dev)
    peaks = measured_peaks()

    name, M, K, L = workload_by_name(args.workload)
    layout = nv.SF_PLAIN if args.layout == "plain" else nv.SF_PERMUTED_128x4

    # the other workloads and layouts first (the headline line is printed last)
    per_workload = []
    if not args.no_extra:
        for wname, wM, wK, wL in synthetic.WORKLOADS:
            for lay_name in ("plain", "permuted"):
                if (wname, lay_name) == (name, args.layout):
                    continue
                line = config_line(torch, nv, dev, stream, peaks, wname, wM, wK, wL, lay_name,
                                   args.steps, args.warmup)
                per_workload.append(line)
                if rank == 0:
                    print(json.dumps(line), flush=True)

    p = synthetic.make_problem(M, K, L, seed=0)
    nbytes = synthetic.algorithmic_bytes(M, K, L)
    l2 = l2_bytes(torch, dev)
    sets = rotating_sets(nbytes, args.steps, l2)
    prob = DeviceProblem(torch, nv, p, M, K, L, layout, dev, sets)

    sampler = ClockSampler(gpu_id_for_smi(torch, local)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    us, (t0, t1), calls, windows = time_graph(torch, nv, prob, args.steps, args.warmup, stream)
    if sampler:
        sampler.stop()
    us_job = max_over_ranks(us) / world  # all ranks' calls / the slowest rank's time
    us_rank = max_over_ranks(us)

    single_med, single_min = time_single_flushed(torch, nv, prob, 30, stream)
    del prob
    torch.cuda.empty_cache()
    e2e_steps = max(5, min(args.e2e_steps, int(4e9 / nbytes)))
    e2e_us, h2d, d2h = time_e2e(torch, nv, p, M, K, L, dev, e2e_steps, stream)
    e2e_us = max_over_ranks(e2e_us) / world

    if rank != 0:
        return
    cores = host_cores()
    cpu_us, cpu_sample = oracle_us_per_call(p, M, K, L, budget_s=10.0, threads=cores)
    cpu1_us, _ = oracle_us_per_call(p, M, K, L, budget_s=3.0, threads=1)
    achieved = nbytes / (us_rank * 1e-6) / 1e9
    single_gbs = nbytes / (single_med * 1e-6) / 1e9
    plan = nv.nvfp4_gemv_plan(M, K, L, layout, torch.cuda.get_device_properties(dev).multi_processor_count)
    line = {
        "metric": METRIC, "value": round(us_job, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_job / 1e3, 7),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1xe4m3->f32->f16", "data": "synthetic",
        "config": {"workload": name, "M": M, "K": K, "L": L, "scale_layout": args.layout,
                   "l2": l2_state(nbytes, sets, l2),
                   "launch": "CUDA graph of back-to-back nvfp4_gemv calls with programmatic "
                             "stream serialization: each call's CTAs start, and prefetch their "
                             "first A lines into L2, while the previous call's last CTAs finish",
                   "timing": f"{windows} event-bracketed windows of {args.steps} calls, median",
                   "bytes_per_call": nbytes, "schedule": plan,
                   "kernel": KERNEL_NAMES[plan["kernel"]]},
        "gb_per_s": round(achieved, 1),
        "pct_of_hbm_peak": round(100 * achieved / peaks["hbm_gbs"], 2),
        "single_call_l2_flushed_us": {"median": round(single_med, 3), "min": round(single_min, 3),
                                      "pct_of_hbm_peak": round(100 * single_gbs / peaks["hbm_gbs"], 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(name, args.layout, plan),
                     "peak_source": peaks["source"]},
        "cpu_baseline": {"value": round(cpu_us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": cpu_sample, "one_core_value": round(cpu1_us, 1)},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": calls,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "per_workload": [{k: w[k] for k in ("workload", "scale_layout", "kernel", "us_per_call",
                                             "pct_of_hbm_peak", "single_call_l2_flushed_us")}
                         for w in per_workload],
    }
    print(json.dumps(line), flush=True)

    if args.all_configs:
        # the scale repack (plain -> 128x4 atoms) of each workload's sfa, graph-replayed
        # over rotating buffers; bytes = plain scales read + permuted atoms written
        for wname, wM, wK, wL in synthetic.WORKLOADS:
            wp = synthetic.make_problem(wM, wK, wL, seed=0)
            src0 = torch.from_numpy(wp["sfa"]).to(dev)
            out_bytes = nv.nvfp4_permuted_scale_bytes(wM, wK, wL)
            rbytes = src0.numel() + out_bytes
            rsteps = 64
            sets = rotating_sets(rbytes, rsteps, l2)
            srcs = [src0.clone() for _ in range(sets)]
            dsts = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(sets)]
            del src0

            class _Repack:
                def call(self, nv_, i, h):
                    nv_.nvfp4_repack_scales(srcs[i % sets].data_ptr(), dsts[i % sets].data_ptr(),
                                            wM, wK, wL, h)

            rus, _, _, _ = time_graph(torch, nv, _Repack(), rsteps, 64, stream, 0.25, period=sets)
            gbs = rbytes / (rus * 1e-6) / 1e9
            print(json.dumps({"workload": wname, "kernel": "repack_scales (sfa)",
                              "us_per_call": round(rus, 3), "bytes_per_call": rbytes,
                              "gb_per_s": round(gbs, 1),
                              "pct_of_hbm_peak": round(100 * gbs / peaks["hbm_gbs"], 2),
                              "rotating_sets": sets, "calls": rsteps}), flush=True)
            del srcs, dsts
            torch.cuda.empty_cache()
        # the extended entry point on the headline shape
        wname, wM, wK, wL = synthetic.WORKLOADS[1]
        wp = synthetic.make_problem(wM, wK, wL, seed=0)
        wbytes = synthetic.algorithmic_bytes(wM, wK, wL) + 2 * wL * wM  # + the bias
        wsteps = 64
        wsets = rotating_sets(wbytes, wsteps, l2)
        wprob = ExtProblem(torch, nv, wp, wM, wK, wL, nv.SF_PLAIN, dev, wsets)
        wus, _, _, _ = time_graph(torch, nv, wprob, wsteps, 64, stream, 0.25)
        gbs = wbytes / (wus * 1e-6) / 1e9
        print(json.dumps({"workload": wname, "scale_layout": "plain",
                          "path": "nvfp4_gemv_ex: alpha 0.5, fp16 bias, b in an [L][8][K/2] buffer",
                          "us_per_call": round(wus, 3), "gb_per_s": round(gbs, 1),
                          "pct_of_hbm_peak": round(100 * gbs / peaks["hbm_gbs"], 2),
                          "rotating_sets": wsets, "calls": wsteps}), flush=True)
        del wprob
        torch.cuda.empty_cache()
        # the small-N GEMM (tensor-core kernel) on the decode-batch workloads;
        # bytes = A + sfa + N x (b + sfb) read + N x c written
        for gname, gM, gN, gK, gL in synthetic.GEMM_WORKLOADS:
            gp = synthetic.make_gemm_problem(gM, gN, gK, gL, seed=0)
            gbytes = synthetic.gemm_algorithmic_bytes(gM, gN, gK, gL)
            gsteps = 64
            gsets = rotating_sets(gbytes, gsteps, l2)
            a0 = torch.from_numpy(gp["a"]).to(dev)
            b0 = torch.from_numpy(gp["b"]).to(dev)
            sa0 = nv.repack_scales(torch.from_numpy(gp["sfa"]).to(dev))
            sb0 = nv.repack_scales(torch.from_numpy(gp["sfb"]).to(dev))
            gs = [(a0.clone(), b0.clone(), sa0.clone(), sb0.clone(),
                   torch.empty(gL * gN * gM, dtype=torch.float16, device=dev)) for _ in range(gsets)]
            del a0, b0, sa0, sb0

            class _Gemm:
                def call(self, nv_, i, h):
                    x = gs[i % gsets]
                    nv_.nvfp4_gemm_small_n(x[0].data_ptr(), x[1].data_ptr(), x[2].data_ptr(),
                                           x[3].data_ptr(), x[4].data_ptr(), gM, gN, gK, gL,
                                           stream=h)

            gus, _, _, _ = time_graph(torch, nv, _Gemm(), gsteps, 64, stream, 0.25, period=gsets)
            gbs = gbytes / (gus * 1e-6) / 1e9
            print(json.dumps({"workload": gname, "path": "nvfp4_gemm_small_n (tensor cores)",
                              "N": gN, "us_per_call": round(gus, 3), "bytes_per_call": gbytes,
                              "gb_per_s": round(gbs, 1),
                              "pct_of_hbm_peak": round(100 * gbs / peaks["hbm_gbs"], 2),
                              "rotating_sets": gsets, "calls": gsteps}), flush=True)
            del gs
            torch.cuda.empty_cache()
        assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0, "a tensor-core pipeline wait ran out"


def workload_by_name(name: str):
    """(name, M, K, L) of a benchmark workload, or of any "M<m>_K<k>_L<l>"."""
    for w in synthetic.WORKLOADS:
        if w[0] == name:
            return w
    m = re.fullmatch(r"M(\d+)_K(\d+)_L(\d+)", name)
    if not m:
        raise SystemExit(f"unknown workload {name!r}")
    return (name, int(m.group(1)), int(m.group(2)), int(m.group(3)))


def run_profile_case(args):
    """Plain calls of one workload, nothing else on the GPU but input upload."""
    import torch

    import nvfp4_block_scaled_gemv_gb300 as nv
    from nvfp4_block_scaled_gemv_gb300 import build as libbuild

    libbuild.build()
    dev = torch.device("cuda", 0)
    if args.gemm_workload:
        gname, gM, gN, gK, gL = next(w for w in synthetic.GEMM_WORKLOADS
                                     if w[0] == args.gemm_workload)
        gp = synthetic.make_gemm_problem(gM, gN, gK, gL, seed=0)
        a = torch.from_numpy(gp["a"]).to(dev)
        b = torch.from_numpy(gp["b"]).to(dev)
        sfa = nv.repack_scales(torch.from_numpy(gp["sfa"]).to(dev))
        sfb = nv.repack_scales(torch.from_numpy(gp["sfb"]).to(dev))
        c = torch.empty(gL * gN * gM, dtype=torch.float16, device=dev)
        gstream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        for _ in range(args.warmup + args.steps):
            nv.nvfp4_gemm_small_n(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                                  c.data_ptr(), gM, gN, gK, gL, stream=gstream.cuda_stream)
        gstream.synchronize()
        assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0
        print(f"profile case done: {gname} small-N GEMM {args.warmup}+{args.steps} calls")
        return
    name, M, K, L = workload_by_name(args.workload)
    layout = nv.SF_PLAIN if args.layout == "plain" else nv.SF_PERMUTED_128x4
    p = synthetic.make_problem(M, K, L, seed=0)
    stream = torch.cuda.Stream(device=dev)
    if args.repack:
        src = torch.from_numpy(p["sfa"]).to(dev)
        dst = torch.empty(nv.nvfp4_permuted_scale_bytes(M, K, L), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for _ in range(args.warmup + args.steps):
            nv.nvfp4_repack_scales(src.data_ptr(), dst.data_ptr(), M, K, L, stream.cuda_stream)
        stream.synchronize()
        print(f"profile case done: {name} sfa repack {args.warmup}+{args.steps} calls")
        return
    prob = DeviceProblem(torch, nv, p, M, K, L, layout, dev, args.rotate or 2)
    torch.cuda.synchronize()
    sched = [int(v) for v in args.schedule.split(",")] if args.schedule else None

    def one(i):
        if sched is None:
            prob.call(nv, i, stream.cuda_stream)
        else:
            s = prob.sets[i % len(prob.sets)]
            nv.nvfp4_gemv_explicit(s["a"].data_ptr(), s["b"].data_ptr(), s["sfa"].data_ptr(),
                                   s["sfb"].data_ptr(), s["c"].data_ptr(), M, K, L, layout,
                                   *sched, stream=stream.cuda_stream)

    if args.graph:
        # the benchmark's launch form: the calls replayed from one CUDA graph
        # (warm-up calls run eagerly before the capture)
        for i in range(args.warmup):
            one(i)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(args.steps):
                one(i)
        graph.replay()
    else:
        for i in range(args.warmup + args.steps):
            one(i)
    stream.synchronize()
    print(f"profile case done: {name} {args.layout} {args.warmup}+{args.steps} calls "
          f"over {len(prob.sets)} input sets{' (graph)' if args.graph else ''}")


def main():
    args = parse_args()
    if args.ncu:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
