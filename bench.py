"""Benchmark of the skinny BF16 linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload router|smallest|decode|mlp|prefill] [--pdl]

Default workload: the MoE router sweep, M = 1..16 x (K, N) in {(4096,256),
(6144,256), (7168,256), (7168,384), (2880,128)} (80 shapes), seeded synthetic
bf16 inputs (workloads.py).  One step runs every shape once per weight copy in
its rotation: each shape owns R copies of W whose total exceeds 256 MB, so
every call reads its weights from HBM (L2-cold; x, 2..230 KB, stays L2-hot
as an activation would).  The R back-to-back calls of a shape are one CUDA
graph; CUDA events on the launching stream bracket each graph, so a shape's
time per call is its events' elapsed time / R.

metric / value: mean microseconds per call over the 80 shapes (lower is
better).  roofline: the dominant kernel's algorithmic bytes (2NK + 2MK + 2MN)
per launch over its measured average launch time, against the measured HBM
copy bandwidth.  e2e: the same calls through the public API from pinned host
buffers, with x and W copied in and out copied back inside the timed region.
cpu_baseline / --impl reference: the CPU oracle (tests' reference
implementation, f64) on the same shapes, on the host's cores.

Multi-GPU: the path does not shard across GPUs in this library (replicas
only); under torchrun each rank runs the same sweep on its own GPU and rank 0
reports the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

L2_COLD_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def algo_bytes(M, N, K, bias):
    return 2 * N * K + 2 * M * K + 2 * M * N + (2 * N if bias else 0)


def algo_flops(M, N, K, bias):
    return 2 * M * N * K + (M * N if bias else 0)


def max_over_ranks(value: float, device="cpu") -> float:
    """The slowest rank's time (every rank gets it).  Works on any torch.distributed backend."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_value(per_rank_us_per_call: float, world: int) -> float:
    """Whole-job us per call when `world` replicas each ran the same calls in the same
    (max-over-ranks) time: the job completed world times as many calls."""
    return per_rank_us_per_call / world


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_points(name):
    if name == "all":
        return wl.router_smallest() + wl.router_sweep() + wl.decode_proj() + wl.mlp_bias()
    return {"router": wl.router_sweep, "smallest": wl.router_smallest, "decode": wl.decode_proj,
            "mlp": wl.mlp_bias, "prefill": wl.prefill}[name]()


def workload_desc(name):
    return {
        "router": "MoE router sweep: M=1..16 x (K,N) in {(4096,256),(6144,256),(7168,256),(7168,384),(2880,128)}, no bias",
        "smallest": "router smallest case: M=4, K=2048, N=256, no bias",
        "decode": "decode attention-input projection: M in {1,2,4,8,16,32,64}, K=7168, N=2112, no bias",
        "mlp": "dense MLP with bias: M in {1,8,64,256}, K=4096, N=14336",
        "prefill": "prefill: M in {2048,8192} x (K,N) in {(7168,2112),(4096,14336),(7168,7168)}, bias on/off",
        "all": "every skinny workload shape (router, decode, MLP)",
    }[name]


def kernel_source_hash(kernel_name):
    src = {"dotprod": ("dotprod.cuh", "dotprod.cu"), "splitk": ("splitk.cu",), "splitk_ws": ("splitk.cu",),
           "tile": ("tile.cuh", "tile.cu"), "tile_t": ("tile.cuh", "tile_t.cu"), "stream": ("stream.cu",),
           "tile2": ("tile2.cu",), "warprow": ("warprow.cu",), "warpmma": ("warpmma.cu", "warpmma_ks.cu"),
           "dotmma": ("dotmma.cu",), "dotmma_ws": ("dotmma.cu",)}.get(kernel_name)
    if src is None:
        return None
    h = hashlib.sha256()
    for f in src + ("common.cuh", "kernels.h"):
        h.update(open(os.path.join(ROOT, "moe_router_gemm_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel_name, shapes):
    """Mean DRAM bytes per launch over `shapes` (M, N, K) from the committed ncu summary
    (profiles/dram_traffic.txt), or None if a shape is missing or the kernel source
    changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(kernel_name)
    if want is None:
        return None
    table = {}
    for line in open(p):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        # kernel M N K dram_bytes_per_launch source_hash
        if len(f) >= 6 and f[0] == kernel_name:
            table[(int(f[1]), int(f[2]), int(f[3]))] = (float(f[4]), f[5])
    vals = []
    for shp in shapes:
        if shp not in table or table[shp][1] != want:
            return None
        vals.append(table[shp][0])
    return int(sum(vals) / len(vals)) if vals else None


# clock-event reasons that make a timed region unrepresentative (sw_power_cap is kept and noted)
SLOWDOWN_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def slowdowns(clocks):
    """The reasons in a ClockSampler record that call for timing the region again."""
    return sorted(set(clocks.get("reasons", [])) & SLOWDOWN_REASONS)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def cpu_model():
    """The host CPU's model name (/proc/cpuinfo, else lscpu), for the baseline's record."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


class OracleSample:
    """A bounded sample of the workload for the CPU oracle, run on host threads.

    Shapes are taken cheapest first until the estimated cost of one pass fills
    the budget; a shape too large for the budget on its own contributes its
    first rows only.  The oracle is called as it stands; ctypes releases the
    GIL, so threads evaluate different shapes (or row blocks) concurrently."""

    def __init__(self, points, budget_s=15.0, threads=None, rate_macs_per_s=0.5e9):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.threads = threads or os.cpu_count() or 1
        budget = budget_s * rate_macs_per_s * self.threads
        order = sorted(range(len(points)), key=lambda i: points[i]["M"] * points[i]["N"] * points[i]["K"])
        self.jobs = []      # (inputs, rows or None)
        self.calls = 0.0    # fraction of full calls one pass covers
        self.flops = 0.0
        acc = 0.0
        for i in order:
            pt = points[i]
            M, N, K = pt["M"], pt["N"], pt["K"]
            cost = M * N * K
            rows = None
            if acc + cost > budget:
                if self.jobs and acc > 0.5 * budget:
                    break
                nrows = max(1, int((budget - acc) // (N * K)))
                if nrows >= M:
                    nrows = M
                else:
                    rows = np.arange(nrows, dtype=np.int64)
                cost = nrows * N * K
            x, W, b = wl.make_inputs(M, N, K, pt["seed"], pt["bias"])
            self.jobs.append(((wl.bits(x), wl.bits(W), wl.bits(b)), rows))
            frac = 1.0 if rows is None else len(rows) / M
            self.calls += frac
            self.flops += algo_flops(M, N, K, pt["bias"]) * frac
            acc += cost
        self.desc = (f"{len(self.jobs)} of {len(points)} shapes"
                     + ("" if all(r is None for _, r in self.jobs) else " (largest on leading rows only)")
                     + f", one oracle call each, {self.threads} host threads")

    def _one(self, job):
        (x, W, b), rows = job
        if rows is None:
            return self.oracle.linear_bf16(x, W, b)
        return self.oracle.linear_rows_bf16(x, W, b, rows)

    def run(self, passes):
        import concurrent.futures as cf
        with cf.ThreadPoolExecutor(max_workers=self.threads) as ex:
            t0 = time.perf_counter()
            for _ in range(passes):
                list(ex.map(self._one, self.jobs))
            return time.perf_counter() - t0

    def value(self, wall, passes, large):
        if large:
            return self.flops * passes / wall / 1e12
        return wall / (self.calls * passes) * 1e6


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Shape:
    def __init__(self, pt, device, lib, plan_override=None, pdl=False):
        self.pt = pt
        M, N, K, bias = pt["M"], pt["N"], pt["K"], pt["bias"]
        self.M, self.N, self.K, self.bias = M, N, K, bias
        x, W, b = wl.make_inputs(M, N, K, pt["seed"], bias)
        self.host = (x, W, b)
        wbytes = 2 * N * K
        self.R = max(2, -(-L2_COLD_BYTES // wbytes)) if wbytes < L2_COLD_BYTES else 2
        self.x = x.to(device)
        W0 = W.to(device)
        self.Ws = [W0] + [W0.clone() for _ in range(self.R - 1)]
        self.b = b.to(device) if b is not None else None
        self.out = torch.empty(M, N, dtype=torch.bfloat16, device=device)
        # The library's recommended call: a workspace, so the dispatcher may pick
        # the cluster-free split-K where that is faster.
        self.ws = lib.new_workspace(max(256, lib.workspace_size(M, N, K)), device)
        self.plan = plan_override or lib.plan_ws(M, N, K, self.ws.numel())
        self.plan.flags = 1 if pdl else 0  # BF16L_FLAG_PDL, else the default launch mode
        self.kernel = lib.KERNEL_NAMES[self.plan.kernel]
        self.lib = lib
        self.graph = None

    def call(self, i):
        self.lib.run(self.x, self.Ws[i % self.R], self.b, self.out, plan_=self.plan, workspace=self.ws)

    def time_graph(self, stream, replays, warm=False):
        """Median in-graph microseconds per call over `replays` replays of one graph of R calls."""
        with torch.cuda.stream(stream):
            self.capture(stream, warm=warm)
            self.graph.replay()  # warm-up replay (brings the weight into L2 for the warm form)
            ms = []
            for _ in range(replays):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                self.graph.replay()
                b.record(stream)
                ms.append((a, b))
        torch.cuda.synchronize()
        self.graph = None
        return 1000.0 * statistics.median([a.elapsed_time(b) for a, b in ms]) / self.R

    def capture(self, stream, warm=False):
        """One graph of R back-to-back calls: on the R weight copies in turn (L2-cold),
        or all on copy 0 (L2-warm: after the first call the weight is L2-resident
        wherever it fits)."""
        for i in range(min(self.R, 3)):  # initialise outside capture
            self.call(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(self.R):
                self.call(0 if warm else i)
        self.graph = g


def gpu_arm(args, points, rank, world):
    import moe_router_gemm_gb300 as lib
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)

    shapes = [Shape(pt, device, lib, plan_override=forced_plan(lib, args.plan), pdl=args.pdl) for pt in points]
    with torch.cuda.stream(stream):
        for s in shapes:
            s.capture(stream)
    torch.cuda.synchronize()

    def step(events=None):
        for j, s in enumerate(shapes):
            if events is not None:
                events[j][0].record(stream)
            s.graph.replay()
            if events is not None:
                events[j][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    def timed_region():
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in shapes] for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for k in range(args.steps):
                step(ev[k])
            t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return ev, t0.elapsed_time(t1), sampler.stop()

    ev, total_ms, clocks = timed_region()
    # A region that saw a hardware or thermal slowdown is timed once more (on every rank, if any saw one).
    slowed = slowdowns(clocks)
    if (max_over_ranks(1.0 if slowed else 0.0, device="cuda") if world > 1 else (1.0 if slowed else 0.0)) > 0:
        ev, total_ms, clocks = timed_region()
        clocks = dict(clocks, remeasured_after=slowed or ["another rank's slowdown"])
    per_shape_us = []
    for j, s in enumerate(shapes):
        ms = [ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(args.steps)]
        per_shape_us.append(1000.0 * statistics.median(ms) / s.R)
    launches = args.steps * sum(s.R for s in shapes)

    # ---- the same shapes in the other launch modes: early weights (BF16L_FLAG_PDL) and serial ----
    def variant_us(flags):
        for s_ in shapes:
            s_.plan.flags = flags
        with torch.cuda.stream(stream):
            for s_ in shapes:
                s_.capture(stream)
        torch.cuda.synchronize()
        ms = [[] for _ in shapes]
        with torch.cuda.stream(stream):
            for k in range(max(3, args.steps // 2)):
                for j, s_ in enumerate(shapes):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    s_.graph.replay()
                    b.record(stream)
                    ms[j].append((a, b))
        torch.cuda.synchronize()
        for s_ in shapes:
            s_.plan.flags = base_flags
        return [1000.0 * statistics.median([a.elapsed_time(b) for a, b in ms[j]]) / s_.R
                for j, s_ in enumerate(shapes)]

    base_flags = 1 if args.pdl else 0
    pdl_us = serial_us = None
    if not args.pdl and not args.no_pdl_variant:
        pdl_us = variant_us(1)     # BF16L_FLAG_PDL
        serial_us = variant_us(2)  # BF16L_FLAG_SERIAL

    # ---- L2-warm: the same calls, every one on the same weight copy ----
    warm_us = None
    if not args.no_pdl_variant:
        for s_ in shapes:
            s_.plan.flags = 1 if args.pdl else 0
        with torch.cuda.stream(stream):
            for s_ in shapes:
                s_.capture(stream, warm=True)
                s_.graph.replay()  # brings the weight into L2
        torch.cuda.synchronize()
        warm_ms = [[] for _ in shapes]
        with torch.cuda.stream(stream):
            for k in range(max(3, args.steps // 2)):
                for j, s_ in enumerate(shapes):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    s_.graph.replay()
                    b.record(stream)
                    warm_ms[j].append((a, b))
        torch.cuda.synchronize()
        warm_us = [1000.0 * statistics.median([a.elapsed_time(b) for a, b in warm_ms[j]]) / s_.R
                   for j, s_ in enumerate(shapes)]

    # ---- e2e: public API from pinned host buffers, copies inside the timed region ----
    e2e = e2e_arm(args, shapes, lib, device, stream)

    # ---- the measured per-call floors and the other workloads of the metric (outside the timed region) ----
    floor, records = None, None
    if args.workload == "router" and not args.no_workloads and not args.only and not args.plan:
        floor = floor_record(shapes, lib, device, stream, max(3, args.sub_replays))
        for s_ in shapes:  # keep each shape's description, free its device buffers
            s_.graph, s_.Ws, s_.x, s_.out, s_.ws, s_.b = None, [], None, None, None, None
        torch.cuda.empty_cache()
        peaks = load_peaks()
        records = {}
        for name in ("smallest", "decode", "mlp", "prefill"):
            records[name] = workload_record(name, lib, device, stream, peaks, max(3, args.sub_replays))
        records["prefill_mxfp8"] = mxfp8_record(lib, device, stream, peaks, max(3, args.sub_replays))

    return dict(shapes=shapes, per_shape_us=per_shape_us, total_ms=total_ms, launches=launches,
                clocks=clocks, e2e=e2e, pdl_us=pdl_us, serial_us=serial_us, warm_us=warm_us, floor=floor,
                records=records)


def plan_str(p):
    d = p.as_dict()
    return (f"{d['kernel_name']}(threads={d['threads']},rows={d['rows_per_cta']},tokens={d['tokens_per_cta']},"
            f"split={d['split_k']},stages={d['stages']},grid={d['grid']})")


def workload_record(name, lib, device, stream, peaks, replays):
    """One workload's shapes through the dispatcher: L2-cold and L2-warm us per call, and each shape's
    fraction of its roofline (HBM for arithmetic intensity below the ridge point, else the bf16 tensor
    peak), with the kernel that ran.  Shapes are timed one at a time and freed (prefill holds GBs)."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    rows, tot_flops, tot_us, hbm_fracs = [], 0.0, 0.0, []
    for pt in workload_points(name):
        s = Shape(pt, device, lib)
        cold = s.time_graph(stream, replays)
        warm = s.time_graph(stream, replays, warm=True)
        nbytes, flops = algo_bytes(s.M, s.N, s.K, s.bias), algo_flops(s.M, s.N, s.K, s.bias)
        r = {"M": s.M, "N": s.N, "K": s.K, "bias": s.bias, "kernel": s.kernel, "plan": plan_str(s.plan),
             "us_cold": round(cold, 3), "us_warm": round(warm, 3), "weight_copies": s.R}
        if flops / nbytes < ridge:
            gbs = nbytes / (cold * 1e-6) / 1e9
            r.update(bound="hbm", GBps=round(gbs, 1), frac=round(gbs / peaks["hbm_gbs"], 4),
                     frac_warm=round(nbytes / (warm * 1e-6) / 1e9 / peaks["hbm_gbs"], 4))
            hbm_fracs.append(r["frac"])
        else:
            tf = flops / (cold * 1e-6) / 1e12
            r.update(bound="tensor", TFLOPs=round(tf, 1), frac=round(tf / peaks["bf16_tflops"], 4),
                     frac_sustained=round(tf / peaks["bf16_tflops_sustained"], 4))
            tot_flops += flops
            tot_us += cold
        rows.append(r)
        del s
        torch.cuda.empty_cache()
    rec = {"workload": workload_desc(name), "unit": "us/call", "shapes": rows,
           "mean_us_cold": round(statistics.mean(r["us_cold"] for r in rows), 3),
           "mean_us_warm": round(statistics.mean(r["us_warm"] for r in rows), 3)}
    if hbm_fracs:
        rec["hbm_frac_min"], rec["hbm_frac_max"] = min(hbm_fracs), max(hbm_fracs)
    if tot_us:
        tf = tot_flops / (tot_us * 1e-6) / 1e12
        rec["tensor_TFLOPs"] = round(tf, 1)
        rec["tensor_frac"] = round(tf / peaks["bf16_tflops"], 4)
        rec["tensor_frac_sustained"] = round(tf / peaks["bf16_tflops_sustained"], 4)
    return rec


FLOOR_CONFIGS = ((152, 1024), (304, 512), (608, 256), (1216, 128), (304, 1024), (608, 512), (1216, 256),
                 (152, 512), (304, 256), (608, 128))


def floor_record(shapes, lib, device, stream, replays):
    """Per-call floors measured the way the router calls are: (1) an empty kernel launched back to back
    in a graph (the launch cost alone), (2) for each router weight size, a pure 16-byte-load read of the
    same rotated weight copies (L2-cold), the best over a few grid shapes.  No kernel that must read W
    can beat (2); the router shapes' fraction of the HBM roofline is bounded by it."""
    sink = torch.zeros(max(g for g, _ in FLOOR_CONFIGS), dtype=torch.int32, device=device)

    def graph_us(calls, n):
        with torch.cuda.stream(stream):
            for c in calls[:2]:
                c()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in calls:
                    c()
            g.replay()
            ms = []
            for _ in range(replays):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                ms.append((a, b))
        torch.cuda.synchronize()
        return 1000.0 * statistics.median([a.elapsed_time(b) for a, b in ms]) / n

    n_empty = 256
    ser = lib.FLAG_SERIAL
    launch_us = graph_us([lambda: lib.probe_read(None, 152, 32, sink, stream=stream, flags=ser)] * n_empty, n_empty)
    launch1_us = graph_us([lambda: lib.probe_read(None, 1, 32, sink, stream=stream, flags=ser)] * n_empty, n_empty)
    launch_pdl_us = graph_us([lambda: lib.probe_read(None, 152, 32, sink, stream=stream)] * n_empty, n_empty)
    read = {}
    seen = set()
    for s in shapes:
        key = f"K{s.K}_N{s.N}"
        if key in seen:
            continue
        seen.add(key)
        best, best_serial = None, None
        for grid, threads in FLOOR_CONFIGS:
            for flags in (0, ser):
                calls = [(lambda w=w, g_=grid, t=threads, f=flags: lib.probe_read(w, g_, t, sink, stream=stream,
                                                                                 flags=f)) for w in s.Ws]
                us = graph_us(calls, len(calls))
                if flags == 0 and (best is None or us < best[0]):
                    best = (us, grid, threads)
                if flags == ser and (best_serial is None or us < best_serial[0]):
                    best_serial = (us, grid, threads)
        nbytes = 2 * s.N * s.K
        read[key] = {"us": round(best[0], 3), "weight_bytes": nbytes, "grid": best[1], "threads": best[2],
                     "GBps": round(nbytes / (best[0] * 1e-6) / 1e9, 1), "us_serial": round(best_serial[0], 3)}
    return {"note": "in-graph us per launch, L2-cold rotation as for the router calls: an empty kernel (serial "
                    "launches, and in the library's launch mode), and a read of each router weight with 16-byte "
                    "loads and no arithmetic, launched as the library's kernels are (us) and serially "
                    "(us_serial), best of the grid shapes tried; bf16_linear_probe_read",
            "empty_launch_us": round(launch_us, 3), "empty_launch_1cta_us": round(launch1_us, 3),
            "empty_launch_pdl_us": round(launch_pdl_us, 3), "read_weight": read}


def forced_plan(lib, spec):
    """The plan given by --plan (kernel name, threads, rows, tokens, split, stages[, chunks per stage]), or None."""
    if not spec:
        return None
    f = spec.split(",")
    names = ("threads", "rows_per_cta", "tokens_per_cta", "split_k", "stages", "chunks_per_stage")
    return lib.make_plan(f[0], **{k: int(v) for k, v in zip(names, f[1:])})


def eager_profile(args, points):
    """Profiling mode (for ncu launch lists): no graphs, two rotation copies per shape."""
    import moe_router_gemm_gb300 as lib
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    device = torch.device("cuda", torch.cuda.current_device())
    shapes = [Shape(pt, device, lib, plan_override=forced_plan(lib, args.plan), pdl=args.pdl) for pt in points]
    for s in shapes:
        s.R = min(s.R, 2)
        s.Ws = s.Ws[:2]
    torch.cuda.empty_cache()
    for _ in range(args.warmup):
        for s in shapes:
            s.call(0)
    torch.cuda.synchronize()
    res = {}
    for s in shapes:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for k in range(args.steps):
            s.call(k)
        b.record()
        torch.cuda.synchronize()
        res[f"M{s.M}_N{s.N}_K{s.K}"] = {"kernel": s.kernel, "eager_us_per_call": 1000 * a.elapsed_time(b) / args.steps,
                                      "plan": s.plan.as_dict()}
    print(json.dumps({"mode": "eager", "steps": args.steps, "shapes": res}))


WS_KERNELS = (3, 9)  # the cluster-free split-K forms, which need a caller workspace


def candidate_plans(lib, M, N, K):
    """Every plan worth timing for one shape (the tuning space of the sweep)."""
    cands = []
    if M <= 16:
        # token groups: 0 = one CTA loops over groups of 8; t > 0 = ceil(M / t) CTAs per row slice
        groups = [0] + sorted({-(-M // g) for g in (2, 3, 4) if -(-M // g) < M and -(-M // g) <= 8})
        for t in groups:
            for R in (1, 2, 4):
                for threads in (128, 256):
                    cands.append(lib.make_plan("dotprod", threads=threads, rows_per_cta=R, tokens_per_cta=t))
                    if M <= 4:  # x straight from L2 instead of a staged copy
                        cands.append(lib.make_plan("dotprod", threads=threads, rows_per_cta=R, tokens_per_cta=t,
                                                   stages=1))
    if K % 8 == 0 and M <= 64:
        chunks = -(-K // 64)
        tokens = max(8, -(-M // 8) * 8)
        for rows in (16, 32, 48, 64, 96, 128, 192, 256):
            if rows > max(16, 2 * N):
                continue
            for split in (1, 2, 3, 4, 6, 8, 12, 16):
                if split > chunks:
                    continue
                tiles = -(-N // rows)
                if tiles * split < 16 or tiles * split > 4 * 152:
                    continue
                per = -(-chunks // split)
                p = lib.make_plan("splitk", threads=128, rows_per_cta=rows, tokens_per_cta=tokens,
                                  split_k=split, stages=1)
                # deepest ring that fits (the planner's rule), found by trying
                for st in (16, 14, 12, 10, 8, 7, 6, 5, 4, 3, 2, 1):
                    p.stages = min(st, per)
                    try:
                        lib.plan_check(M, N, K, p)
                        break
                    except Exception:
                        continue
                cands.append(p)
                if K % 64 == 0 and split <= -(-chunks // 2):  # two K chunks per stage: half the TMA loads
                    for st in (8, 6, 5, 4, 3, 2, 1):
                        q = lib.make_plan("splitk", threads=128, rows_per_cta=rows, tokens_per_cta=tokens,
                                          split_k=split, stages=min(st, -(-per // 2)), chunks_per_stage=2)
                        try:
                            lib.plan_check(M, N, K, q)
                        except Exception:
                            continue
                        cands.append(q)
                        if M > 8 and tiles * split > 152 and q.stages > 2:
                            cands.append(lib.make_plan("splitk", threads=128, rows_per_cta=rows,
                                                       tokens_per_cta=tokens, split_k=split, stages=2,
                                                       chunks_per_stage=2))
                        break
                if M > 8 and tiles * split > 152:  # more CTAs than SMs: shallower rings, two or three per SM
                    for st in (6, 4, 3, 2):
                        if st < p.stages:
                            q = lib.make_plan("splitk", threads=128, rows_per_cta=rows, tokens_per_cta=tokens,
                                              split_k=split, stages=st)
                            try:
                                lib.plan_check(M, N, K, q)
                                cands.append(q)
                            except Exception:
                                pass
    if K % 8 == 0 and M <= 64:
        chunks = -(-K // 64)
        tokens = max(8, -(-M // 8) * 8)
        for rows in (16, 32, 64, 128, 256):
            if rows > max(16, 2 * N):
                continue
            for split in (2, 4, 8, 12, 16, 24, 32, 48, 64):
                tiles = -(-N // rows)
                if split > chunks or tiles * split < 32 or tiles * split > 4 * 152:
                    continue
                per = -(-chunks // split)
                p = lib.make_plan("splitk_ws", threads=128, rows_per_cta=rows, tokens_per_cta=tokens,
                                  split_k=split, stages=1)
                for st in (16, 14, 12, 10, 8, 7, 6, 5, 4, 3, 2, 1):
                    p.stages = min(st, per)
                    try:
                        lib.plan_check(M, N, K, p)
                        break
                    except Exception:
                        continue
                cands.append(p)
    if K % 8 == 0 and M <= 4 and K <= 8192:
        for rg in (1, 2, 4):
            if rg == 4 and M > 3:
                continue
            for st in (4, 6, 8, 12, 16):
                p = lib.make_plan("stream", threads=288, rows_per_cta=rg, stages=st)
                try:
                    lib.plan_check(M, N, K, p)
                except Exception:
                    continue
                cands.append(p)
    if K % 8 == 0 and M <= 8 and M * K * 2 <= 200 * 1024:
        for t, w, c in ((512, 1, 2), (512, 2, 2), (512, 4, 2), (1024, 1, 1), (1024, 2, 1), (1024, 4, 1),
                        (256, 1, 4), (256, 2, 4), (128, 1, 8), (128, 2, 8), (128, 4, 8)):
            p = lib.make_plan("warprow", threads=t, rows_per_cta=w, stages=c)
            try:
                lib.plan_check(M, N, K, p)
            except Exception:
                continue
            cands.append(p)
    if K % 8 == 0 and M <= 16 and M * K * 2 <= 200 * 1024:
        for t, w, c in ((512, 1, 2), (512, 2, 2), (512, 4, 2), (512, 8, 2), (1024, 1, 1), (1024, 4, 1),
                        (1024, 8, 1), (1024, 16, 1), (256, 1, 4), (256, 2, 4), (256, 8, 4), (128, 2, 8), (128, 4, 8)):
            p = lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c)
            try:
                lib.plan_check(M, N, K, p)
            except Exception:
                continue
            cands.append(p)
    if K % 8 == 0 and M <= 16 and N > 1024:  # x fragments from L2 (any K)
        for t, w, c in ((512, 4, 1), (512, 8, 1), (512, 16, 1), (256, 4, 2), (256, 8, 2), (128, 4, 4)):
            for ng in (0, 2, 4):  # one, two or four 8-row groups per warp
                cands.append(lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c, split_k=1,
                                           tokens_per_cta=ng))
    if K % 8 == 0 and M <= 64 and (N >= 1024 or M > 4):  # the warp-MMA kernel's cluster form: K over S CTAs
        cfgs = (((1024, 8, 1), (1024, 4, 1), (1024, 16, 1), (512, 4, 2), (512, 8, 2), (256, 2, 4), (256, 4, 4),
                 (128, 2, 8), (128, 4, 8))
                if M <= 16 else ((512, 4, 1), (512, 8, 1), (512, 16, 1), (256, 2, 2), (256, 4, 2), (256, 8, 2)))
        for S in (2, 4, 8, 16):
            for t, w, c in cfgs:
                for gpc in ((0,) if N >= 1024 else (0, 2, 4)):  # router N: several row groups per cluster
                    if gpc > (t // 32) // w:
                        continue
                    p = lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c, split_k=S, tokens_per_cta=gpc)
                    try:
                        lib.plan_check(M, N, K, p)
                    except Exception:
                        continue
                    cands.append(p)
    if K % 8 == 0 and 16 < M <= 64:  # the router MMA split-K in 16-token groups
        for S, t, xr in itertools.product((1, 2, 4, 8), (128, 256), (1,)):
            p = lib.make_plan("dotmma", threads=t, rows_per_cta=8, split_k=S, stages=xr)
            try:
                lib.plan_check(M, N, K, p)
            except Exception:
                continue
            cands.append(p)
    if K % 8 == 0 and M <= 16 and N <= 1024:
        for S, t, xr in itertools.product((8, 16, 32), (128, 256), (0, 1)):
            p = lib.make_plan("dotmma_ws", threads=t, rows_per_cta=8, split_k=S, stages=xr)
            try:
                lib.plan_check(M, N, K, p)
            except Exception:
                continue
            cands.append(p)
        for S, t, xr in itertools.product((2, 4, 8, 16), (128, 256), (0, 1)):
            if True:
                p = lib.make_plan("dotmma", threads=t, rows_per_cta=8, split_k=S, stages=xr)
                try:
                    lib.plan_check(M, N, K, p)
                except Exception:
                    continue
                cands.append(p)
    if K % 8 == 0 and M > 64:
        for st in (6, 5, 4):
            for bn in (256, 192):  # W rows per pair tile
                cands.append(lib.make_plan("tile2", threads=192, rows_per_cta=bn, tokens_per_cta=256, stages=st))
    if K % 8 == 0 and M > 32:  # the plain tile: W-tile widths, ring depths, raster groups
        for bn in (128, 192, 224, 240, 256):
            most = tile_max_stages(bn)
            for st in (most, most - 1):
                for grp in (0, 1, 2, 4, 16):
                    cands.append(lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128, stages=st,
                                               split_k=grp))
            if K % 64 == 0 and M <= 1024:  # two K chunks per stage (bandwidth-bound sizes)
                for grp in (0, 16):
                    cands.append(lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128,
                                               stages=max(2, most // 2), split_k=grp, chunks_per_stage=2))
    if K % 8 == 0 and 16 < M <= 512:  # the swap-AB tile: W rows on the MMA M side, tokens on N
        for bn in (32, 64, 128, 192, 256):
            if bn > 2 * max(32, M) or 4 * bn < M:
                continue
            most = tile_max_stages(bn)
            for st in (most, max(2, most - 2)):
                for grp in (0, 1):
                    cands.append(lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=bn,
                                               stages=st, split_k=grp))
            if K % 64 == 0:  # two K chunks per stage
                for st in sorted({most // 2, max(2, most // 2 - 1)}, reverse=True):
                    if st >= 2:
                        cands.append(lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=bn,
                                                   stages=st, split_k=0, chunks_per_stage=2))
    return cands


def tile_max_stages(bn):
    """Ring stages of the tile kernels that fit 227 KB of shared memory (at most 8)."""
    return min(8, (232448 - 1024 - 256) // (128 * 128 + bn * 128))


def sweep(args, points):
    """Time every candidate plan of every shape (L2-cold graphs) and write the dispatch table."""
    import moe_router_gemm_gb300 as lib
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)
    results = []
    out_dir = args.out_dir
    os.makedirs(out_dir, exist_ok=True)
    for pt in points:
        base = Shape(pt, device, lib)
        R = min(base.R, 64)  # 64 rotated copies keep every call L2-cold for these sizes
        rows = []
        cands = candidate_plans(lib, pt["M"], pt["N"], pt["K"])
        if args.sweep_kernels:  # a partial sweep over some kernels only
            keep = set(args.sweep_kernels.split(","))
            cands = [p for p in cands if lib.KERNEL_NAMES[p.kernel] in keep]
        need = max([lib.workspace_size(pt["M"], pt["N"], pt["K"], p) for p in cands] + [256])
        base.ws = lib.new_workspace(need, device)
        for p in cands:
            base.plan = p
            try:
                with torch.cuda.stream(stream):
                    for i in range(2):
                        base.call(i)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(R):
                            base.call(i)
                    g.replay()
                    torch.cuda.synchronize()
                    best = 1e9
                    for _ in range(3):
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        g.replay()
                        b.record(stream)
                        torch.cuda.synchronize()
                        best = min(best, 1000.0 * a.elapsed_time(b) / R)
                rows.append((best, p.as_dict()))
            except Exception as e:  # an unusable candidate is skipped, not fatal
                rows.append((float("inf"), dict(p.as_dict(), error=str(e)[:80])))
        rows.sort(key=lambda r: r[0])
        if not rows:  # a partial sweep with no candidate for this shape
            continue
        best_plain = next((r for r in rows if r[1].get("kernel") not in WS_KERNELS), rows[0])
        default = lib.plan(pt["M"], pt["N"], pt["K"]).as_dict()
        results.append({"M": pt["M"], "N": pt["N"], "K": pt["K"], "best_us": rows[0][0], "best": rows[0][1],
                        "best_plain_us": best_plain[0], "best_plain": best_plain[1],
                        "default": default, "top": [(round(t, 3), d) for t, d in rows[:5]]})
        print(json.dumps({"shape": [pt["M"], pt["N"], pt["K"]], "best_us": round(rows[0][0], 3),
                          "best": rows[0][1]}), flush=True)
        del base
        torch.cuda.empty_cache()
    with open(os.path.join(out_dir, "sweep_results.json"), "w") as f:
        json.dump(results, f, indent=1)
    lines = ["// Measured GB300 dispatch entries (python bench.py --sweep): fastest plan per shape, L2-cold.",
             "// {K, N, M, kernel, threads, rows_per_cta, tokens_per_cta, split_k, stages[, chunks_per_stage]},"]
    for r in sorted(results, key=lambda r: (r["K"], r["N"], r["M"])):
        entries = [(r["best"], r["best_us"])]
        if r["best"].get("kernel") in WS_KERNELS:  # needs a workspace: follow it with the best plan that needs none
            entries.append((r["best_plain"], r["best_plain_us"]))
        for b, us in entries:
            kc = f", {b['chunks_per_stage']}" if b.get("chunks_per_stage", 0) > 1 else ""
            lines.append(f"{{{r['K']}, {r['N']}, {r['M']}, {b['kernel']}, {b['threads']}, {b['rows_per_cta']}, "
                         f"{b['tokens_per_cta']}, {b['split_k']}, {b['stages']}{kc}}},  // {us:.3f} us")
    with open(os.path.join(out_dir, "dispatch_table.inc"), "w") as f:
        f.write("\n".join(lines) + "\n")


def e2e_arm(args, shapes, lib, device, stream):
    host = []
    for s in shapes:
        x, W, b = s.host
        host.append((x.pin_memory(), W.pin_memory(), b.pin_memory() if b is not None else None,
                     torch.empty(s.M, s.N, dtype=torch.bfloat16).pin_memory()))
    # one device staging buffer per shape: bf16_linear_host copies x, W (and bias) into it, runs the
    # planned kernel and copies out back, all on the stream (one C-ABI call per shape and step)
    staging = [lib.new_host_staging(s.M, s.N, s.K, s.b is not None, device=device) for s in shapes]
    h2d = sum(h[0].numel() * 2 + h[1].numel() * 2 + (h[2].numel() * 2 if h[2] is not None else 0) for h in host)
    d2h = sum(h[3].numel() * 2 for h in host)

    def one_step():
        for (hx, hW, hb, ho), st in zip(host, staging):
            lib.bf16_linear_host(hx, hW, hb, ho, staging=st, stream=stream)

    steps = max(1, min(args.steps, 5))
    with torch.cuda.stream(stream):
        for _ in range(2):
            one_step()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            one_step()
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"us_per_call": 1000.0 * ms / len(shapes), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def fp8_arm(args, points):
    """Per-tensor FP8 linear (bf16_linear_fp8) on the same shapes, L2-cold, beside the bf16 call.

    Weights are e4m3 codes (quantised once, on the device, with the library's own
    static quantisation) rotated over copies totalling >= 256 MB; one CUDA graph of
    R back-to-back calls per shape; algorithmic bytes NK + MK + 2MN (+2N bias)."""
    import moe_router_gemm_gb300 as lib
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()
    res = {}
    for pt in points:
        M, N, K, bias = pt["M"], pt["N"], pt["K"], pt["bias"]
        if K % 16:
            continue
        x, W, b = wl.make_inputs(M, N, K, pt["seed"], bias)
        sx = torch.tensor([float(x.float().abs().max()) / 448.0], dtype=torch.float32, device=device)
        sw = torch.tensor([float(W.float().abs().max()) / 448.0], dtype=torch.float32, device=device)
        xq = lib.quant_fp8(x.to(device), sx)
        w0 = lib.quant_fp8(W.to(device), sw)
        R = max(2, -(-L2_COLD_BYTES // (N * K)))
        Ws = [w0] + [w0.clone() for _ in range(R - 1)]
        bd = b.to(device) if b is not None else None
        out = torch.empty(M, N, dtype=torch.bfloat16, device=device)
        def timed(plan):
            with torch.cuda.stream(stream):
                for i in range(2):
                    lib.bf16_linear_fp8(xq, Ws[i % R], sx, sw, bd, out=out, stream=stream, plan_=plan)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(R):
                        lib.bf16_linear_fp8(xq, Ws[i], sx, sw, bd, out=out, stream=stream, plan_=plan)
                g.replay()
                torch.cuda.synchronize()
                ms = []
                for _ in range(max(3, args.steps)):
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    g.replay()
                    e.record(stream)
                    torch.cuda.synchronize()
                    ms.append(a.elapsed_time(e))
            return 1000.0 * statistics.median(ms) / R

        us = timed(None)
        nbytes = N * K + M * K + 2 * M * N + (2 * N if bias else 0)
        key = f"M{M}_N{N}_K{K}"
        res[key] = {"us": round(us, 3), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                    "pct_hbm_roofline": round(100.0 * nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 1),
                    "split_k": lib.fp8_split(M, N, K, torch.cuda.get_device_properties(device).multi_processor_count)}
        if args.sweep_fp8:  # every (split, threads) the explicit-plan entry accepts
            tried = []
            for S, t in itertools.product((1, 2, 4, 8, 16), (128, 256)):
                if S > (K // 16 + 3) // 4:
                    continue
                tried.append((round(timed(lib.make_plan("dotmma", threads=t, rows_per_cta=8, split_k=S)), 3),
                              "split", S, t))
            if M <= 16 and M * K <= 200 * 1024:
                for t, w, c in ((1024, 8, 1), (1024, 16, 1), (512, 4, 2), (512, 8, 2), (256, 8, 4), (256, 2, 4)):
                    if c * (M * K + (16384 if w > 1 else 512) + 1024) > 232448:
                        continue
                    p = lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c)
                    tried.append((round(timed(p), 3), "warpmma", w, t, c))
            res[key]["sweep"] = sorted(tried)[:4]
        del Ws
        torch.cuda.empty_cache()
    mean = statistics.mean(v["us"] for v in res.values()) if res else None
    print(json.dumps({"mode": "fp8", "metric": "per-tensor FP8 linear us per call (L2-cold)",
                      "mean_us": None if mean is None else round(mean, 4), "unit": "us/call",
                      "workload": workload_desc(args.workload), "shapes": res}))


def mxfp8_shape(lib, device, stream, pt, steps, peaks, plan=None):
    """One shape of the MXFP8 linear (bf16_linear_mxfp8), L2-cold: x and W quantised once on the device
    with bf16_quant_mxfp8, the weight codes and scales rotated over copies totalling >= 256 MB, one CUDA
    graph of R back-to-back calls; algorithmic bytes NK + N(K/32) + MK + M(K/32) + 2MN (+2N bias), flops
    2MNK.  Shapes above the e4m3 ridge (twice the measured bf16 burst peak, the nominal ratio, over the
    HBM copy peak) are reported against that tensor peak, the others against HBM.  Returns
    (record, time_fn) where time_fn(plan) re-times the shape with another plan."""
    M, N, K, bias = pt["M"], pt["N"], pt["K"], pt["bias"]
    fp8_tflops = 2.0 * peaks["bf16_tflops"]
    x, W, b = wl.make_inputs(M, N, K, pt["seed"], bias)
    xq, xs = lib.quant_mxfp8(x.to(device))
    wq0, ws0 = lib.quant_mxfp8(W.to(device))
    R = max(2, -(-L2_COLD_BYTES // (N * K)))
    Wq = [wq0] + [wq0.clone() for _ in range(R - 1)]
    Ws = [ws0] + [ws0.clone() for _ in range(R - 1)]
    bd = b.to(device) if b is not None else None
    out = torch.empty(M, N, dtype=torch.bfloat16, device=device)

    def time_us(pl=None):
        with torch.cuda.stream(stream):
            for i in range(2):
                lib.bf16_linear_mxfp8(xq, xs, Wq[i % R], Ws[i % R], bd, out=out, stream=stream, plan_=pl)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(R):
                    lib.bf16_linear_mxfp8(xq, xs, Wq[i], Ws[i], bd, out=out, stream=stream, plan_=pl)
            g.replay()
            torch.cuda.synchronize()
            ms = []
            for _ in range(max(3, steps)):
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                e.record(stream)
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(e))
        del g
        return 1000.0 * statistics.median(ms) / R

    us = time_us(plan)
    nbytes = N * K + N * (K // 32) + M * K + M * (K // 32) + 2 * M * N + (2 * N if bias else 0)
    flops = 2.0 * M * N * K
    tensor = flops / nbytes > fp8_tflops * 1e12 / (peaks["hbm_gbs"] * 1e9)
    rec = {"M": M, "N": N, "K": K, "bias": bias, "us": round(us, 3), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
           "TFLOPs": round(flops / (us * 1e-6) / 1e12, 1), "bound": "tensor" if tensor else "hbm",
           "frac": round(flops / (us * 1e-6) / 1e12 / fp8_tflops if tensor
                         else nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    return rec, time_us


def mxfp8_record(lib, device, stream, peaks, steps):
    """The MXFP8 linear on the prefill workload's shapes (its tile form), for the default bench line."""
    rows, tot_flops, tot_us = [], 0.0, 0.0
    for pt in workload_points("prefill"):
        rec, time_fn = mxfp8_shape(lib, device, stream, pt, steps, peaks)
        del time_fn  # frees the shape's weight copies
        rows.append(rec)
        tot_flops += 2.0 * rec["M"] * rec["N"] * rec["K"]
        tot_us += rec["us"]
        torch.cuda.empty_cache()
    tf = tot_flops / (tot_us * 1e-6) / 1e12
    return {"workload": workload_desc("prefill") + "; MXFP8 operands (bf16_quant_mxfp8 of the same inputs)",
            "unit": "us/call", "shapes": rows, "tensor_TFLOPs": round(tf, 1),
            "e4m3_peak_TFLOPs": round(2.0 * peaks["bf16_tflops"], 1),
            "tensor_frac": round(tf / (2.0 * peaks["bf16_tflops"]), 4),
            "peak_note": "twice the measured bf16 burst peak (the nominal e4m3:bf16 ratio)"}


def mxfp8_arm(args, points):
    """MXFP8 linear (bf16_linear_mxfp8) on the workload's shapes, L2-cold (mxfp8_shape).  With
    --sweep-fp8 the tile form's tactics (rows per tile, ring depth, raster group) are timed too and the
    best is reported."""
    import moe_router_gemm_gb300 as lib
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()
    fp8_tflops = 2.0 * peaks["bf16_tflops"]
    res = {}
    for pt in points:
        M, N, K, bias = pt["M"], pt["N"], pt["K"], pt["bias"]
        if K % 32:
            continue
        rec, time_us = mxfp8_shape(lib, device, stream, pt, args.steps, peaks)
        if args.sweep_fp8 and M > 16 and K % 128 == 0:
            tried = []
            for bq, most in ((128, 6), (256, 4)):
                for st in (most, most - 1):
                    for grp in (0, 1, 4, 16):
                        p = lib.make_plan("tile", threads=320, rows_per_cta=bq, stages=st, split_k=grp)
                        tried.append((time_us(p), f"tile bq={bq} stages={st} group={grp}"))
            tried.sort()
            rec["best_tile_us"], rec["best_tile"] = round(tried[0][0], 3), tried[0][1]
            rec["tile_top5"] = [[round(u, 3), d] for u, d in tried[:5]]
        res[f"M{M}_N{N}_K{K}" + ("_bias" if bias else "")] = rec
        del time_us
        torch.cuda.empty_cache()
    mean = statistics.mean(v["us"] for v in res.values()) if res else None
    print(json.dumps({"mode": "mxfp8", "metric": "MXFP8 linear us per call (L2-cold)",
                      "mean_us": None if mean is None else round(mean, 4), "unit": "us/call",
                      "peaks": {"hbm_gbs": peaks["hbm_gbs"], "e4m3_tflops": fp8_tflops,
                                "e4m3_note": "twice the measured bf16 burst (nominal e4m3:bf16 ratio)"},
                      "workload": workload_desc(args.workload), "shapes": res}))


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="router", choices=["router", "smallest", "decode", "mlp", "prefill", "all"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-fp8", action="store_true",
                    help="with --fp8: also time every (split, threads); with --mxfp8: the tile form's tactics")
    ap.add_argument("--fp8", action="store_true",
                    help="time the per-tensor FP8 linear (bf16_linear_fp8) on the workload's shapes instead")
    ap.add_argument("--mxfp8", action="store_true",
                    help="time the MXFP8 linear (bf16_linear_mxfp8) on the workload's shapes instead")
    ap.add_argument("--pdl", action="store_true",
                    help="launch with programmatic dependent launch (BF16L_FLAG_PDL): back-to-back calls overlap")
    ap.add_argument("--no-pdl-variant", action="store_true",
                    help="skip the extra passes that re-time every shape with programmatic dependent launch "
                         "and L2-warm")
    ap.add_argument("--plan", default=None,
                    help="force one plan on every shape: kernel,threads,rows_per_cta,tokens_per_cta,split_k,stages "
                         "(kernel by name, e.g. tile2,192,256,256,0,6); for profiling one kernel")
    ap.add_argument("--only", action="append", default=[],
                    help="restrict to shapes M,N,K[,bias] (repeatable); for profiling")
    ap.add_argument("--sweep-kernels", default="",
                    help="with --sweep: time only the candidates of these kernels (comma-separated names)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every candidate plan of the workload's shapes and write dispatch_table.inc "
                         "and sweep_results.json into --out-dir")
    ap.add_argument("--out-dir", default=".", help="with --sweep: where the sweep writes its files")
    ap.add_argument("--no-workloads", action="store_true",
                    help="router sweep only: skip the per-workload records (smallest, decode, MLP, prefill) "
                         "and the measured floors")
    ap.add_argument("--sub-replays", type=int, default=5,
                    help="graph replays per shape for the per-workload records")
    ap.add_argument("--eager", action="store_true",
                    help="profiling mode: each step calls every shape once per rotation copy, no graphs, "
                         "no e2e/cpu legs; prints per-shape timings only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3  # at least three warm-up steps

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    points = workload_points(args.workload)
    if args.only:
        points = []
        for spec in args.only:
            f = [int(v) for v in spec.split(",")]
            M, N, K = f[:3]
            points.append(dict(name=f"only_M{M}_N{N}_K{K}", M=M, N=N, K=K, bias=bool(f[3]) if len(f) > 3 else False,
                               seed=7 + M + N + K))
    peaks = load_peaks()
    large = args.workload == "prefill"
    metric = ("bf16 GEMM TFLOP/s (prefill, tile path)" if large else
              "M\u226416 bf16 GEMM \u00b5s & % HBM roofline (L2-cold); large-M TFLOP/s % bf16 peak")
    unit = "TFLOP/s" if large else "us/call"
    config = {"workload": workload_desc(args.workload), "shapes": len(points),
              "value": ("TFLOP/s over the prefill shapes" if large else
                        "mean us per call over the workload's shapes, L2-cold (the router sweep by default; "
                        "the other workloads of the metric, with their roofline fractions, under 'workloads')"),
              "l2": "cold: weights rotated over copies totalling >=256 MB per shape; x L2-hot",
              "timing": "CUDA graph of R back-to-back calls per shape, CUDA events on the launching stream",
              "launch": ("early weights (BF16L_FLAG_PDL)" if args.pdl else
                         "the library's default: programmatic dependent launch, every read after the "
                         "grid-dependency wait"),
              "pdl": bool(args.pdl)}

    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        smp = OracleSample(points, budget_s=args.cpu_budget / max(1, args.steps))
        smp.run(args.warmup)  # untimed warm-up passes (at least three)
        wall = smp.run(args.steps)
        value = smp.value(wall, args.steps, large)
        line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wall / args.steps,
                "higher_is_better": large, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": unit, "cores": smp.threads, "cpu_model": cpu_model(), "kind": "oracle",
                                 "sample": smp.desc},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
        torch.cuda.set_device(local_rank)
    else:
        torch.cuda.set_device(0)

    if args.eager:
        eager_profile(args, points)
        return
    if args.sweep:
        sweep(args, points)
        return
    if args.fp8:
        fp8_arm(args, points)
        return
    if args.mxfp8:
        mxfp8_arm(args, points)
        return
    r = gpu_arm(args, points, rank, world)
    shapes, per_us = r["shapes"], r["per_shape_us"]
    total_ms = r["total_ms"]
    if world > 1:
        total_ms = max_over_ranks(total_ms, device="cuda")

    # dominant kernel: the largest share of measured time
    share = {}
    for s, us in zip(shapes, per_us):
        share.setdefault(s.kernel, [0.0, 0, 0.0, []])
        share[s.kernel][0] += us
        share[s.kernel][1] += 1
        share[s.kernel][2] += algo_flops(s.M, s.N, s.K, s.bias) if large else algo_bytes(s.M, s.N, s.K, s.bias)
        share[s.kernel][3].append(s)
    dom = max(share, key=lambda k: share[k][0])
    dom_us, dom_n, dom_work, dom_shapes = share[dom]
    if large:
        achieved = dom_work / (dom_us * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        bound, runit = "tensor", "TFLOP/s"
    else:
        achieved = dom_work / (dom_us * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        bound, runit = "hbm", "GB/s"
    # traffic: ncu DRAM bytes per launch, averaged over the dominant kernel's shapes (as `achieved` is)
    traffic = ncu_traffic(dom, [(s.M, s.N, s.K) for s in dom_shapes])
    algo_per_launch = dom_work / dom_n

    calls_per_step = sum(s.R for s in shapes)
    if large:
        flops_step = sum(algo_flops(s.M, s.N, s.K, s.bias) * s.R for s in shapes)
        value = flops_step * args.steps * world / (total_ms * 1e-3) / 1e12
    else:
        value = replica_value(statistics.mean(per_us), world)
    ms_per_step = total_ms / args.steps

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        smp = OracleSample(points, budget_s=args.cpu_budget)
        wall = smp.run(1)
        cpu = {"value": smp.value(wall, 1, large), "unit": unit, "cores": smp.threads, "cpu_model": cpu_model(), "kind": "oracle",
               "sample": smp.desc}

    e2e = r["e2e"]
    if large:
        e2e_value = sum(algo_flops(s.M, s.N, s.K, s.bias) for s in shapes) / (e2e["us_per_call"] * len(shapes) * 1e-6) / 1e12
    else:
        e2e_value = e2e["us_per_call"]

    per_shape = {}
    for s, us in zip(shapes, per_us):
        key = f"K{s.K}_N{s.N}"
        per_shape.setdefault(key, []).append(round(us, 3))
    if r["floor"] is not None:
        rf = r["floor"]["read_weight"]
        floors = [rf[f"K{s.K}_N{s.N}"]["us"] for s in shapes]
        r["floor"]["router_mean_read_floor_us"] = round(statistics.mean(floors), 3)
        r["floor"]["router_mean_frac_of_floor"] = round(statistics.mean(f / u for f, u in zip(floors, per_us)), 4)
        r["floor"]["read_floor_frac_hbm"] = round(statistics.mean(
            algo_bytes(s.M, s.N, s.K, s.bias) / (f * 1e-6) / 1e9 / peaks["hbm_gbs"] for s, f in zip(shapes, floors)), 4)
    line = {
        "metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": large,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "roofline": {"bound": bound, "kernel": dom, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_per_launch": round(algo_per_launch) if not large else None,
                     "averaged_over": f"{dom_n} shapes run by the {dom} kernel",
                     "peak_source": peaks["source"]},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 4), "unit": unit, "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "kernel_share": {k: round(v[0] / sum(x[0] for x in share.values()), 4) for k, v in share.items()},
        "serial_variant": None if r["serial_us"] is None else {
            "note": "same shapes and rotation, launched with BF16L_FLAG_SERIAL (no programmatic dependent "
                    "launch: each call starts only after the previous one completed); timed after the main region",
            "value": round(statistics.mean(r["serial_us"]), 4) if not large else None,
            "unit": unit,
            "per_shape_us": {k: [round(u, 3) for s_, u in zip(shapes, r["serial_us"]) if f"K{s_.K}_N{s_.N}" == k]
                             for k in per_shape}},
        "pdl_variant": None if r["pdl_us"] is None else {
            "note": "same shapes and rotation, launched with BF16L_FLAG_PDL (weights fetched before the "
                    "grid-dependency wait, so back-to-back calls overlap); timed after the main region",
            "value": round(statistics.mean(r["pdl_us"]), 4) if not large else None,
            "unit": unit,
            "per_shape_us": {k: [round(u, 3) for s_, u in zip(shapes, r["pdl_us"]) if f"K{s_.K}_N{s_.N}" == k]
                             for k in per_shape}},
        "l2_warm": None if r["warm_us"] is None else {
            "note": "same calls, every one on the same weight copy (L2-resident after the first where it fits "
                    "in L2); effective GB/s = algorithmic bytes / time, against the HBM copy peak",
            "value": round(statistics.mean(r["warm_us"]), 4) if not large else round(
                sum(algo_flops(s.M, s.N, s.K, s.bias) for s in shapes)
                / (sum(r["warm_us"]) * 1e-6) / 1e12, 2),
            "unit": unit,
            "per_shape_us": {k: [round(u, 3) for s_, u in zip(shapes, r["warm_us"]) if f"K{s_.K}_N{s_.N}" == k]
                             for k in per_shape},
            "pct_hbm_roofline_per_shape": None if large else {
                k: [round(100.0 * algo_bytes(s.M, s.N, s.K, s.bias) / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 1)
                    for s, us in zip(shapes, r["warm_us"]) if f"K{s.K}_N{s.N}" == k] for k in per_shape}},
        "floor": r["floor"],
        "workloads": r["records"],
        "per_shape_us": per_shape,
        "pct_hbm_roofline_per_shape": None if large else {
            k: [round(100.0 * algo_bytes(s.M, s.N, s.K, s.bias) / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 1)
                for s, us in zip(shapes, per_us) if f"K{s.K}_N{s.N}" == k] for k in per_shape},
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
