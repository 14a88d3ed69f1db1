#!/usr/bin/env python
"""Throughput of the 2D Gaussian-splatting rasterizer on one B300 (or N
independent replicas, one per GPU) -> one JSON line on stdout.

A step is one pass of the whole path over one synthetic image:
project -> bin_and_sort -> render_fwd -> loss_l2 -> render_bwd
(forward-only workloads stop after render_fwd).  The default workload is
768x512 RGB with 50,000 Gaussians, accumulated sum, L2 loss.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference]

`value` is steps per second over the timed region with inputs resident in
HBM (CUDA events, one CUDA graph replay per step, the L2 cache flushed
before every step).  `e2e` repeats the step through the same C calls with
the inputs copied from pinned host memory and the loss and gradients copied
back inside the timed region.  `--impl reference` times the CPU oracle on
this machine's host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd iters/s & render FPS @768×512, 50K Gaussians; % of FP32/SFU roofline"
COUNTS = os.path.join(ROOT, "tests", "golden", "workload_counts.json")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
CSRC = os.path.join(ROOT, "raster_gaussian_02_b300", "csrc")

# Algorithmic work per touching (pixel, Gaussian) pair, the unit of work:
# FP32 flops (FMA = 2) of the per-pixel formulation of each pass, and SFU
# exp2 evaluations.  Sum forward: dx, dy (2), q (7), exponent scale (1),
# 3 colour FMAs (6) = 16.  Sum backward, every pixel forming its own share
# of each gradient: the recomputed weight (10), 3 colour-gradient FMAs (6),
# g.rgb (5), dL/dq (2), the mean's two terms (11) and the inverse
# covariance's three (10): 44 by this count, about 40 as the unit is quoted,
# and 40 is taken.  Composite adds about 6 (forward) and 10 (backward).
FLOPS = {"fwd_sum": 16, "bwd_sum": 40, "fwd_comp": 22, "bwd_comp": 50, "fused_comp": 72}
EX2 = {"fwd_sum": 1, "bwd_sum": 1, "fwd_comp": 1, "bwd_comp": 1, "fused_comp": 2}
# What the kernels execute per touching pair after factoring (for
# comparison): the sum backward takes the inverse covariance out of its
# pixel sums and the row offset dy out of each row's, 23 flops per pixel
# plus about 3 per pixel of row work.
FLOPS_EXECUTED = {"fwd_sum": 16, "bwd_sum": 26, "fwd_comp": 22, "bwd_comp": 38, "fused_comp": 60}
# Per-SM rates per clock: 128 FP32 FMA lanes; 32 ex2 results from the SFU
# (the probe in libgs2d_probe.so measures 28-30 per SM per clock on 148 SMs
# at 2032 MHz, more than 16 could give).
SM_FP32_LANES, SM_SFU_LANES = 128, 32
# The workloads measured after the headline one in the same run.
EXTRA_CONFIGS = ["heavy_2048x1360_300k", "composite_768x512_50k", "render_4096x4096_2m",
                 "sweep_768x512_10k", "sweep_768x512_50k", "sweep_768x512_200k", "sweep_768x512_1m"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gs2d", choices=["gs2d", "reference"])
    ap.add_argument("--workload", default="image_768x512_50k")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of a CUDA graph")
    ap.add_argument("--path", choices=("fused", "separate"), default="fused",
                    help="training step: the fused fwd+L2+bwd call, or the three separate calls")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (heavy, composite, 4096x4096, N sweep)")
    ap.add_argument("--config-steps", type=int, default=30, help="timed steps per other workload")
    return ap.parse_args()


def make_workload(name: str, seed_offset: int = 0):
    from raster_gaussian_02_b300 import synth
    if name.startswith("sweep_768x512_"):
        n = {"10k": 10_000, "50k": 50_000, "200k": 200_000, "1m": 1_000_000}[name.split("_")[-1]]
        return synth.render_uniform(768, 512, n, seed=5000 + n + seed_offset)
    fn = synth.WORKLOADS[name]
    import inspect
    seed = inspect.signature(fn).parameters["seed"].default
    return fn(seed=seed + seed_offset)


def describe(wl) -> str:
    mode = "alpha-composited" if wl.mode == 1 else "accumulated-sum"
    what = "fwd+L2+bwd" if wl.target is not None else "forward only"
    return (f"{wl.width}x{wl.height} RGB, {wl.n:,} Gaussians, {mode} {what}, tile 16, "
            f"{wl.cutoff_sigma:g}-sigma cutoff")


def load_json(path):
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi every 50 ms
    while the timed region runs (started before it, stopped after it)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def _reader(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[0].isdigit():
                self.rows.append((time.perf_counter(), parts))

    def __enter__(self):
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.t = threading.Thread(target=self._reader, daemon=True)
        self.t.start()
        t0 = time.perf_counter()
        while not self.rows and time.perf_counter() - t0 < 5.0:  # first sample before timing
            time.sleep(0.01)
        self.start = time.perf_counter()
        return self

    def __exit__(self, *a):
        self.stop = time.perf_counter()
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        inside = [p for t, p in self.rows if self.start - 0.06 <= t <= self.stop + 0.06] if self.rows else []
        rows = inside or [p for _, p in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(p[1]) for p in rows) if v is not None]
        mx = [v for v in (num(p[2]) for p in rows) if v is not None]
        reasons = set()
        for p in rows:
            for name, flag in zip(self.NAMES, p[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------- aggregation ---

def aggregate_replicas(local_ms: float, steps: int, world: int, device=None):
    """Whole-job throughput of `world` independent replicas: every rank ran
    `steps` steps in `local_ms`; the job time is the slowest rank's.  Returns
    (steps per second over all ranks, job time in ms).  Needs an initialised
    process group when world > 1 (gloo on CPU tensors, nccl on `device`)."""
    job_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([job_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        job_ms = float(t.item())
    return world * steps / (job_ms / 1e3), job_ms


# ------------------------------------------------------------ reference ---

def oracle_step(wl, omp: bool = False):
    import oracle
    cfg = oracle.Config(wl.width, wl.height, wl.mode, wl.cutoff_sigma, wl.t_min, param=wl.param)
    if wl.target is None:
        s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)
        s.render(omp=omp)
        return
    oracle.step(cfg, wl.xy, wl.chol, wl.rgb, wl.target, wl.depth, wl.opacity, wl.background, omp=omp)


def probe_peaks(dev, sms: int):
    """Measured FP32 FMA and SFU ex2 throughput (libgs2d_probe.so), a
    cross-check of the derived peaks: median of 10 timed launches of each
    probe after 3 warm-up launches, 8 blocks of 256 threads per SM."""
    import ctypes as C

    import torch

    from raster_gaussian_02_b300 import build as lib_build
    L = C.CDLL(lib_build.build_probe())
    L.gs2d_probe_fp32_fma.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_float, C.c_float, C.c_void_p]
    L.gs2d_probe_ex2.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]
    blocks = 8 * sms
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev)

    def rate(launch, work):
        for _ in range(3):
            if launch() != 0:
                raise RuntimeError("probe launch failed")
        ms = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            launch()
            b.record(s)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return work / (statistics.median(ms) * 1e-3)

    fma_iters, ex2_iters = 4096, 512
    fma = rate(lambda: L.gs2d_probe_fp32_fma(out.data_ptr(), blocks, fma_iters, 0.999, 1e-3, s.cuda_stream),
               2.0 * blocks * 256 * 8 * fma_iters)
    ex2 = rate(lambda: L.gs2d_probe_ex2(out.data_ptr(), blocks, ex2_iters, s.cuda_stream),
               1.0 * blocks * 256 * 8 * ex2_iters)
    return {"fp32_tflops": fma / 1e12, "ex2_per_s": ex2,
            "method": f"{blocks} blocks x 256 threads x 8 independent chains; "
                      f"{fma_iters} FMAs / {ex2_iters} ex2.approx per chain; median of 10"}


def cpu_baseline(wl, budget_s: float, min_steps: int = 2):
    """The CPU oracle timed on this machine's host cores: as it stands,
    single-threaded, full steps of the same workload for about budget_s
    seconds (at least min_steps); then the same steps through its OpenMP
    timing driver (the same per-pixel functions, tile rows over all host
    threads) for about a third of that."""
    import oracle
    unit = "iters/s" if wl.target is not None else "frames/s"

    def run(omp, budget, least):
        oracle_step(wl, omp)  # builds the library, warms caches
        t0 = time.perf_counter()
        k = 0
        while k < least or time.perf_counter() - t0 < budget:
            oracle_step(wl, omp)
            k += 1
        return k, time.perf_counter() - t0

    k, dt = run(False, budget_s, min_steps)
    threads = oracle.omp_threads(0)
    k2, dt2 = run(True, budget_s / 3, min_steps)
    single = {"value": k / dt, "unit": unit, "cores": 1,
              "sample": f"{k} full steps of the same workload, single-threaded C oracle, {dt:.1f} s"}
    omp = {"value": k2 / dt2, "unit": unit, "cores": threads, "nproc": os.cpu_count(),
           "sample": f"{k2} full steps of the same workload, the oracle's per-pixel functions over "
                     f"{threads} OpenMP threads (tile rows), {dt2:.1f} s"}
    return {"value": single["value"], "unit": unit, "cores": 1, "kind": "oracle",
            "sample": single["sample"], "single": single, "omp": omp}


def cpu_config(wl):
    """One full step of a workload through the oracle's OpenMP driver on all
    host threads (the larger workloads: one step is the sample)."""
    import oracle
    threads = oracle.omp_threads(0)
    t0 = time.perf_counter()
    oracle_step(wl, omp=True)
    dt = time.perf_counter() - t0
    return {"value": 1.0 / dt, "unit": "iters/s" if wl.target is not None else "frames/s",
            "cores": threads, "kind": "oracle",
            "sample": f"one full step, the oracle's per-pixel functions over {threads} OpenMP "
                      f"threads, {dt:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = make_workload(args.workload)
    oracle_step(wl)
    t1 = time.perf_counter()
    oracle_step(wl)
    per = time.perf_counter() - t1
    budget = 150.0
    warm = max(0, min(args.warmup, int(0.2 * budget / max(per, 1e-9))))
    steps = max(1, min(args.steps, int(budget / max(per, 1e-9))))
    for _ in range(warm):
        oracle_step(wl)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(wl)
    dt = time.perf_counter() - t0
    v = steps / dt
    unit = "iters/s" if wl.target is not None else "frames/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": 1e3 * dt / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "name": args.workload,
                   "note": f"--steps {args.steps} --warmup {args.warmup} requested; capped to "
                           f"about {budget:.0f} s of CPU time"},
        "cpu_baseline": {"value": v, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} full steps, single-threaded C oracle (fp64 values)"},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ gs2d ---

_COMMENTS = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is compiled from, comments removed: the
    .cu file that defines it and every shared header.  A stored traffic
    figure is used only while this matches, so editing one kernel voids only
    its own figures, and editing a comment voids none."""
    base = kernel.split("<", 1)[0]
    pat = re.compile(r"__global__[^;{]*?\b" + re.escape(base) + r"\s*\(", re.S)
    h = hashlib.sha256()
    found = False
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name)) as f:
            text = f.read()
        code = _COMMENTS.sub("", text)
        if name.endswith(".cuh"):
            h.update(name.encode() + code.encode())
        elif name.endswith(".cu") and pat.search(code):
            h.update(name.encode() + code.encode())
            found = True
    return h.hexdigest()[:16] if found else ""


def kernel_kind(name: str):
    """The raster work a kernel does (a key of FLOPS), or None."""
    for prefix, kind in (("k_render_bwd_sum", "bwd_sum"), ("k_render_fwd_sum", "fwd_sum"),
                         ("k_render_bwd_comp", "bwd_comp"), ("k_render_fwd_comp", "fwd_comp"),
                         ("k_fused_comp", "fused_comp")):
        if name.startswith(prefix):
            return kind
    return None


class Peaks:
    """FP32 and SFU peaks for the ALU roofline, derived from the SM count and
    the maximum SM clock."""

    def __init__(self, props, clocks):
        peaks = load_json(PEAKS) or {}
        self.sms = props.multi_processor_count
        self.sm_max = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2032.0)
        self.fp32 = self.sms * SM_FP32_LANES * 2 * self.sm_max * 1e6 / 1e12  # TFLOP/s
        self.sfu = self.sms * SM_SFU_LANES * self.sm_max * 1e6  # ex2 / s
        self.basis = (f"{self.sms} SMs x {SM_FP32_LANES} FP32 lanes x 2 x {self.sm_max:.0f} MHz; "
                      f"SFU {self.sms} x {SM_SFU_LANES} ex2/clock x {self.sm_max:.0f} MHz (max SM "
                      f"clock; at the sampled clock the fraction is frac x {self.sm_max:.0f}/median MHz)")


def roofline(peaks: Peaks, kernel: str, ms: float, touching_pairs, traffic=None, step_ms=None):
    """ALU roofline of one raster kernel: algorithmic FP32 work (touching
    pairs x FLOPS per pair) and SFU work (touching pairs x EX2 per pair) over
    the kernel's device time `ms`.  frac = max(FP32 fraction, SFU fraction)."""
    kind = kernel_kind(kernel)
    if kind is None or not touching_pairs or not ms:
        return None
    flops = FLOPS[kind]
    achieved = touching_pairs * flops / (ms * 1e-3) / 1e12
    fp32_frac = achieved / peaks.fp32
    sfu_frac = touching_pairs * EX2[kind] / (ms * 1e-3) / peaks.sfu
    out = {"bound": "alu", "achieved": achieved, "peak": peaks.fp32, "unit": "TFLOP/s",
           "frac": max(fp32_frac, sfu_frac), "fp32_frac": fp32_frac, "sfu_frac": sfu_frac,
           "traffic": traffic, "kernel": kernel, "ms": ms, "touching_pairs": touching_pairs,
           "flops_per_pair": flops, "ex2_per_pair": EX2[kind],
           "flops_per_pair_executed": FLOPS_EXECUTED[kind],
           "fp32_frac_executed": touching_pairs * FLOPS_EXECUTED[kind] / (ms * 1e-3) / 1e12 / peaks.fp32,
           "peak_basis": peaks.basis,
           "time_basis": "median device time of this kernel over traced CUDA-graph replays of the "
                         "step, each after an L2 flush (CUDA events recorded just before and just "
                         "after the kernel on its stream)"}
    if step_ms is not None:
        out["kernel_ms_le_step_ms"] = bool(ms <= step_ms)
    return out


class WorkloadRun:
    """One workload on one GPU: inputs resident in HBM, a Rasterizer with pair
    headroom, and the calls of a step, replayable as CUDA graphs."""

    def __init__(self, name, dev, stream, flush_buf, rank=0, path="fused", use_graph=True):
        import numpy as np
        import torch

        from raster_gaussian_02_b300 import gs2d

        self.name, self.dev, self.stream, self.flush_buf = name, dev, stream, flush_buf
        self.use_graph = use_graph
        self._graphs = []
        wl = self.wl = make_workload(name, seed_offset=rank)
        self.fwd_only = wl.target is None
        # The step's inputs live in one device buffer (each part 16-byte
        # aligned), so that the end-to-end leg moves them with one copy.
        parts = [wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background, wl.target]
        offs, total = [], 0
        for a in parts:
            offs.append(total)
            if a is not None:
                total += (a.size + 3) // 4 * 4
        self.host_pack = np.zeros(max(total, 4), np.float32)
        for a, o in zip(parts, offs):
            if a is not None:
                self.host_pack[o:o + a.size] = np.ascontiguousarray(a, np.float32).ravel()
        self.d_pack = torch.from_numpy(self.host_pack).to(dev)
        self._layout = [None if a is None else (o, a.size, a.shape) for a, o in zip(parts, offs)]
        self.use_buffer(self.d_pack)
        R = self.R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                                     device=dev, param=wl.param)
        R.project(self.xy, self.chol, self.rgb, self.depth, self.opac)
        self.P = R.bin_and_sort(sync=True)
        R._alloc_pairs(int(self.P * 1.25) + 4096)  # headroom, as a fitting loop would keep
        self.fused = path == "fused"

    def use_buffer(self, d_pack):
        """Points the step's inputs at views of a device buffer laid out like
        host_pack (calls() made afterwards read from it)."""
        views = [None if L is None else d_pack[L[0]:L[0] + L[1]].view(L[2]) for L in self._layout]
        self.xy, self.chol, self.rgb, self.depth, self.opac, self.bg, self.target = views

    def calls(self, kind):
        """The library calls of one step of `kind`, as (call name, callable):
        fused (the two fused calls), separate (the five calls), render
        (projection + binning, forward) or cached (forward only)."""
        R = self.R
        a = (self.xy, self.chol, self.rgb, self.depth, self.opac)
        pbs = ("project_bin_and_sort", lambda: R.project_bin_and_sort(*a, sync=False))
        fwd = ("render_fwd", lambda: R.render_fwd(self.bg))
        if kind == "cached":
            return [fwd]
        if kind == "render":
            return [pbs, fwd]
        if kind == "fused":
            return [pbs, ("render_fwd_bwd_l2", lambda: R.render_fwd_bwd_l2(self.target, self.bg))]
        out = [("project", lambda: R.project(*a)),
               ("bin_and_sort", lambda: R.bin_and_sort(sync=False)), fwd]
        if not self.fwd_only:
            out += [("loss_l2", lambda: R.loss_l2(self.target)), ("render_bwd", R.render_bwd)]
        return out

    def step_kind(self):
        if self.fwd_only:
            return "render"
        return "fused" if self.fused else "separate"

    def fn(self, kind):
        cs = self.calls(kind)

        def run():
            for _, f in cs:
                f()
        return run

    def graph(self, fn, force=False):
        """A replay callable of fn captured as one CUDA graph (fn itself when
        graphs are off, unless force)."""
        import torch
        if not self.use_graph and not force:
            return fn
        with torch.cuda.stream(self.stream):
            fn()
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        self._graphs.append(g)
        return g.replay

    def timed(self, fn, steps, warm, flush=True):
        """Per-step device time (ms), the L2 flushed before each step."""
        import torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        with torch.cuda.stream(self.stream):
            for _ in range(warm):
                fn()
            torch.cuda.synchronize()
            for a, b in ev:
                if flush:
                    self.flush_buf.fill_(1.0)
                a.record(self.stream)
                fn()
                b.record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def traced(self, kind, reps):
        """Device time of every kernel and of every call of one step, from a
        CUDA graph of the step whose calls each run under a kernel trace,
        replayed `reps` times, each after an L2 flush.  Returns (kernels,
        calls, launches): kernels = [(name, median ms)] in launch order,
        calls = {call: median ms from its first kernel's start to its last
        kernel's end}, launches = kernels launched per step."""
        import torch

        from raster_gaussian_02_b300 import gs2d
        cs = self.calls(kind)
        traces = [gs2d.KernelTrace(64, device=self.dev) for _ in cs]

        def run():
            for (_, f), tr in zip(cs, traces):
                with tr:
                    f()
        with torch.cuda.stream(self.stream):
            run()
            run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            run()
        per_kernel, per_call = None, {c: [] for c, _ in cs}
        with torch.cuda.stream(self.stream):
            for r in range(reps + 2):
                self.flush_buf.fill_(1.0)
                g.replay()
                torch.cuda.synchronize()
                if r < 2:
                    continue  # warm-up replays
                flat = [d for tr in traces for d in tr.durations()]
                if per_kernel is None:
                    per_kernel = [(n, []) for n, _ in flat]
                for (_, lst), (_, ms) in zip(per_kernel, flat):
                    lst.append(ms)
                for (c, _), tr in zip(cs, traces):
                    k = len(tr.names)
                    if k:
                        per_call[c].append(tr.events[0].elapsed_time(tr.events[2 * k - 1]))
        kernels = [(n, statistics.median(v)) for n, v in (per_kernel or [])]
        calls = {c: statistics.median(v) for c, v in per_call.items() if v}
        launches = sum(tr.launched for tr in traces)
        del g
        return kernels, calls, launches

    def call_ms(self, kind, repeats=10, reps=20):
        """Device time of each call of a `kind` step on its own: the call
        captured `repeats` times back to back in one CUDA graph, replayed
        `reps` times (each after an L2 flush); median replay time / repeats."""
        out = {}
        for name, f in self.calls(kind):
            def rep(f=f):
                for _ in range(repeats):
                    f()
            out[name] = statistics.median(self.timed(self.graph(rep, force=True), reps, 3)) / repeats
        self._graphs = []
        return out

    def release(self):
        """Frees this workload's device memory."""
        import torch
        self._graphs = []
        for k in ("R", "d_pack", "xy", "chol", "rgb", "depth", "opac", "bg", "target"):
            setattr(self, k, None)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def trace_floor(dev, stream, reps=50):
    """The kernel trace's floor: the traced interval (median over graph
    replays) of the smallest kernels the library launches, the L2 loss of a
    1x1 image (one block each).  Every traced kernel time includes about
    this much of launch and event overhead."""
    import torch

    from raster_gaussian_02_b300 import gs2d
    z = lambda *sh: torch.zeros(*sh, dtype=torch.float32, device=dev)
    img, tgt, loss, dimg = z(3, 1, 1), z(3, 1, 1), z(1), z(3, 1, 1)
    ws = torch.zeros(16384, dtype=torch.uint8, device=dev)
    tr = gs2d.KernelTrace(4, device=dev)

    def run():
        with tr:
            gs2d.check(gs2d.gs2d_loss_l2(1, 1, img, tgt, loss, dimg, ws, stream), "gs2d_loss_l2")
    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    per = {}
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        for n, ms in tr.durations():
            per.setdefault(n, []).append(ms)
    return min(statistics.median(v) for v in per.values())


def kernel_table(kernels, step_ms=None):
    """Per kernel name: launches per step, summed median ms, share of the
    traced kernels' total (and of the step)."""
    agg = {}
    for n, ms in kernels:
        a = agg.setdefault(n, {"launches": 0, "ms": 0.0})
        a["launches"] += 1
        a["ms"] += ms
    tot = sum(a["ms"] for a in agg.values()) or 1.0
    for a in agg.values():
        a["share"] = a["ms"] / tot
        if step_ms:
            a["share_of_step"] = a["ms"] / step_ms
    return dict(sorted(agg.items(), key=lambda kv: -kv[1]["ms"]))


def dominant_raster(kernels):
    """The raster kernel with the largest median time: (name, ms).  Event
    timestamps come in steps of about 1 us, so kernels within 2 % of the
    longest count as tied; of those, the one with the most algorithmic work
    per pair is taken."""
    rast = [(n, ms) for n, ms in kernels if kernel_kind(n)]
    if not rast:
        return None
    top = max(ms for _, ms in rast)
    tied = [(n, ms) for n, ms in rast if ms >= 0.98 * top]
    return max(tied, key=lambda x: (FLOPS[kernel_kind(x[0])], x[1]))


def first_of(kernels, kinds):
    for n, ms in kernels:
        if kernel_kind(n) in kinds:
            return n, ms
    return None


def stored_traffic(db, kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from an ncu capture,
    or None when none was taken or the kernel's sources changed since."""
    tr = db.get(f"{kernel}:{workload}")
    return tr["bytes"] if tr and tr.get("source_hash") == kernel_source_hash(kernel) else None


def measure_config(name, dev, stream, flush_buf, peaks, counts, steps, warm, reps, cpu=False):
    """Graph-replayed throughput and a kernel-time roofline of one workload."""
    t0 = time.perf_counter()
    w = WorkloadRun(name, dev, stream, flush_buf)
    kind = w.step_kind()
    step_ms = statistics.median(w.timed(w.graph(w.fn(kind)), steps, warm))
    kernels, calls, launches = w.traced(kind, reps)
    out = {"workload": describe(w.wl), "pairs": int(w.P),
           "unit": "frames/s" if w.fwd_only else "iters/s", "value": 1e3 / step_ms,
           "ms_per_step": step_ms, "steps": steps, "call_ms": calls,
           "kernels": kernel_table(kernels, step_ms), "gpu_launches_per_step": launches}
    render_ms = step_ms
    if not w.fwd_only:
        render_ms = statistics.median(w.timed(w.graph(w.fn("render")), steps, warm))
        out["render_fps"] = 1e3 / render_ms
    out["cached_render_fps"] = 1e3 / statistics.median(w.timed(w.graph(w.fn("cached")), steps, warm))
    tp = (counts.get(name) or {}).get("touching_pairs")
    traffic_db = load_json(TRAFFIC) or {}
    dom = dominant_raster(kernels)
    if dom:
        out["roofline"] = roofline(peaks, dom[0], dom[1], tp, stored_traffic(traffic_db, dom[0], name),
                                   step_ms=step_ms)
    if not w.fwd_only:
        rk, _, _ = w.traced("render", reps)
        f = first_of(rk, ("fwd_sum", "fwd_comp"))
        if f:
            out["roofline_fwd"] = roofline(peaks, f[0], f[1], tp, stored_traffic(traffic_db, f[0], name),
                                           step_ms=render_ms)
    w.release()
    if cpu:
        out["cpu_baseline"] = cpu_config(w.wl)
    out["wall_s"] = time.perf_counter() - t0
    return out


def run_gs2d(args):
    import torch
    import torch.distributed as dist

    from raster_gaussian_02_b300 import build as lib_build
    from raster_gaussian_02_b300 import gs2d

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        lib_build.build()
    if world > 1:
        dist.barrier()
    gs2d.lib()

    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    w = WorkloadRun(args.workload, dev, stream, flush_buf, rank=rank, path=args.path,
                    use_graph=not args.no_graph)
    R, fwd_only, kind = w.R, w.fwd_only, w.step_kind()
    run_step = w.graph(w.fn(kind))

    # ---- headline: K steps, max over ranks
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with sampler:
        step_ms = w.timed(run_step, args.steps, args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    st, _, _ = gs2d.gs2d_read_status(R.workspace)
    if st != gs2d.GS2D_OK:
        raise RuntimeError(f"device status after the timed region: {gs2d.status_string(st)}")
    value, total_ms = aggregate_replicas(sum(step_ms), args.steps, world, dev)
    clocks = sampler.summary()
    med_step = statistics.median(step_ms)

    # ---- per-kernel and per-call device times of the same step (traced
    # graph replays, L2 flushed before each), of the separate calls, and of
    # the render-only step
    k2 = max(20, min(args.steps, 200))
    kernels, calls, launches = w.traced(kind, k2)
    _, phases_traced, _ = w.traced("separate", k2)
    render_kernels, render_calls, _ = w.traced("render", k2)
    phases = w.call_ms("separate")
    phases.update({k: v for k, v in w.call_ms("fused" if not fwd_only else "render").items()
                   if k not in phases})
    floor_ms = trace_floor(dev, stream)
    k3 = max(20, min(args.steps, 400))
    path_ms = {}
    if not fwd_only:
        other = "separate" if kind == "fused" else "fused"
        path_ms[kind] = med_step
        path_ms[other] = statistics.median(w.timed(w.graph(w.fn(other)), k3, 5))
    render_ms = statistics.median(w.timed(w.graph(w.fn("render")), k3, 5))
    cached_ms = statistics.median(w.timed(w.graph(w.fn("cached")), k3, 5))
    # the same step launched eagerly (no CUDA graph), or through a graph when
    # the headline ran eagerly
    if args.no_graph:
        alt_graph_ms = statistics.median(w.timed(w.graph(w.fn(kind), force=True), k3, 5))
        eager_ms = med_step
    else:
        alt_graph_ms = med_step
        eager_ms = statistics.median(w.timed(w.fn(kind), k3, 5))

    # ---- roofline of the dominant raster kernel (FP32/SFU bound)
    counts = load_json(COUNTS) or {}
    props = torch.cuda.get_device_properties(dev)
    peaks = Peaks(props, clocks)
    probe = probe_peaks(dev, props.multi_processor_count)
    probe["fp32_of_derived"] = probe["fp32_tflops"] / peaks.fp32
    probe["ex2_of_derived"] = probe["ex2_per_s"] / peaks.sfu
    traffic_db = load_json(TRAFFIC) or {}
    # the stored counts are for rank 0's seed
    tp = (counts.get(args.workload) or {}).get("touching_pairs") if rank == 0 else None

    def traffic(kernel):
        return stored_traffic(traffic_db, kernel, args.workload)

    dom = dominant_raster(kernels)
    rl = roofline(peaks, dom[0], dom[1], tp, traffic(dom[0]), step_ms=med_step) if dom else None
    f = first_of(render_kernels, ("fwd_sum", "fwd_comp"))
    rl_fwd = roofline(peaks, f[0], f[1], tp, traffic(f[0]), step_ms=render_ms) if f else None
    b = first_of(kernels, ("bwd_sum", "bwd_comp", "fused_comp"))
    rl_bwd = roofline(peaks, b[0], b[1], tp, traffic(b[0]), step_ms=med_step) if b else None

    # Gaussian-pixel evaluations: the touching pairs (algorithmic) and the
    # tile-level candidates, 256 pixels for every (tile, Gaussian) pair
    evals = None
    if tp:
        cand = 256 * int(w.P)
        evals = {"touching_pairs": tp, "tile_candidates": cand, "touching_fraction": tp / cand}
        if f:
            evals["fwd_touching_per_s"] = tp / (f[1] * 1e-3)
            evals["fwd_candidates_per_s"] = cand / (f[1] * 1e-3)
        if b:
            evals["bwd_touching_per_s"] = tp / (b[1] * 1e-3)

    # ---- end to end through the same calls, host buffers, copies inside:
    # every step copies its inputs (parameters and target, one pinned buffer)
    # to the device and reads its result back (the loss; the image when the
    # workload renders only)
    h_pack = torch.from_numpy(w.host_pack).pin_memory()
    out = R.image if fwd_only else R.loss
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = h_pack.numel() * h_pack.element_size()  # the bytes copied (parts padded to 16 B)
    d2h = h_out.numel() * h_out.element_size()
    d_pack = w.d_pack

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        run_step()
        h_out.copy_(out, non_blocking=True)

    k4 = max(20, min(args.steps, 500))
    serial_ms = w.timed(e2e_step, k4, 5)
    # the host link alone: the same input copy without the step
    copy_ms = statistics.median(w.timed(lambda: d_pack.copy_(h_pack, non_blocking=True), k4, 5))
    # Pipelined, as a training loop runs: two device input buffers; step i's
    # inputs are copied on a second stream into buffer i % 2 while step i - 1
    # computes (the copy waits for step i - 2, the last reader of that
    # buffer); the step waits for its copy, then its loss is read back.
    d_packs = [d_pack, torch.empty_like(d_pack)]
    pipe_graphs = []
    for b in range(2):
        d_packs[b].copy_(h_pack)
        w.use_buffer(d_packs[b])
        pipe_graphs.append(w.graph(w.fn(kind), force=True))
    w.use_buffer(d_pack)
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_pipelined(K):
        copied = [torch.cuda.Event() for _ in range(K)]
        done = [torch.cuda.Event() for _ in range(K)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        copy_stream.wait_event(t0)
        for i in range(K):
            b = i % 2
            if i >= 2:
                copy_stream.wait_event(done[i - 2])
            with torch.cuda.stream(copy_stream):
                d_packs[b].copy_(h_pack, non_blocking=True)
                copied[i].record(copy_stream)
            stream.wait_event(copied[i])
            with torch.cuda.stream(stream):
                pipe_graphs[b]()
                h_out.copy_(out, non_blocking=True)
                done[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_pipelined(5)
    e2e_total = e2e_pipelined(k4)
    e2e_val, _ = aggregate_replicas(e2e_total, k4, world, dev)
    serial_val, _ = aggregate_replicas(sum(serial_ms), k4, world, dev)

    # ---- the selective Adam step (not part of the timed step): the step's
    # xy, shape and rgb rows with the step's gradients, moments from zero and
    # the pair counts as the selection; HBM-bound, 28 bytes per updated
    # element (p, g, m, v read; p, m, v written) plus the counts
    adam = None
    if not fwd_only:
        nG = w.wl.n
        params = [w.xy.clone(), w.chol.clone(), w.rgb.clone()]
        grads = [R.d_xy[:nG], R.d_shape[:nG], R.d_rgb[:nG]]
        moms = [(torch.zeros_like(q), torch.zeros_like(q)) for q in params]
        cnt = R.count[:nG]

        def adam_all():
            for q, g, (m1, m2) in zip(params, grads, moms):
                gs2d.adam_step(q, g, m1, m2, 1, 1e-3, count=cnt, stream=stream)
        adam_ms = statistics.median(w.timed(w.graph(adam_all, force=True), k3, 5))
        rows = int((cnt > 0).sum().item())
        upd = rows * sum(int(q[0].numel()) for q in params)
        abytes = 28 * upd + 4 * nG * len(params)
        hbm = float((load_json(PEAKS) or {}).get("hbm_gbs") or 0.0)
        agbs = abytes / (adam_ms * 1e-3) / 1e9
        adam = {"ms": adam_ms, "launches": len(params), "rows": nG, "rows_updated": rows,
                "elements_updated": upd, "bytes": abytes, "gbs": agbs,
                "hbm_frac": agbs / hbm if hbm else None,
                "how": "three gs2d_adam_step calls (xy, shape, rgb) as one CUDA graph, L2 flushed before each"}
        params = grads = moms = cnt = None

    # ---- the other workloads (one GPU only): graph-replayed throughput and
    # kernel-time rooflines
    configs = None
    if world == 1 and not args.no_configs:
        R = out = d_pack = d_packs = run_step = e2e_step = pipe_graphs = None  # drop the headline's buffers
        w.release()
        configs = {}
        for name in EXTRA_CONFIGS:
            if name != args.workload:
                configs[name] = measure_config(name, dev, stream, flush_buf, peaks, counts,
                                               args.config_steps, 3, 10,
                                               cpu=not args.no_cpu_baseline)

    # ---- CPU baseline (one GPU only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w.wl, args.cpu_seconds)

    unit = "iters/s" if not fwd_only else "frames/s"
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": describe(w.wl), "name": args.workload, "pairs": int(w.P),
                       "l2": "256 MiB buffer written before every timed step",
                       "graph": not args.no_graph,
                       "path": ("fused fwd+L2+bwd call" if kind == "fused" else
                                "separate forward, loss and backward calls") if not fwd_only else
                               "forward",
                       "replicas": "each rank renders its own independently seeded image"},
            "render_fps": 1e3 / render_ms, "cached_render_fps": 1e3 / cached_ms,
            "paths_iters_s": {k: 1e3 / v for k, v in path_ms.items()},
            "graph_vs_eager": {"graph_iters_s": 1e3 / alt_graph_ms, "eager_iters_s": 1e3 / eager_ms,
                               "note": "median step, same L2 flush; eager = one launch per kernel"},
            "gaussian_pixel_evals": evals,
            "peak_probe": probe,
            "kernels": kernel_table(kernels, med_step),
            "step_call_ms": calls,
            "phase_ms": phases,
            "adam": adam,
            "phase_basis": "device time of each call on its own: the call captured 10 times back "
                           "to back in one CUDA graph, median of 20 replays (each after an L2 "
                           "flush) / 10",
            "phase_ms_traced": phases_traced,
            "trace_floor_ms": floor_ms,
            "trace_note": "kernel times come from CUDA events recorded just before and just after "
                          "each kernel in a graph of the step; each includes about trace_floor_ms "
                          "of launch and event overhead, so the fractions derived from them are "
                          "lower bounds",
            "render_kernels": kernel_table(render_kernels, render_ms),
            "render_call_ms": render_calls,
            "roofline": rl,
            "roofline_fwd": rl_fwd, "roofline_bwd": rl_bwd,
            "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "h2d_copy_ms": copy_ms,
                    "h2d_gbs": h2d / (copy_ms * 1e-3) / 1e9, "steps": k4,
                    "how": "each step copies its inputs from pinned host memory (one buffer) and "
                           "reads its result back; the copy of step i+1 runs on a second stream "
                           "into a second device buffer while step i computes",
                    "serial_value": serial_val,
                    "serial_how": "copy, step and read-back one after the other on one stream"},
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "configs": configs,
            "wall_s": wall,
            "gpu": props.name,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gs2d(args)


if __name__ == "__main__":
    sys.exit(main())
