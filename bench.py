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

# Algorithmic FP32 work per touching (pixel, Gaussian) pair, FMA = 2 flops:
#   forward  dx, dy (2) + q (7) + exponent scale (1) + 3 colour FMAs (6) = 16
#   backward dx, dy (2) + q (7) + scale (1) + 3 colour-gradient FMAs (6)
#            + dL/dw = g.rgb (5) + t = w dL/dw (1) + 4 moment sums (5) = 27
# plus one SFU exp2 per pair in both.
FLOPS_FWD, FLOPS_BWD = 16, 27
# Per-SM rates per clock: 128 FP32 FMA lanes; 32 ex2 results from the SFU
# (the probe in libgs2d_probe.so measures 9.0e12 ex2/s on 148 SMs at 2032
# MHz, i.e. 30 per SM per clock, twice the 16 of earlier parts).
SM_FP32_LANES, SM_SFU_LANES = 128, 32


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

def oracle_step(wl):
    import oracle
    cfg = oracle.Config(wl.width, wl.height, wl.mode, wl.cutoff_sigma, wl.t_min, param=wl.param)
    if wl.target is None:
        s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)
        s.render()
        return
    oracle.step(cfg, wl.xy, wl.chol, wl.rgb, wl.target, wl.depth, wl.opacity, wl.background)


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
    """The CPU oracle as it stands, single-threaded, full steps of the same
    workload for about budget_s seconds (at least min_steps)."""
    oracle_step(wl)  # builds the oracle library, warms caches
    t0 = time.perf_counter()
    k = 0
    while k < min_steps or time.perf_counter() - t0 < budget_s:
        oracle_step(wl)
        k += 1
    dt = time.perf_counter() - t0
    return {"value": k / dt, "unit": "iters/s" if wl.target is not None else "frames/s",
            "cores": 1, "kind": "oracle",
            "sample": f"{k} full steps of the same workload, single-threaded C oracle, {dt:.1f} s"}


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

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def run_gs2d(args):
    import numpy as np
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

    wl = make_workload(args.workload, seed_offset=rank)
    fwd_only = wl.target is None
    # The step's inputs live in one device buffer (each part 16-byte aligned),
    # so that the end-to-end leg moves them with one host-to-device copy.
    parts = [wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background, wl.target]
    offs, total = [], 0
    for a in parts:
        offs.append(total)
        if a is not None:
            total += (a.size + 3) // 4 * 4
    host_pack = np.zeros(max(total, 4), np.float32)
    for a, o in zip(parts, offs):
        if a is not None:
            host_pack[o:o + a.size] = np.ascontiguousarray(a, np.float32).ravel()
    d_pack = torch.from_numpy(host_pack).to(dev)
    views = [None if a is None else d_pack[o:o + a.size].view(a.shape) for a, o in zip(parts, offs)]
    xy, chol, rgb, depth, opac, bg, target = views

    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min, device=dev,
                        param=wl.param)
    R.project(xy, chol, rgb, depth, opac)
    P = R.bin_and_sort(sync=True)
    R._alloc_pairs(int(P * 1.25) + 4096)  # headroom, as a fitting loop would keep
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step_separate():
        R.project(xy, chol, rgb, depth, opac)
        R.bin_and_sort(sync=False)
        R.render_fwd(bg)
        if not fwd_only:
            R.loss_l2(target)
            R.render_bwd()

    def step_fused():
        R.project_bin_and_sort(xy, chol, rgb, depth, opac, sync=False)
        R.render_fwd_bwd_l2(target, bg)

    use_fused = args.path == "fused" and not fwd_only
    step = step_fused if use_fused else step_separate

    def render():
        R.project_bin_and_sort(xy, chol, rgb, depth, opac, sync=False)
        R.render_fwd(bg)

    def cached():
        R.render_fwd(bg)

    if fwd_only and args.path == "fused":
        step = render  # the render step through the combined projection + binning call

    def graph_of_forced(fn):
        with torch.cuda.stream(stream):
            fn()
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g.replay

    def graph_of(fn):
        return fn if args.no_graph else graph_of_forced(fn)

    run_step, run_render, run_cached = graph_of(step), graph_of(render), graph_of(cached)

    def timed(fn, steps, warm, flush=True):
        """Per-step device time (ms) with the L2 flushed before each step."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        with torch.cuda.stream(stream):
            for _ in range(warm):
                fn()
            torch.cuda.synchronize()
            for a, b in ev:
                if flush:
                    flush_buf.fill_(1.0)
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    # ---- headline: K steps, max over ranks
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with sampler:
        step_ms = timed(run_step, args.steps, args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    st, pairs_now, flags = gs2d.gs2d_read_status(R.workspace)
    if st != gs2d.GS2D_OK:
        raise RuntimeError(f"device status after the timed region: {gs2d.status_string(st)}")
    value, total_ms = aggregate_replicas(sum(step_ms), args.steps, world, dev)
    clocks = sampler.summary()

    # ---- secondary numbers (each after an L2 flush, same stream)
    k2 = max(20, min(args.steps, 400))
    render_ms = statistics.median(timed(run_render, k2, 5))
    cached_ms = statistics.median(timed(run_cached, k2, 5))
    # the same step launched eagerly (no CUDA graph), or through a graph when
    # the headline ran eagerly
    if args.no_graph:
        alt_graph_ms = statistics.median(timed(graph_of_forced(step), k2, 5))
        eager_ms = statistics.median(step_ms)
    else:
        alt_graph_ms = statistics.median(step_ms)
        eager_ms = statistics.median(timed(step, k2, 5))
    path_ms = {}
    if not fwd_only:
        other = step_separate if use_fused else step_fused
        path_ms[args.path] = statistics.median(step_ms)
        path_ms["separate" if use_fused else "fused"] = statistics.median(timed(graph_of(other), k2, 5))
    phases = {}
    if True:  # eager, one call per timing pair
        names = ["project", "bin_and_sort", "render_fwd"] + (
            [] if fwd_only else ["loss_l2", "render_bwd", "render_fwd_bwd_l2"])
        fns = {"project": lambda: R.project(xy, chol, rgb, depth, opac),
               "bin_and_sort": lambda: R.bin_and_sort(sync=False),
               "render_fwd": lambda: R.render_fwd(bg),
               "loss_l2": lambda: R.loss_l2(target), "render_bwd": lambda: R.render_bwd(),
               "render_fwd_bwd_l2": lambda: R.render_fwd_bwd_l2(target, bg)}
        per = {k: [] for k in names}
        with torch.cuda.stream(stream):
            for _ in range(k2):
                for k in names:
                    flush_buf.fill_(1.0)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fns[k]()
                    b.record(stream)
                    per[k].append((a, b))
        torch.cuda.synchronize()
        phases = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in per.items()}

    # ---- roofline of the dominant raster kernel (FP32/SFU bound)
    counts = (load_json(COUNTS) or {}).get(args.workload)
    props = torch.cuda.get_device_properties(dev)
    peaks = load_json(PEAKS) or {}
    sm_max = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2032.0)
    fp32_peak = props.multi_processor_count * SM_FP32_LANES * 2 * sm_max * 1e6 / 1e12  # TFLOP/s
    sfu_peak = props.multi_processor_count * SM_SFU_LANES * sm_max * 1e6  # exp2 / s
    probe = probe_peaks(dev, props.multi_processor_count)
    probe["fp32_of_derived"] = probe["fp32_tflops"] / fp32_peak
    probe["ex2_of_derived"] = probe["ex2_per_s"] / sfu_peak
    traffic_db = load_json(TRAFFIC) or {}
    src_hash = kernel_source_hash()
    seed_mismatch = rank != 0  # the stored counts are for rank 0's seed

    def roofline(kernel, ms, flops_per_pair):
        if not counts or seed_mismatch:
            return None
        tp = counts["touching_pairs"]
        achieved = tp * flops_per_pair / (ms * 1e-3) / 1e12
        sfu_frac = tp / (ms * 1e-3) / sfu_peak
        tr = traffic_db.get(f"{kernel}:{args.workload}")
        traffic = tr["bytes"] if tr and tr.get("source_hash") == src_hash else None
        return {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": achieved / fp32_peak, "sfu_frac": sfu_frac, "traffic": traffic,
                "kernel": kernel, "ms": ms, "touching_pairs": tp, "flops_per_pair": flops_per_pair,
                "peak_basis": f"{props.multi_processor_count} SMs x {SM_FP32_LANES} FP32 lanes x 2 x "
                              f"{sm_max:.0f} MHz (max SM clock; fraction of measured-clock peak = "
                              f"frac x {sm_max:.0f}/median MHz)"}

    # Gaussian-pixel evaluations: the touching pairs (algorithmic) and the
    # tile-level candidates, 256 pixels for every (tile, Gaussian) pair
    evals = None
    if counts and not seed_mismatch:
        tp, cand = counts["touching_pairs"], 256 * int(P)
        evals = {"touching_pairs": tp, "tile_candidates": cand, "touching_fraction": tp / cand,
                 "fwd_touching_per_s": tp / (phases["render_fwd"] * 1e-3),
                 "fwd_candidates_per_s": cand / (phases["render_fwd"] * 1e-3)}
        if not fwd_only:
            evals["bwd_touching_per_s"] = tp / (phases["render_bwd"] * 1e-3)
    rl_fwd = roofline("render_fwd", phases["render_fwd"], FLOPS_FWD)
    rl_bwd = None if fwd_only else roofline("render_bwd", phases["render_bwd"], FLOPS_BWD)
    dominant = rl_fwd
    if rl_bwd and phases["render_bwd"] >= phases["render_fwd"]:
        dominant = rl_bwd

    # ---- end to end through the same calls, host buffers, copies inside:
    # every step copies its inputs (parameters and target, one pinned buffer)
    # to the device and reads its result back (the loss; the image when the
    # workload renders only)
    h_pack = torch.from_numpy(host_pack).pin_memory()
    out = R.image if fwd_only else R.loss
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = h_pack.numel() * h_pack.element_size()  # the bytes copied (parts padded to 16 B)
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        run_step()
        h_out.copy_(out, non_blocking=True)

    k3 = max(20, min(args.steps, 500))
    e2e_ms = timed(e2e_step, k3, 5)
    e2e_val, _ = aggregate_replicas(sum(e2e_ms), k3, world, dev)
    # the host link alone: the same input copy without the step
    copy_ms = statistics.median(timed(lambda: d_pack.copy_(h_pack, non_blocking=True), k3, 5))

    # ---- CPU baseline (rank 0, one GPU only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    per_step_kernels = kernels_per_step(R, wl, args.path == "fused", fwd_only)
    unit = "iters/s" if not fwd_only else "frames/s"
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": describe(wl), "name": args.workload, "pairs": int(P),
                       "l2": "256 MiB buffer written before every timed step",
                       "graph": not args.no_graph,
                       "path": ("fused fwd+L2+bwd call" if use_fused else
                                "separate forward, loss and backward calls") if not fwd_only else
                               "forward",
                       "replicas": "each rank renders its own independently seeded image"},
            "render_fps": 1e3 / render_ms, "cached_render_fps": 1e3 / cached_ms,
            "paths_iters_s": {k: 1e3 / v for k, v in path_ms.items()},
            "graph_vs_eager": {"graph_iters_s": 1e3 / alt_graph_ms, "eager_iters_s": 1e3 / eager_ms,
                               "note": "median step, same L2 flush; eager = one launch per kernel"},
            "gaussian_pixel_evals": evals,
            "peak_probe": probe,
            "phase_ms": phases,
            "roofline": dominant,
            "roofline_fwd": rl_fwd, "roofline_bwd": rl_bwd,
            "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "h2d_copy_ms": copy_ms,
                    "h2d_gbs": h2d / (copy_ms * 1e-3) / 1e9},
            "gpu_launches": per_step_kernels * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "wall_s": wall,
            "gpu": props.name,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def kernels_per_step(R, wl, fused: bool, fwd_only: bool) -> int:
    """The library's kernel launches in one step (memsets not counted), from
    the same rules the library uses to pick its kernels."""
    comp = wl.mode == 1
    T = R.num_tiles
    count_sort = T <= 2048 and wl.n <= (1 << 20)
    if count_sort:
        binning = 3 + (1 if comp else 0)  # tile histogram, tile scan, scatter (+ depth sort)
    else:
        passes = ((T - 1).bit_length() + (32 if comp else 0) + 7) // 8
        partitions = (R.capacity + 2047) // 2048
        binning = 2 + passes + (passes - 1) + (passes if partitions > 128 else 0) + 1
    # the fused step projects inside the counting sort's histogram kernel
    k = (0 if fused and count_sort else 1) + binning
    if fwd_only:
        return k + 1
    if fused:
        return k + (2 if comp else 3)  # (fused kernel | forward+loss, backward) + gather
    return k + 1 + 2 + 2  # forward, loss (2), backward + gather


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gs2d(args)


if __name__ == "__main__":
    sys.exit(main())
