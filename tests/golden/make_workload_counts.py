"""Writes tests/golden/workload_counts.json: for each benchmark workload, the
number of valid Gaussians, of (tile, Gaussian) pairs P and of touching
(pixel, Gaussian) pairs, all counted by the CPU oracle on the seeded
synthetic inputs.  The benchmark reads these counts as the algorithmic work
of a forward or backward pass (the unit of work is one touching pair).

Run from the repository root:  python tests/golden/make_workload_counts.py
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from raster_gaussian_02_b300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workload_counts.json")


def count(wl):
    cfg = oracle.Config(wl.width, wl.height, wl.mode, wl.cutoff_sigma, wl.t_min)
    s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)
    fwd = s.render()
    return dict(width=wl.width, height=wl.height, n=wl.n, mode=wl.mode, valid=s.proj.valid,
                pairs=s.num_pairs, touching_pairs=fwd["masked"])


def main():
    names = sys.argv[1:] or list(synth.WORKLOADS) + [f"sweep_768x512_{k}" for k in
                                                      ("10k", "50k", "200k", "1m")]
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for name in names:
        t = time.time()
        if name.startswith("sweep_768x512_"):
            n = {"10k": 10_000, "50k": 50_000, "200k": 200_000, "1m": 1_000_000}[name.split("_")[-1]]
            wl = synth.render_uniform(768, 512, n, seed=5000 + n)
        else:
            wl = synth.WORKLOADS[name]()
        data[name] = count(wl)
        print(name, data[name], f"{time.time() - t:.1f}s", flush=True)
    json.dump(data, open(OUT, "w"), indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
