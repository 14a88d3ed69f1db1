"""Summarises an ncu launch list (``--metrics gpu__time_duration.sum --csv``)
per kernel: launches, total device time, mean per launch and share.

  python profiles/summarize_launches.py gpurun_out/launches.csv
"""
import collections
import csv
import re
import sys

SCALE = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3}


def short(name: str) -> str:
    name = re.sub(r"\(.*", "", name)
    name = name.replace("void ", "").replace("gs2d::<unnamed>::", "")
    return name[:48]


def main(path):
    rows = list(csv.reader(open(path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    k, m, v, u = (h.index(x) for x in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    agg = collections.defaultdict(lambda: [0, 0.0])
    for r in rows[hi + 1:]:
        if len(r) <= v or r[m] != "gpu__time_duration.sum":
            continue
        t = float(r[v].replace(",", "")) * SCALE[r[u]]
        a = agg[short(r[k])]
        a[0] += 1
        a[1] += t
    ours = {n: a for n, a in agg.items() if n.startswith("k_")}
    tot = sum(a[1] for a in ours.values())
    print(f"{'kernel':48s} {'launches':>8s} {'total us':>10s} {'us/launch':>10s} {'share':>6s}")
    for n, (c, t) in sorted(ours.items(), key=lambda x: -x[1][1]):
        print(f"{n:48s} {c:8d} {t:10.1f} {t / c:10.2f} {100 * t / tot:5.1f}%")
    other = sum(a[1] for n, a in agg.items() if not n.startswith("k_"))
    print(f"(other kernels in the process, e.g. the L2 flush: {other:.1f} us, not in the shares)")


if __name__ == "__main__":
    main(sys.argv[1])
