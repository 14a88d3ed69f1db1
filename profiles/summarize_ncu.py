"""Summarises an ncu report exported with ``ncu -i REPORT --page raw --csv``
into a markdown table: duration, SM activity, issue activity, instruction
counts, lane efficiency, pipe utilisation, DRAM bytes and the top stall
reasons per captured kernel.

  ncu -i gpurun_out/prof.ncu-rep --page raw --csv > prof.csv
  python profiles/summarize_ncu.py prof.csv
"""
import csv
import sys

METRICS = [
    ("duration (us)", "gpu__time_duration.sum", 1.0),
    ("grid x block", None, None),
    ("registers/thread", "launch__registers_per_thread", 1.0),
    ("SM active / elapsed cycles", None, None),
    ("issue active (% of active)", "smsp__issue_active.avg.pct_of_peak_sustained_active", 1.0),
    ("warp instructions", "smsp__inst_executed.sum", 1.0),
    ("active lanes per instruction", "smsp__thread_inst_executed_per_inst_executed.ratio", 1.0),
    ("warps active per SM", "sm__warps_active.avg.per_cycle_active", 1.0),
    ("FMA pipe (% active)", "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active", 1.0),
    ("ALU pipe (% active)", "sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active", 1.0),
    ("XU (MUFU) pipe (% active)", "sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active", 1.0),
    ("DRAM read (MB)", "dram__bytes_read.sum", None),
    ("DRAM write (MB)", "dram__bytes_write.sum", None),
    ("smem bank conflicts", "l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum", 1.0),
]

SCALE_MB = {"byte": 1e-6, "Kbyte": 1e-3, "Mbyte": 1.0, "Gbyte": 1e3}


def main(path):
    rows = list(csv.reader(open(path)))
    h, units, data = rows[0], rows[1], rows[2:]
    col = {n: i for i, n in enumerate(h)}

    def get(r, n):
        return r[col[n]] if n in col else ""

    stalls = [n for n in h if n.startswith("smsp__average_warps_issue_stalled") and
              n.endswith("_per_issue_active.ratio")]
    names = [get(r, "Kernel Name").split("(")[0].split("::")[-1] for r in data]
    print("| metric | " + " | ".join(names) + " |")
    print("|---|" + "---|" * len(data))
    for label, m, _ in METRICS:
        vals = []
        for r in data:
            if label == "grid x block":
                vals.append(f"{get(r, 'launch__grid_size')} x {get(r, 'launch__block_size')}")
            elif label == "SM active / elapsed cycles":
                a = float(get(r, "sm__cycles_active.avg") or 0)
                e = float(get(r, "sm__cycles_elapsed.avg") or 1)
                vals.append(f"{a:,.0f} / {e:,.0f} ({100 * a / e:.0f} %)")
            elif m.startswith("dram__bytes"):
                u = units[col[m]]
                vals.append(f"{float(get(r, m) or 0) * SCALE_MB.get(u, 1.0):.2f}")
            else:
                v = get(r, m)
                try:
                    f = float(v)
                    vals.append(f"{f:,.0f}" if f >= 1000 else f"{f:.2f}")
                except ValueError:
                    vals.append(v or "n/a")
        print(f"| {label} | " + " | ".join(vals) + " |")
    tops = []
    for r in data:
        st = sorted(((float(get(r, n) or 0), n[len("smsp__average_warps_issue_stalled_"):-len(
            "_per_issue_active.ratio")]) for n in stalls), reverse=True)[:4]
        tops.append(", ".join(f"{n} {v:.1f}" for v, n in st))
    print("| top stalls (warps per issue) | " + " | ".join(tops) + " |")


if __name__ == "__main__":
    main(sys.argv[1])
