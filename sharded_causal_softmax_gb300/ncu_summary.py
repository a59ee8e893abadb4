"""Summarise an ncu launch list (``--metrics gpu__time_duration.sum --csv``)
into per-kernel launches, total time and share; and pull the roofline
counters of a ``--set full`` report.  Used to write the text summaries kept
under profiles/.

    python -m sharded_causal_softmax_gb300.ncu_summary launches <launches.csv>
    python -m sharded_causal_softmax_gb300.ncu_summary counters <report.ncu-rep>
"""
from __future__ import annotations

import csv
import io
import re
import subprocess
import sys
from collections import defaultdict

COUNTERS = ["gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
            "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed",
            "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
            "smsp__inst_executed.sum",
            "l1tex__data_pipe_lsu_wavefronts_mem_shared.sum.pct_of_peak_sustained_elapsed",
            "l1tex__data_pipe_tc_wavefronts_mem_shared.sum.pct_of_peak_sustained_elapsed",
            "l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum",
            "l1tex__m_l1tex2xbar_write_bytes_mem_global_op_tma_red.sum",
            "sm__mem_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
            "sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active",
            "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active",
            "sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active",
            "smsp__issue_active.avg.pct_of_peak_sustained_active", "sm__warps_active.avg.pct_of_peak_sustained_active",
            "smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio",
            "smsp__average_warps_issue_stalled_wait_per_issue_active.ratio",
            "smsp__average_warps_issue_stalled_short_scoreboard_per_issue_active.ratio",
            "smsp__average_warps_issue_stalled_branch_resolving_per_issue_active.ratio",
            "launch__registers_per_thread", "launch__grid_size", "launch__block_size",
            "sm__cycles_elapsed.avg.per_second"]

_UNIT = {"ns": 1e-6, "nsecond": 1e-6, "us": 1e-3, "usecond": 1e-3, "ms": 1.0, "msecond": 1.0,
         "s": 1e3, "second": 1e3}


def _short(name: str) -> str:
    m = re.search(r"(\w+_kernel)", name)
    return m.group(1) if m else name.split("(")[0][:60]


def launches(path: str) -> str:
    text = open(path).read()
    start = text.find('"ID"')
    rows = list(csv.DictReader(io.StringIO(text[start:])))
    per = defaultdict(lambda: [0, 0.0])
    for r in rows:
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        ms = float(r["Metric Value"].replace(",", "")) * _UNIT.get(r.get("Metric Unit"), 1.0)
        k = _short(r["Kernel Name"])
        per[k][0] += 1
        per[k][1] += ms
    total = sum(v[1] for v in per.values())
    out = [f"{'kernel':36s} {'launches':>8s} {'total ms':>10s} {'share':>7s}"]
    for k, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        out.append(f"{k:36s} {n:8d} {t:10.3f} {100 * t / total:6.1f}%")
    out.append(f"{'total':36s} {sum(v[0] for v in per.values()):8d} {total:10.3f}")
    return "\n".join(out)


def counters(path: str) -> str:
    raw = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True, text=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    hdr, units = rows[0], rows[1]
    out = []
    for vals in rows[2:]:
        kname = vals[hdr.index("Kernel Name")] if "Kernel Name" in hdr else "?"
        out.append(f"kernel: {_short(kname)}")
        for c in COUNTERS:
            if c in hdr:
                i = hdr.index(c)
                out.append(f"  {c:78s} {vals[i]:>14s} {units[i]}")
    return "\n".join(out)


def traffic(path: str, kernel: str, workload: str, scale: float, sources, match: str | None = None) -> dict:
    """Record dram read+write bytes of the captured launch of `kernel`,
    scaled by `scale` (units of the bench launch / units of the captured
    launch), with a hash of the kernel's sources (the bench reports the
    figure only while the sources are unchanged).  With `match`, the bytes
    of every captured launch whose kernel name matches that regex are added
    up (one library call made of several kernels); else the first launch."""
    import hashlib
    import json
    import os
    raw = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True, text=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    hdr, units = rows[0], rows[1]
    mult = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    ki = hdr.index("Kernel Name")
    picked = [v for v in rows[2:] if re.search(match, v[ki])] if match else rows[2:3]

    def get(vals, name):
        i = hdr.index(name)
        return float(vals[i].replace(",", "")) * mult.get(units[i], 1)

    bytes_ = sum(get(v, "dram__bytes_read.sum") + get(v, "dram__bytes_write.sum") for v in picked)
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc")
    h = hashlib.sha256()
    for n in sources:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    rec = {"workload": workload, "dram_bytes_per_launch": bytes_ * scale, "captured_bytes": bytes_,
           "scale": scale, "source_hash": h.hexdigest()[:16], "report": os.path.basename(path)}
    out = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "traffic.json")
    data = {}
    if os.path.exists(out):
        with open(out) as f:
            data = json.load(f)
    data[kernel] = rec
    with open(out, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    return rec


if __name__ == "__main__":
    what, path = sys.argv[1], sys.argv[2]
    if what == "launches":
        print(launches(path))
    elif what == "counters":
        print(counters(path))
    elif what == "traffic":
        # traffic <report> <kernel> <workload> <scale> <source files...> [--match <regex>]
        rest = sys.argv[6:]
        match = None
        if "--match" in rest:
            i = rest.index("--match")
            match = rest[i + 1]
            rest = rest[:i] + rest[i + 2:]
        print(traffic(path, sys.argv[3], sys.argv[4], float(sys.argv[5]), rest, match))
