"""Turn ncu CSVs of DRAM counters into profiles/traffic.json for bench.py.

    python -m bwd_gemm_epilogue_gb300.traffic_summary "<how the CSVs were taken>" [kind=]a.csv [[kind=]b.csv ...]

Each CSV comes from one ncu capture of `--metrics dram__bytes_read.sum,
dram__bytes_write.sum,gpu__time_duration.sum` (one pass) on one or more launches of the
target block's kernels.  Launches are mapped to kernel kinds by their template arguments
(gemm_kernel<EPI, CG, SCHED, OP>, bf16 operands; plain or demangled kernel names) unless
the argument names the kind (`fwd_down=dram_fwd_down.csv`: the down projection and the grouped
backward can both run as <4, 2, 1, 0>, a list launch of 256 x 512 tiles), averaged per kind, and written with a hash of the kernel sources: bench.py reports a
kind's traffic only while the sources still hash the same (a changed kernel invalidates
its counters).
"""
from __future__ import annotations

import csv
import json
import os
import re
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)

# template arguments of the target step's four launches -> bench kind names
# (EPI 4: the store epilogue over 256 x 512 tiles, which the grouped backward uses at this size)
KINDS = {("1", "2", "0"): "fwd_preact", ("0", "2", "0"): "fwd_down", ("2", "2", "0"): "bwd_grad_h",
         ("0", "2", "1"): "bwd_gemms", ("4", "2", "1"): "bwd_gemms", ("4", "2", "0"): "fwd_down"}


def summarize(path: str, kind: str | None = None) -> dict:
    rows = list(csv.reader(open(path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, ii, mi, ui, vi = (h.index(c) for c in ("Kernel Name", "ID", "Metric Name", "Metric Unit", "Metric Value"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1, "us": 1e3, "ms": 1e6}
    per_launch = {}
    for r in rows[hi + 1:]:
        if len(r) <= vi:
            continue
        m = re.search(r"gemm_kernel<(?:\(int\))?(\d+), (?:\(int\))?(\d+), (?:\(int\))?(\d+)(?:, (?:\(int\))?(\d+))?>",
                      r[ki])
        if not m or m.group(4) not in (None, "0") or (kind is None and m.groups()[:3] not in KINDS):
            continue
        d = per_launch.setdefault(r[ii], {"kind": kind or KINDS[m.groups()[:3]]})
        d[r[mi]] = float(r[vi].replace(",", "")) * scale.get(r[ui], 1)
    acc = {}
    for d in per_launch.values():
        a = acc.setdefault(d["kind"], [0, 0.0, 0.0, 0.0])
        a[0] += 1
        a[1] += d.get("dram__bytes_read.sum", 0.0)
        a[2] += d.get("dram__bytes_write.sum", 0.0)
        a[3] += d.get("gpu__time_duration.sum", 0.0)
    return {k: {"launches": n, "dram_read_bytes_per_launch": round(r / n),
                "dram_write_bytes_per_launch": round(w / n),
                "dram_bytes_per_launch": round((r + w) / n),
                "ncu_duration_ns_per_launch": round(t / n)} for k, (n, r, w, t) in acc.items()}


def main():
    import bench
    command, paths = sys.argv[1], sys.argv[2:]
    kernels = {}
    for arg in paths:
        kind, sep, path = arg.partition("=")
        kernels.update(summarize(path, kind) if sep else summarize(arg))
    out = {"source_hash": bench.kernel_source_hash(), "command": command,
           "workload": "target step: M=11136, D=Dout=3584, H=14336", "kernels": kernels}
    dst = os.path.join(ROOT, "profiles", "traffic.json")
    json.dump(out, open(dst, "w"), indent=1)
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
