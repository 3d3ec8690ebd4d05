"""Summarise an Nsight Compute launch list (``ncu --csv --log-file``) per kernel.

    python -m iteration_level_selective_gb300.ncu_summary launches.csv \
        [--traffic profiles/traffic.json --workload gpt2-trace --scale S]
    python -m iteration_level_selective_gb300.ncu_summary --raw capture_raw.csv

The second form reads the raw page of a capture (``ncu -i X.ncu-rep --page raw
--csv > capture_raw.csv``) and prints the figures the profile summaries quote,
one column per captured launch.

prints one markdown row per kernel (launches, total device time, share,
average time, DRAM bytes per launch when the capture has the
``dram__bytes_read.sum`` / ``dram__bytes_write.sum`` counters) and, with
``--traffic``, records the measured DRAM bytes per launch of each kernel class
the benchmark reports (``gemm_tc_bf16``, ``attention``, ``layernorm``,
``embed``) under the workload's name, together with a hash of the kernel
sources so that a stale figure is never reported after the kernels change.
``--scale`` multiplies the bytes (a capture of a smaller case scaled to the
full launch by the units processed).  The attention class counts one launch
per layer, so its bytes are those of both attention kernels over the number
of launches of the ragged (CUDA-core) kernel.
"""
from __future__ import annotations

import argparse
import collections
import csv
import hashlib
import io
import json
import os
import re
import sys

CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc")

_TIME = {"ns": 1e-6, "nsecond": 1e-6, "us": 1e-3, "usecond": 1e-3, "ms": 1.0, "msecond": 1.0, "s": 1e3,
         "second": 1e3}
_BYTES = {"byte": 1.0, "b": 1.0, "kbyte": 1e3, "kb": 1e3, "mbyte": 1e6, "mb": 1e6, "gbyte": 1e9, "gb": 1e9}

CLASSES = {
    "gemm_tc_bf16": ("gemm_tc_bf16_kernel", "gemm_tc_cluster_kernel", "gemm_tc_pair_kernel"),
    "attention": ("attention_kernel", "prefill_attention_tc_kernel"),
    "layernorm": ("layernorm_kernel",),
    "embed": ("embed_kernel",),
}
# classes whose kernels are alternatives (one launch each): bytes over all their launches;
# the others count the launches of their first kernel (attention: one per layer)
ALTERNATIVES = {"gemm_tc_bf16"}


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(csrc: str = CSRC) -> str:
    """Hash of the CUDA/C++ sources' code (comments and layout do not count:
    a profile stays valid across comment edits); the benchmark uses the same."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def short_name(full: str) -> str:
    """'void orca::(anonymous namespace)::gemm_tc_bf16_kernel<128>(...)' -> 'gemm_tc_bf16_kernel'
    (ncu also prints the anonymous namespace as '<unnamed>')."""
    head = re.split(r"[<(]", full.replace("(anonymous namespace)", "").replace("<unnamed>", ""), maxsplit=1)[0]
    return head.split("::")[-1].split()[-1]


def read_launches(path: str):
    """{launch id: {"kernel": name, metric: value in ms or bytes}}."""
    with open(path, newline="") as f:
        text = f.read()
    start = text.find('"ID"')
    if start < 0:
        raise ValueError(f"{path}: no ncu CSV header")
    launches = collections.OrderedDict()
    for row in csv.DictReader(io.StringIO(text[start:])):
        lid = row["ID"]
        ent = launches.setdefault(lid, {"kernel": short_name(row["Kernel Name"])})
        name, unit = row["Metric Name"], row["Metric Unit"].strip().lower()
        try:
            val = float(row["Metric Value"].replace(",", ""))
        except ValueError:
            continue
        if name == "gpu__time_duration.sum":
            ent["ms"] = val * _TIME.get(unit, 1e-6)
        elif name in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            ent[name] = val * _BYTES.get(unit, 1.0)
    return launches


def summarise(launches):
    per = collections.OrderedDict()
    for ent in launches.values():
        k = per.setdefault(ent["kernel"], {"launches": 0, "ms": 0.0, "dram": 0.0, "has_dram": False})
        k["launches"] += 1
        k["ms"] += ent.get("ms", 0.0)
        if "dram__bytes_read.sum" in ent or "dram__bytes_write.sum" in ent:
            k["has_dram"] = True
            k["dram"] += ent.get("dram__bytes_read.sum", 0.0) + ent.get("dram__bytes_write.sum", 0.0)
    return per


def markdown(per) -> str:
    total = sum(v["ms"] for v in per.values()) or 1.0
    n = sum(v["launches"] for v in per.values())
    out = [f"Launches: {n}; total kernel time {total:.2f} ms.", "",
           "| kernel | launches | total ms | share | avg us/launch | DRAM MB/launch |",
           "|---|---|---|---|---|---|"]
    for k, v in sorted(per.items(), key=lambda kv: -kv[1]["ms"]):
        dram = f"{v['dram'] / v['launches'] / 1e6:.3f}" if v["has_dram"] else "-"
        out.append(f"| {k} | {v['launches']} | {v['ms']:.3f} | {v['ms'] / total:.3f} | "
                   f"{1000 * v['ms'] / v['launches']:.2f} | {dram} |")
    return "\n".join(out)


def traffic_by_class(per, scale: float = 1.0):
    res = {}
    for cls, names in CLASSES.items():
        present = [n for n in names if n in per and per[n]["has_dram"]]
        if not present:
            continue
        if cls in ALTERNATIVES:
            n_launch = sum(per[n]["launches"] for n in names if n in per)
        else:
            n_launch = per[present[0]]["launches"]   # the first name present counts the class's launches
        res[cls] = scale * sum(per[n]["dram"] for n in present) / n_launch
    return res


# (label, metric name, scale to the printed unit: None = print as captured)
RAW_ROWS = (
    ("duration (us)", "gpu__time_duration.sum", _TIME),
    ("SM clock (GHz)", "sm__cycles_elapsed.avg.per_second", None),
    ("tensor pipe active, % of elapsed", "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", None),
    ("XU pipe (exp), % of active", "sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active", None),
    ("ALU pipe, % of active", "sm__inst_executed_pipe_alu.avg.pct_of_peak_sustained_active", None),
    ("warps active, % of peak", "sm__warps_active.avg.pct_of_peak_sustained_active", None),
    ("SM throughput, %", "sm__throughput.avg.pct_of_peak_sustained_elapsed", None),
    ("DRAM throughput, % of peak", "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", None),
    ("DRAM bytes per second", "dram__bytes.sum.per_second", None),
    ("DRAM read (GB)", "dram__bytes_read.sum", _BYTES),
    ("DRAM write (GB)", "dram__bytes_write.sum", _BYTES),
    ("L2 hit rate, %", "lts__t_sector_hit_rate.pct", None),
    ("grid", "launch__grid_size", None),
    ("block", "launch__block_size", None),
    ("cluster", "launch__cluster_dim_x", None),
    ("registers / thread", "launch__registers_per_thread", None),
    ("dynamic shared memory", "launch__shared_mem_per_block_dynamic", None),
)
STALL = "smsp__pcsamp_warps_issue_stalled_"


def _num(v: str) -> float:
    return float(v.replace(",", ""))


def raw_summary(text: str) -> str:
    """Markdown table of RAW_ROWS (and the three largest sampled warp-stall
    reasons) from an ncu raw-page CSV: header row, units row, one row per
    launch."""
    rows = list(csv.reader(io.StringIO(text)))
    rows = [r for r in rows if r]
    head, units, data = rows[0], rows[1], rows[2:]
    col = {k: i for i, k in enumerate(head)}
    names = [short_name(r[col["Kernel Name"]]) if "Kernel Name" in col else f"launch {j}" for j, r in enumerate(data)]
    out = ["| metric | " + " | ".join(names) + " |", "|---|" + "---|" * len(data)]
    for label, key, conv in RAW_ROWS:
        if key not in col:
            continue
        cells = []
        for r in data:
            v, u = r[col[key]], units[col[key]].strip()
            try:
                x = _num(v)
            except ValueError:
                cells.append(v)
                continue
            if conv is _TIME:
                x *= _TIME.get(u.lower(), 1.0) * 1e3   # -> us
            elif conv is _BYTES:
                x *= _BYTES.get(u.lower(), 1.0) / 1e9  # -> GB
            cells.append(f"{x:.4g}" + ("" if conv is not None or not u else f" {u}"))
        out.append(f"| {label} | " + " | ".join(cells) + " |")
    stalls = [k for k in head if k.startswith(STALL) and not k.endswith("_not_issued")]
    if stalls:
        cells = []
        for r in data:
            vals = []
            for k in stalls:
                try:
                    vals.append((_num(r[col[k]]), k[len(STALL):]))
                except ValueError:
                    pass
            top = sorted(vals, reverse=True)[:3]
            cells.append(", ".join(f"{n} {int(c)}" for c, n in top))
        out.append("| top sampled stall reasons | " + " | ".join(cells) + " |")
    return "\n".join(out)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("csv")
    ap.add_argument("--raw", action="store_true", help="the csv is a capture's raw page (ncu -i --page raw --csv)")
    ap.add_argument("--traffic", help="JSON file to record per-launch DRAM bytes in")
    ap.add_argument("--workload", default="gpt2-trace")
    ap.add_argument("--scale", type=float, default=1.0)
    ap.add_argument("--note", default="")
    args = ap.parse_args(argv)
    if args.raw:
        with open(args.csv) as f:
            print(raw_summary(f.read()))
        return 0
    per = summarise(read_launches(args.csv))
    print(markdown(per))
    if args.traffic:
        d = {}
        if os.path.exists(args.traffic):
            with open(args.traffic) as f:
                d = json.load(f)
        h = source_hash()
        ent = d.setdefault(args.workload, {})
        for cls, b in traffic_by_class(per, args.scale).items():
            ent[cls] = {"bytes_per_launch": b, "source_hash": h, "scale": args.scale, "note": args.note}
        with open(args.traffic, "w") as f:
            json.dump(d, f, indent=1)
            f.write("\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
