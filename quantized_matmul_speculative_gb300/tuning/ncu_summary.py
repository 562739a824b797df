"""Write a short markdown summary of Nsight Compute output for profiles/.

Inputs: the CSV launch list of an ``ncu --metrics gpu__time_duration.sum``
pass, and a ``--page raw --csv`` export of a ``--set full`` capture of the
dominant kernel.  The summary records the hash of the kernel sources it was
taken on; bench.py uses its DRAM traffic only while that hash still matches.

    python -m quantized_matmul_speculative_gb300.tuning.ncu_summary \
        --launches launches.csv --raw raw.csv --workload NAME --out profiles/qmm_tma_NAME.md \
        --list-cmd "..." --full-cmd "..."
"""
from __future__ import annotations

import argparse
import collections
import csv
import hashlib
from pathlib import Path

CSRC = Path(__file__).resolve().parents[1] / "csrc"
# Sources of the TMA kernel families; a profile is valid only for the hash of these.
KERNEL_SOURCES = ("qmm_tma.cuh", "qmm_tma_launch.cuh", "qmm_own.cuh", "qmm_own_launch.cuh", "qmm_group.cuh",
                  "qmm_device.cuh", "qmm_gather.cuh", "qmm_tiles.h", "qmm_geometry.h")

RAW_METRICS = [
    ("gpu__time_duration.sum", "duration (serialized, cold)"),
    ("dram__bytes_read.sum", "DRAM bytes read"),
    ("dram__bytes_write.sum", "DRAM bytes written"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput % of peak"),
    ("sm__throughput.avg.pct_of_peak_sustained_elapsed", "SM throughput % of peak"),
    ("smsp__issue_active.avg.pct_of_peak_sustained_active", "issue slots used %"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", "tensor pipe active %"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active %"),
    ("smsp__inst_executed.sum", "warp instructions"),
    ("l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum", "shared-memory bank conflicts"),
    ("launch__registers_per_thread", "registers / thread"),
    ("launch__shared_mem_per_block_dynamic", "dynamic shared memory / CTA"),
    ("launch__grid_size", "CTAs"),
    ("launch__cluster_dim_x", "cluster size"),
]


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        h.update((CSRC / name).read_bytes())
    return h.hexdigest()[:16]


def to_float(s: str) -> float:
    return float(s.replace(",", ""))


def launch_table(path: Path):
    rows = list(csv.reader(path.open()))
    hi = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    h = rows[hi]
    ki, vi, ui = h.index("Kernel Name"), h.index("Metric Value"), h.index("Metric Unit")
    scale = {"ns": 1e-3, "us": 1.0, "usecond": 1.0, "nsecond": 1e-3, "ms": 1e3}
    agg = collections.defaultdict(list)
    for r in rows[hi + 1:]:
        if len(r) > vi and r[vi]:
            agg[r[ki].split("(")[0]].append(to_float(r[vi]) * scale.get(r[ui], 1.0))
    total = sum(sum(v) for v in agg.values())
    return [(k, len(v), sum(v), 100.0 * sum(v) / total) for k, v in sorted(agg.items(), key=lambda kv: -sum(kv[1]))]


def raw_metrics(path: Path):
    rows = list(csv.reader(path.open()))
    h, units, data = rows[0], rows[1], rows[2:]
    out = {"kernel": data[0][h.index("Kernel Name")]}
    for name, _ in RAW_METRICS:
        if name in h:
            i = h.index(name)
            out[name] = ([d[i] for d in data], units[i])
    stalls = {}
    for i, c in enumerate(h):
        if c.startswith("smsp__average_warps_issue_stalled_") and c.endswith("_per_issue_active.ratio"):
            try:
                v = to_float(data[0][i])
            except ValueError:
                continue
            if v >= 0.1:
                stalls[c.replace("smsp__average_warps_issue_stalled_", "").replace("_per_issue_active.ratio", "")] = v
    out["stalls"] = stalls
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--launches", required=True)
    ap.add_argument("--raw", required=True)
    ap.add_argument("--workload", required=True)
    ap.add_argument("--out", required=True)
    ap.add_argument("--list-cmd", required=True)
    ap.add_argument("--full-cmd", required=True)
    ap.add_argument("--note", default="")
    ap.add_argument("--sources", default=",".join(KERNEL_SOURCES),
                    help="comma-separated csrc files whose hash the summary records (default: the TMA families')")
    a = ap.parse_args()
    sources = tuple(x for x in a.sources.split(",") if x)
    lt = launch_table(Path(a.launches))
    rm = raw_metrics(Path(a.raw))
    reads = [to_float(v) for v in rm["dram__bytes_read.sum"][0]]
    writes = [to_float(v) for v in rm["dram__bytes_write.sum"][0]]
    unit_r, unit_w = rm["dram__bytes_read.sum"][1], rm["dram__bytes_write.sum"][1]
    mult = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per_launch = [r * mult.get(unit_r, 1) + w * mult.get(unit_w, 1) for r, w in zip(reads, writes)]
    families = ("qmm_own_kernel", "qmm_tma_kernel", "qmm_mma_kernel", "ggml_to_affine_kernel")
    family = next((f for f in families if f in rm["kernel"]), rm["kernel"])
    lines = [f"# ncu summary: {family} on {a.workload}", ""]
    if a.note:
        lines += [a.note, ""]
    if sources != KERNEL_SOURCES:
        lines += ["Hashed sources: " + ", ".join(f"`{x}`" for x in sources), ""]
    lines += ["kernel_source_hash: " + kernel_hash(sources),
              f"dram_bytes_per_launch: {sum(per_launch) / len(per_launch):.0f}", "",
              "## Launch list (per-launch times are cold-cache and serialized; compare shares)", "",
              "Command:", "", "```", a.list_cmd, "```", "",
              "| kernel | launches | total us | share |", "|---|---|---|---|"]
    for k, n, tot, share in lt:
        lines.append(f"| `{k}` | {n} | {tot:.1f} | {share:.1f}% |")
    lines += ["", "## Full capture of the dominant kernel", "", "Command:", "", "```", a.full_cmd, "```", "",
              f"Kernel: `{rm['kernel']}`", "", "| metric | value (per captured launch) |", "|---|---|"]
    for name, label in RAW_METRICS:
        if name in rm:
            vals, unit = rm[name]
            lines.append(f"| {label} (`{name}`) | {', '.join(vals)} {unit} |")
    lines += ["", "Warp stall reasons (cycles per issued instruction, >= 0.1):", ""]
    for k, v in sorted(rm["stalls"].items(), key=lambda kv: -kv[1]):
        lines.append(f"- {k}: {v:.2f}")
    Path(a.out).write_text("\n".join(lines) + "\n")
    print(f"wrote {a.out}")


if __name__ == "__main__":
    main()
