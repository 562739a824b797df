"""Time every kernel variant and split count on the workload shapes.

Each measurement is a CUDA graph of back-to-back calls at one (shape, M,
variant, splits), every call reading a different copy of the weights (copies
in rotation > 4x L2, so HBM is cold), timed with CUDA events; the median of
several replays is kept.  Variants are interleaved per shape so that clock
drift affects all of them alike.  Output: one JSON object per line.

    python -m quantized_matmul_speculative_gb300.tuning.sweep --out sweep.jsonl [--quick]
        [--only-n N ...] [--only-bits B]
"""
from __future__ import annotations

import argparse
import json
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

from quantized_matmul_speculative_gb300 import binding, build, synth, workloads  # noqa: E402


def shapes(quick: bool, extra_m=()):
    """(N, K, bits, group_size, Ms) of every workload shape; `extra_m` adds M
    values to every shape (e.g. rows above 8 on shapes whose workload stops at
    8, so that the dispatcher has measured entries for them too)."""
    out = []
    for w in workloads.ALL:
        pairs = w.variants or ((w.bits, w.group_size),)
        for sh in w.shapes:
            for bits, gs in pairs:
                ms = tuple(w.ms) if not quick else tuple(m for m in w.ms if m in (1, 4, 8, 16))
                ms = tuple(sorted(set(ms) | set(extra_m)))
                out.append((sh.N, sh.K, bits, gs, ms or (w.ms[0],)))
    # merge duplicates (same N, K, bits, gs): union of Ms
    merged = {}
    for N, K, bits, gs, ms in out:
        merged.setdefault((N, K, bits, gs), set()).update(ms)
    return [(N, K, b, g, tuple(sorted(ms))) for (N, K, b, g), ms in merged.items()]


def candidates(nvar: int, groups: int):
    """(variant, splits): the TMA families try every cluster size up to 16
    that divides the group count (non-powers of two balance tiles over
    clusters better on some shapes); the mma family 1, 2, 4, 8."""
    names = binding.variant_names()
    for v in range(nvar):
        if names[v].startswith("tma"):
            for s in range(1, 17):
                if groups % s == 0 and (s <= 8 or s == 16 or s in (10, 12)):
                    yield v, s
        else:
            for s in (1, 2, 4, 8):
                yield v, s


def time_config(torch, copies, x, y, M, N, K, bits, gs, v, s, stream, calls=48, reps=5):
    handle = stream.cuda_stream

    def call(i):
        wq, sc, bi = copies[i % len(copies)]
        binding.small_m_ptr(x.data_ptr(), wq.data_ptr(), sc.data_ptr(), bi.data_ptr(), M, N, K, bits, gs,
                            y.data_ptr(), binding.OUT_BF16, v, s, handle)

    with torch.cuda.stream(stream):
        call(0)  # validates, sets kernel attributes
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            call(i)
    times = []
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / calls)
    del g
    return float(np.median(times)), float(min(times)), float(max(times))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", required=True)
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--only-n", type=int, default=None, help="sweep only shapes with this N (repeatable)",
                    action="append")
    ap.add_argument("--only-bits", type=int, default=None, help="sweep only shapes of this code width")
    ap.add_argument("--extra-m", type=int, action="append", default=[], help="also sweep this M on every shape")
    args = ap.parse_args()
    import torch

    build.build()
    binding.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = binding.variant_names()
    out = open(args.out, "w")
    for N, K, bits, gs, ms in shapes(args.quick, args.extra_m):
        if args.only_n and N not in args.only_n:
            continue
        if args.only_bits and bits != args.only_bits:
            continue
        p = synth.make_problem(1, N, K, bits, gs)
        call_b = workloads.call_bytes(N, K, bits, gs)
        ncopy = max(2, int(np.ceil(4 * l2 / call_b)) + 1)
        wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32))
        sc = torch.from_numpy(p.scales.view(np.float16))
        bi = torch.from_numpy(p.biases.view(np.float16))
        copies = [(wq.to(dev), sc.to(dev), bi.to(dev)) for _ in range(ncopy)]
        x = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty((16, N), dtype=torch.bfloat16, device=dev)
        for M in ms:
            for v, s in candidates(len(names), K // gs):
                t0 = time.time()
                try:
                    med, lo, hi = time_config(torch, copies, x, y, M, N, K, bits, gs, v, s, stream)
                except binding.QmmError as e:
                    if e.status == 3:
                        continue
                    raise
                rec = {"M": M, "N": N, "K": K, "bits": bits, "gs": gs, "variant": names[v], "variant_id": v,
                       "splits": s, "us": round(med, 3), "us_min": round(lo, 3), "us_max": round(hi, 3),
                       "gbs": round(call_b / (med * 1e-6) / 1e9, 1), "wall_s": round(time.time() - t0, 2)}
                out.write(json.dumps(rec) + "\n")
                out.flush()
        del copies
        torch.cuda.empty_cache()
    status = binding.device_status()
    print(json.dumps({"done": True, "device_status": status}))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
