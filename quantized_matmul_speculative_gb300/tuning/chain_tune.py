"""Tune the verify-step shapes in the chain they run in.

The isolated sweep (sweep.py) times each (shape, M, variant, splits) in a
chain of calls to that one shape.  In the whole verify step the four
projections alternate, and a variant's cost depends on its neighbours (how
their CTAs overlap under programmatic dependent launch, cluster placement).
This script builds the 36-layer verify-step chain (as bench.py does) and,
for every M, does coordinate descent over the projections: each in turn
tries its best isolated candidates while the others stay fixed, keeping the
choice that makes the whole step fastest.  Output: one JSON object per
(M, projection) with "source": "chain"; make_table.py lets these entries
override the isolated ones.

    python -m quantized_matmul_speculative_gb300.tuning.chain_tune \\
        --sweep tuning/sweep_gb300.jsonl --out tuning/chain_gb300.jsonl
"""
from __future__ import annotations

import argparse
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

from quantized_matmul_speculative_gb300 import binding, build, synth, workloads  # noqa: E402
from quantized_matmul_speculative_gb300.tuning.make_table import EXCLUDED_SUFFIXES  # noqa: E402


def isolated_candidates(sweep_path: Path, top: int, top_excluded: int):
    """(M, N, K) -> [(variant name, splits)] from the isolated sweep: the `top`
    fastest the table may pick, then the `top_excluded` fastest of the
    variants it never picks on its own (those are judged here, in the chain)."""
    rows, extra = {}, {}
    for line in sweep_path.read_text().splitlines():
        if not line.strip():
            continue
        r = json.loads(line)
        if "us" not in r:
            continue
        dst = extra if r["variant"].endswith(EXCLUDED_SUFFIXES) else rows
        dst.setdefault((r["M"], r["N"], r["K"]), []).append((r["us"], r["variant"], r["splits"]))
    out = {}
    for k, c in rows.items():
        out[k] = [(v, s) for _, v, s in sorted(c)[:top]]
        out[k] += [(v, s) for _, v, s in sorted(extra.get(k, []))[:top_excluded]]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--sweep", required=True)
    ap.add_argument("--out", required=True)
    ap.add_argument("--top", type=int, default=4)
    ap.add_argument("--top-excluded", type=int, default=2)
    ap.add_argument("--passes", type=int, default=2)
    ap.add_argument("--steps", type=int, default=8)
    args = ap.parse_args()
    import torch

    build.build()
    binding.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.Stream(dev)
    handle = stream.cuda_stream
    names = binding.variant_names()
    w = workloads.VERIFY_STEP
    bits, gs = w.bits, w.group_size
    cands = isolated_candidates(Path(args.sweep), args.top, args.top_excluded)

    mats = []
    x0 = None
    for si, sh in enumerate(w.shapes):
        p = synth.make_problem(workloads.shape_seed(w, si), sh.N, sh.K, bits, gs)
        mats.append((sh, torch.from_numpy(binding.pack(p.q, bits).view(np.int32)).to(dev),
                     torch.from_numpy(p.scales.view(np.float16)).to(dev),
                     torch.from_numpy(p.biases.view(np.float16)).to(dev)))
        if si == 0:
            x0 = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
    layers = [[(sh, wq.clone(), sc.clone(), bi.clone()) for sh, wq, sc, bi in mats] for _ in range(w.layers)]
    del mats
    outs = [torch.empty((16 * sh.N,), dtype=torch.bfloat16, device=dev) for sh in w.shapes]
    act = torch.empty((16 * w.shapes[0].K,), dtype=torch.bfloat16, device=dev)
    act.copy_(x0.reshape(-1)[: act.numel()])

    def step_ms(M, choice):
        def one_step():
            src = act
            for lay in layers:
                for j, (sh, wq, sc, bi) in enumerate(lay):
                    v, s = choice[j]
                    binding.small_m_ptr(src.data_ptr(), wq.data_ptr(), sc.data_ptr(), bi.data_ptr(), M, sh.N, sh.K,
                                        bits, gs, outs[j].data_ptr(), binding.OUT_BF16, names.index(v), s, handle)
                    src = outs[j]
        try:
            with torch.cuda.stream(stream):
                one_step()
        except binding.QmmError:
            return float("inf")
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one_step()
        times = []
        with torch.cuda.stream(stream):
            g.replay()
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(args.steps):
                    g.replay()
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b) / args.steps)
        del g
        return float(np.median(times))

    out = open(args.out, "w")
    for M in w.ms:
        keys = [(M, sh.N, sh.K) for sh in w.shapes]
        if not all(k in cands for k in keys):
            continue
        choice = [cands[k][0] for k in keys]
        best = step_ms(M, choice)
        start = best
        for _ in range(args.passes):
            for j, k in enumerate(keys):
                for c in cands[k]:
                    if c == choice[j]:
                        continue
                    trial = list(choice)
                    trial[j] = c
                    t = step_ms(M, trial)
                    if t < best:
                        best, choice = t, trial
        for (m, N, K), (v, s) in zip(keys, choice):
            out.write(json.dumps({"M": m, "N": N, "K": K, "bits": bits, "gs": gs, "variant": v,
                                  "variant_id": names.index(v), "splits": s, "source": "chain",
                                  "step_ms": round(best, 4), "step_ms_isolated_choice": round(start, 4)}) + "\n")
        out.flush()
        print(json.dumps({"M": M, "step_ms": round(best, 4), "from": round(start, 4),
                          "choice": [f"{v}/{s}" for v, s in choice]}), flush=True)
    status = binding.device_status()
    print(json.dumps({"done": True, "device_status": status}))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
