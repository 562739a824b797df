"""Run one shape through the C ABI a few times (for profiler captures).

    python -m quantized_matmul_speculative_gb300.tuning.run_shape --N 34816 --K 5120 --M 1 [--calls 3]
        [--bits 4] [--group 64] [--variant NAME --splits S]

Synthetic inputs from synth.make_problem; the dispatcher's choice unless a
variant is forced.  Prints the choice, the device status word and a checksum.
"""
from __future__ import annotations

import argparse
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

from quantized_matmul_speculative_gb300 import binding, build, synth  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--bits", type=int, default=4)
    ap.add_argument("--group", type=int, default=64)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--variant", default=None)
    ap.add_argument("--splits", type=int, default=-1)
    ap.add_argument("--seed", type=int, default=1)
    args = ap.parse_args()
    import torch

    build.build()
    binding.lib()
    p = synth.make_problem(args.seed, args.N, args.K, args.bits, args.group)
    wq = torch.from_numpy(binding.pack(p.q, args.bits).view(np.int32)).cuda()
    s = torch.from_numpy(p.scales.view(np.float16)).cuda()
    b = torch.from_numpy(p.biases.view(np.float16)).cuda()
    x = torch.from_numpy(p.x.view(np.int16)).cuda().view(torch.bfloat16)[: args.M].contiguous()
    names = binding.variant_names()
    v = names.index(args.variant) if args.variant else -1
    y = None
    for _ in range(args.calls):
        y = binding.small_m(x, wq, s, b, args.bits, args.group, variant=v, splits=args.splits)
    torch.cuda.synchronize()
    chosen, splits = (v, args.splits) if v >= 0 else binding.select_variant(args.M, args.N, args.K, args.bits,
                                                                            args.group)
    status = binding.device_status()
    print(json.dumps({"N": args.N, "K": args.K, "M": args.M, "variant": names[chosen], "splits": splits,
                      "checksum": float(y.float().abs().sum()), "device_status": status}))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
