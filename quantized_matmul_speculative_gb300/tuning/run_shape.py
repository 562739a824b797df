"""Run one shape through the C ABI a few times (for profiler captures).

    python -m quantized_matmul_speculative_gb300.tuning.run_shape --N 34816 --K 5120 --M 1 [--calls 3]
        [--bits 4] [--group 64] [--variant NAME --splits S]
        [--mode plain | gather --E 128 --T 4 --topk 8 | mx --fmt mxfp4 | ggml --kind q4_0]

Synthetic inputs from synth (make_problem, make_moe, make_mx,
make_ggml_blocks); the dispatcher's choice unless a variant is forced.  The
gathered mode routes T tokens to topk experts of an E-matrix stack (M = T); the
ggml mode converts the blocks on the device once per call before the product.
Prints the choice, the device status word and a checksum.
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
    ap.add_argument("--mode", choices=("plain", "gather", "mx", "ggml"), default="plain")
    ap.add_argument("--E", type=int, default=128)
    ap.add_argument("--T", type=int, default=4)
    ap.add_argument("--topk", type=int, default=8)
    ap.add_argument("--fmt", choices=sorted(binding.MX_FORMATS), default="mxfp4")
    ap.add_argument("--kind", choices=sorted(binding.GGML_TYPES), default="q4_0")
    args = ap.parse_args()
    import torch

    build.build()
    binding.lib()
    names = binding.variant_names()
    v = names.index(args.variant) if args.variant else -1
    M = args.T if args.mode == "gather" else args.M
    info = {"mode": args.mode, "N": args.N, "K": args.K, "M": M}

    def cuda_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    if args.mode == "gather":
        mp = synth.make_moe(args.seed, args.E, args.N, args.K, args.bits, args.group, args.T, args.topk)
        wq = torch.from_numpy(binding.pack(mp.q.reshape(args.E * args.N, args.K), args.bits).view(np.int32))
        wq = wq.reshape(args.E, args.N, -1).cuda()
        s = torch.from_numpy(mp.scales.view(np.float16)).cuda()
        b = torch.from_numpy(mp.biases.view(np.float16)).cuda()
        x = cuda_bf16(mp.x[:args.T])
        lhs, rhs = (torch.from_numpy(a).cuda() for a in mp.lists())
        info.update(E=args.E, topk=args.topk, union=int(len(np.unique(mp.experts))))

        def call():
            return binding.gather_small_m(x, wq, s, b, lhs, rhs, args.bits, args.group, variant=v, splits=args.splits)
    elif args.mode == "mx":
        q, sc = synth.make_mx(args.seed, args.N, args.K, args.fmt)
        bits = binding.MX_FORMATS[args.fmt][1]
        wq = torch.from_numpy(binding.pack(q, bits).view(np.int32)).cuda()
        s = torch.from_numpy(sc).cuda()
        x = cuda_bf16(synth.make_x(args.seed, args.K)[:M])
        info.update(fmt=args.fmt)

        def call():
            return binding.small_m_mx(x, wq, s, args.fmt, variant=v, splits=args.splits)
    elif args.mode == "ggml":
        blocks = torch.from_numpy(synth.make_ggml_blocks(args.seed, args.N, args.K, args.kind).reshape(-1)).cuda()
        x = cuda_bf16(synth.make_x(args.seed, args.K)[:M])
        info.update(kind=args.kind)

        def call():
            wq, s, b, bits = binding.from_ggml(args.kind, blocks, args.N, args.K)
            return binding.small_m(x, wq, s, b, bits, 32, variant=v, splits=args.splits)
    else:
        p = synth.make_problem(args.seed, args.N, args.K, args.bits, args.group)
        wq = torch.from_numpy(binding.pack(p.q, args.bits).view(np.int32)).cuda()
        s = torch.from_numpy(p.scales.view(np.float16)).cuda()
        b = torch.from_numpy(p.biases.view(np.float16)).cuda()
        x = cuda_bf16(p.x[:M])
        if v < 0:
            chosen, sp = binding.select_variant(M, args.N, args.K, args.bits, args.group)
            info.update(variant=names[chosen], splits=sp)

        def call():
            return binding.small_m(x, wq, s, b, args.bits, args.group, variant=v, splits=args.splits)

    if v >= 0:
        info.update(variant=names[v], splits=args.splits)
    y = None
    for _ in range(args.calls):
        y = call()
    torch.cuda.synchronize()
    status = binding.device_status()
    info.update(checksum=float(y.float().abs().sum()), device_status=status)
    print(json.dumps(info))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
