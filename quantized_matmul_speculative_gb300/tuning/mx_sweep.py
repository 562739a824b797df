"""Time the microscaling modes (mxfp4, mxfp8, nvfp4) on the warp-owned
variants and cluster sizes, 5120x5120 and 8192x8192, M in {1, 4, 8, 9, 12, 16}
(or --ms): the evidence for qmm_small_m_mx's choices (make_table.py turns it
into the microscaling dispatch table).  Each measurement is a CUDA
graph of 48 calls over rotating weight copies (> 4x L2), median of 5 replays.
One JSON object per (shape, format, M) with the four fastest choices.

    python -m quantized_matmul_speculative_gb300.tuning.mx_sweep --out mx_sweep.jsonl
        [--shapes 2880x2880,5120x5120] [--with-mma] [--ms 1,2,4,8,16]

--shapes replaces the two square shapes (N x K); --with-mma times the mma
variants too.
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
    ap.add_argument("--out", required=True)
    ap.add_argument("--shapes", default="5120x5120,8192x8192")
    ap.add_argument("--with-mma", action="store_true")
    ap.add_argument("--ms", default="1,4,8,9,12,16")
    args = ap.parse_args()
    shapes = [tuple(int(v) for v in sh.split("x")) for sh in args.shapes.split(",")]
    import torch

    build.build()
    binding.lib()
    names = binding.variant_names()
    own = [i for i, n in enumerate(names) if n.startswith("tma_own") and not n.endswith("_half")]
    if args.with_mma:
        own += [i for i, n in enumerate(names) if n.startswith("mma")]
    st = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    out = open(args.out, "w")
    for N, K in shapes:
        for fmt, (f, bits, g) in binding.MX_FORMATS.items():
            q, sc = synth.make_mx(1, N, K, fmt)
            cb = N * K * bits // 8 + N * K // g
            nc = int(np.ceil(4 * l2 / cb)) + 1
            wq = torch.from_numpy(binding.pack(q, bits).view(np.int32)).cuda()
            s8 = torch.from_numpy(sc).cuda()
            copies = [(wq, s8)] + [(wq.clone(), s8.clone()) for _ in range(nc - 1)]
            x = torch.from_numpy(synth.make_x(1, K).view(np.int16)).cuda().view(torch.bfloat16)
            y = torch.empty((16, N), dtype=torch.bfloat16, device="cuda")
            for M in (int(m) for m in args.ms.split(",")):
                res = []
                for v in own:
                    for s in (1, 2, 4, 8):
                        def call(i, v=v, s=s, M=M):
                            wq_d, s_d = copies[i % nc]
                            return binding.lib().qmm_small_m_mx(x.data_ptr(), wq_d.data_ptr(), s_d.data_ptr(), M, N,
                                                                K, f, y.data_ptr(), binding.OUT_BF16, v, s,
                                                                st.cuda_stream)
                        with torch.cuda.stream(st):
                            if call(0) != 0:
                                continue
                        st.synchronize()
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=st):
                            for i in range(48):
                                call(i)
                        ts = []
                        with torch.cuda.stream(st):
                            graph.replay()
                            for _ in range(5):
                                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                                a.record(st)
                                graph.replay()
                                b.record(st)
                                b.synchronize()
                                ts.append(a.elapsed_time(b) * 1e3 / 48)
                        res.append((round(float(np.median(ts)), 3), names[v], s))
                        del graph
                res.sort()
                out.write(json.dumps({"N": N, "K": K, "format": fmt, "M": M, "best": res[:4]}) + "\n")
                out.flush()
            del copies
            torch.cuda.empty_cache()
    status = binding.device_status()
    print(json.dumps({"done": True, "device_status": status}))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
