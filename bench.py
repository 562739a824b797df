"""Benchmark of the small-M quantized matmul on GB300.

Default workload: M sweep on one 5120x5120 4-bit affine g64 layer.  One step
is the whole hot path over one batch of synthetic input: 16 calls, M = 1..16,
each reading the previous call's output as its activations (a dependent
chain, as decode is), each streaming a different copy of the weights so that
the copies in rotation (> 4x L2) keep every call's weights cold in HBM.  The
step is captured in a CUDA graph and replayed.

``value`` is weight+metadata GB/s over the timed steps: the bytes each call
must stream (N*K*bits/8 + 4*N*K/g), summed over the step's calls and over all
ranks, divided by the max-over-ranks step time.  ``e2e`` is the same metric
through the C ABI with every step's activations copied in from pinned host
memory and its outputs read back.

``--impl reference`` times the fp64 CPU oracle (the only reference that
exists for this path) on the host cores, on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import shutil
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from quantized_matmul_speculative_gb300 import synth, workloads  # noqa: E402
from quantized_matmul_speculative_gb300.tuning.ncu_summary import kernel_hash  # noqa: E402

METRIC = "weight GB/s and % of HBM peak per call vs M=1..16 (4-bit affine g64)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    f = ROOT / "profiles" / f"qmm_tma_{workload}.md"
    if not f.exists():
        return None
    text = f.read_text()
    mh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_hash():
        return None
    return float(mt.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = Path(os.environ.get("TMPDIR", "/tmp")) / f"qmm_clocks_{os.getpid()}.csv"

    def __enter__(self):
        if shutil.which("nvidia-smi"):
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path.exists():
            return None
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.path.read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        self.path.unlink(missing_ok=True)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ the workload
def make_m_sweep_problem():
    w = workloads.M_SWEEP
    sh = w.shapes[0]
    p = synth.make_problem(workloads.shape_seed(w, 0), sh.N, sh.K, w.bits, w.group_size)
    return w, sh, p


def cpu_oracle_sample(p: synth.Problem, rows: int, ms):
    """Time the fp64 oracle on the first `rows` weight rows for each M in `ms`;
    returns (weight+meta bytes processed, seconds)."""
    from oracle import oracle

    lib = oracle.load()
    q = np.ascontiguousarray(p.q[:rows])
    wq = lib.pack(q, p.bits)
    s = np.ascontiguousarray(p.scales[:rows])
    b = np.ascontiguousarray(p.biases[:rows])
    t0 = time.perf_counter()
    for M in ms:
        lib.qmm(p.x_rows(M), wq, s, b, p.bits, p.group_size)
    dt = time.perf_counter() - t0
    nbytes = len(ms) * workloads.call_bytes(rows, p.K, p.bits, p.group_size)
    return nbytes, dt


# ------------------------------------------------------------------ further reports
def graph_us_per_call(torch, stream, capture, n_calls, warm=3, reps=5):
    """Median us per call of a CUDA graph of n_calls calls (capture(i) issues
    call i), timed with events on `stream` over `reps` replays."""
    with torch.cuda.stream(stream):
        capture(0)  # eager: sets kernel attributes outside the capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_calls):
            capture(i)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / n_calls)
    del g
    return float(np.median(times))


def configs_report(torch, dev, stream, peak):
    """us per call and weight+metadata GB/s of every workload shape at the
    dispatcher's choice.  Calls rotate over weight copies whose total exceeds
    4x L2; every call waits for the previous one on the stream (the kernels
    wait for their predecessor before reading X)."""
    from quantized_matmul_speculative_gb300 import binding

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = stream.cuda_stream
    names = binding.variant_names()
    out = []
    plan = [(workloads.SINGLE_LAYER, None, None, (4,)),
            (workloads.DENSE_27B_LAYER, None, None, workloads.DENSE_27B_LAYER.ms)]
    plan += [(workloads.GROUP_BIT_SWEEP, b, g, (1, 4, 8, 16)) for b, g in workloads.GROUP_BIT_SWEEP.variants]
    plan.append((workloads.VERIFY_STEP, None, None, (1, 4, 8)))
    plan.append((workloads.INT8_AFFINE, None, None, (1, 4, 8, 16)))
    plan.append((workloads.QMV_WIDE_GATE_UP, None, None, (1, 2, 4, 8, 16)))
    for w, bits, gs, ms in plan:
        bits = bits or w.bits
        gs = gs or w.group_size
        for si, sh in enumerate(w.shapes):
            p = synth.make_problem(workloads.shape_seed(w, si, 0, bits, gs), sh.N, sh.K, bits, gs)
            cb = workloads.call_bytes(sh.N, sh.K, bits, gs)
            ncopy = max(2, int(np.ceil(4 * l2 / cb)) + 1)
            wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32))
            sc = torch.from_numpy(p.scales.view(np.float16))
            bi = torch.from_numpy(p.biases.view(np.float16))
            copies = [(wq.to(dev), sc.to(dev), bi.to(dev)) for _ in range(ncopy)]
            x = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
            y = torch.empty((16, sh.N), dtype=torch.bfloat16, device=dev)
            for M in ms:
                def capture(i, M=M):
                    wq_d, s_d, b_d = copies[i % ncopy]
                    binding.small_m_ptr(x.data_ptr(), wq_d.data_ptr(), s_d.data_ptr(), b_d.data_ptr(), M, sh.N,
                                        sh.K, bits, gs, y.data_ptr(), binding.OUT_BF16, -1, -1, handle)
                us = graph_us_per_call(torch, stream, capture, 64)
                v, sp = binding.select_variant(M, sh.N, sh.K, bits, gs)
                gbs = cb / (us * 1e-6) / 1e9
                out.append({"workload": w.name, "shape": f"{sh.name} {sh.N}x{sh.K}", "bits": bits, "group_size": gs,
                            "M": M, "us_per_call": round(us, 3), "weight_gbs": round(gbs, 1),
                            "frac_hbm": round(gbs / peak, 4), "variant": names[v], "splits": sp})
            del copies
            torch.cuda.empty_cache()
    return out


def verify_step_report(torch, dev, stream, peak, ms=tuple(range(1, 9)), steps=10):
    """The whole verify step: 36 layers x (QKV, O, gate+up, down), 4-bit g64,
    distinct weights per layer (3.9 GB), back to back on one stream.  Each
    projection reads the first M*K elements of the previous projection's
    output buffer as its activations (a real data dependency of the right
    size; the layer math between projections is not part of this op), and the
    next layer's QKV reads the down projection's output."""
    from quantized_matmul_speculative_gb300 import binding

    w = workloads.VERIFY_STEP
    handle = stream.cuda_stream
    bits, gs = w.bits, w.group_size
    mats = []
    for si, sh in enumerate(w.shapes):
        p = synth.make_problem(workloads.shape_seed(w, si), sh.N, sh.K, bits, gs)
        wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32)).to(dev)
        sc = torch.from_numpy(p.scales.view(np.float16)).to(dev)
        bi = torch.from_numpy(p.biases.view(np.float16)).to(dev)
        mats.append((sh, wq, sc, bi))
        if si == 0:
            x0 = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
    # distinct memory per layer (same values): every call streams its own weights from HBM
    layers = [[(sh, wq.clone(), sc.clone(), bi.clone()) for sh, wq, sc, bi in mats] for _ in range(w.layers)]
    del mats
    outs = [torch.empty((16 * sh.N,), dtype=torch.bfloat16, device=dev) for sh in w.shapes]
    act = torch.empty((16 * w.shapes[0].K,), dtype=torch.bfloat16, device=dev)
    act.copy_(x0.reshape(-1)[: act.numel()])
    step_bytes = w.layers * sum(workloads.call_bytes(sh.N, sh.K, bits, gs) for sh in w.shapes)
    res = []
    for M in ms:
        def one_step(M=M):
            src = act
            for lay in layers:
                for j, (sh, wq, sc, bi) in enumerate(lay):
                    binding.small_m_ptr(src.data_ptr(), wq.data_ptr(), sc.data_ptr(), bi.data_ptr(), M, sh.N, sh.K,
                                        bits, gs, outs[j].data_ptr(), binding.OUT_BF16, -1, -1, handle)
                    src = outs[j]
            # the next step's first layer reads the last down projection's output
        with torch.cuda.stream(stream):
            one_step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one_step()
        times = []
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                g.replay()
            b.record(stream)
            b.synchronize()
        ms_step = a.elapsed_time(b) / steps
        gbs = step_bytes / (ms_step * 1e-3) / 1e9
        res.append({"M": M, "steps_per_s": round(1e3 / ms_step, 1), "ms_per_step": round(ms_step, 4),
                    "weight_gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)})
        del g
    del layers
    torch.cuda.empty_cache()
    return {"workload": w.name, "layers": w.layers, "calls_per_step": 4 * w.layers, "bytes_per_step": step_bytes,
            "per_m": res, "chain": "each projection reads the first M*K elements of the previous output"}


def residual_report(torch, dev, stream, ms=(1, 8, 16)):
    """The fused residual add on the 5120x5120 layer at the dispatcher's choice:
    us per call without a residual, with a separate residual buffer, and in
    place (R is Y), bf16.  Same chains as configs_report."""
    from quantized_matmul_speculative_gb300 import binding

    w = workloads.M_SWEEP
    sh = w.shapes[0]
    bits, gs = w.bits, w.group_size
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = stream.cuda_stream
    p = synth.make_problem(workloads.shape_seed(w, 0), sh.N, sh.K, bits, gs)
    cb = workloads.call_bytes(sh.N, sh.K, bits, gs)
    ncopy = max(2, int(np.ceil(4 * l2 / cb)) + 1)
    wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32))
    sc = torch.from_numpy(p.scales.view(np.float16))
    bi = torch.from_numpy(p.biases.view(np.float16))
    copies = [(wq.to(dev), sc.to(dev), bi.to(dev)) for _ in range(ncopy)]
    x = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((16, sh.N), dtype=torch.bfloat16, device=dev)
    r = torch.from_numpy(synth.make_residual(1, 16, sh.N).view(np.int16)).to(dev).view(torch.bfloat16)
    res = []
    for M in ms:
        row = {"M": M}
        for mode in ("plain", "residual", "in_place"):
            def capture(i, M=M, mode=mode):
                wq_d, s_d, b_d = copies[i % ncopy]
                args = (x.data_ptr(), wq_d.data_ptr(), s_d.data_ptr(), b_d.data_ptr())
                if mode == "plain":
                    binding.small_m_ptr(*args, M, sh.N, sh.K, bits, gs, y.data_ptr(), binding.OUT_BF16, -1, -1,
                                        handle)
                else:
                    rp = r.data_ptr() if mode == "residual" else y.data_ptr()
                    binding.small_m_residual_ptr(*args, rp, M, sh.N, sh.K, bits, gs, y.data_ptr(), binding.OUT_BF16,
                                                 -1, -1, handle)
            row[f"us_{mode}"] = round(graph_us_per_call(torch, stream, capture, 64), 3)
        res.append(row)
    del copies
    torch.cuda.empty_cache()
    return {"op": "fused residual add Y = R + X W^T, 5120x5120 4-bit g64, bf16", "per_m": res}


def moe_report(torch, dev, stream, peak):
    """The gathered (MoE) form on a 128-expert top-8 gate+up stack at T = 1, 2,
    4, 8 verify tokens: us per call, and GB/s over the bytes of the experts in
    the routing's union (each streamed once per call).  Calls rotate over
    copies of the whole stack so that every call reads cold HBM."""
    from quantized_matmul_speculative_gb300 import binding

    w = workloads.MOE_GATE_UP
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = stream.cuda_stream
    mp = synth.make_moe(w.seed, w.E, w.N, w.K, w.bits, w.group_size, max(w.ts), w.k)
    wq = torch.from_numpy(binding.pack(mp.q.reshape(w.E * w.N, w.K), w.bits).view(np.int32)).to(dev)
    sc = torch.from_numpy(mp.scales.view(np.float16)).to(dev)
    bi = torch.from_numpy(mp.biases.view(np.float16)).to(dev)
    smallest = workloads.moe_union_bytes(w, mp.experts[:min(w.ts)])
    ncopy = max(2, int(np.ceil(4 * l2 / smallest)) + 1)
    copies = [(wq, sc, bi)] + [(wq.clone(), sc.clone(), bi.clone()) for _ in range(ncopy - 1)]
    x = torch.from_numpy(mp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((max(w.ts) * w.k, w.N), dtype=torch.bfloat16, device=dev)
    res = []
    for T in w.ts:
        experts = mp.experts[:T]
        lhs = torch.from_numpy(np.repeat(np.arange(T, dtype=np.int32), w.k)).to(dev)
        rhs = torch.from_numpy(np.ascontiguousarray(experts.reshape(-1))).to(dev)
        ub = workloads.moe_union_bytes(w, experts)

        def capture(i, T=T, lhs=lhs, rhs=rhs, v=-1):
            wq_d, s_d, b_d = copies[i % ncopy]
            binding.gather_small_m_ptr(x.data_ptr(), wq_d.data_ptr(), s_d.data_ptr(), b_d.data_ptr(), lhs.data_ptr(),
                                       rhs.data_ptr(), T * w.k, T, w.E, w.N, w.K, w.bits, w.group_size, y.data_ptr(),
                                       binding.OUT_BF16, v, -1, handle)
        us = graph_us_per_call(torch, stream, capture, 32)
        tma = binding.variant_names().index("tma_w8_2cta")
        us_tma = graph_us_per_call(torch, stream, lambda i, T=T, lhs=lhs, rhs=rhs: capture(i, T, lhs, rhs, tma), 32)
        mma = binding.variant_names().index("mma_r2_wn2_wk4")
        us_mma = graph_us_per_call(torch, stream, lambda i, T=T, lhs=lhs, rhs=rhs: capture(i, T, lhs, rhs, mma), 32)
        gbs = ub / (us * 1e-6) / 1e9
        res.append({"T": T, "entries": T * w.k, "experts_in_union": int(len(np.unique(experts))),
                    "union_bytes": ub, "us_per_call": round(us, 3), "union_gbs": round(gbs, 1),
                    "frac_hbm": round(gbs / peak, 4), "us_per_call_tma_w8_2cta": round(us_tma, 3),
                    "us_per_call_mma_r2_wn2_wk4": round(us_mma, 3)})
    del copies, wq, sc, bi
    torch.cuda.empty_cache()
    return {"workload": w.name, "per_t": res,
            "note": "gathered form at the library's choice (warp-owned family), and forced onto tma_w8_2cta "
                    "and mma_r2_wn2_wk4; bytes = distinct experts of the routing x expert bytes"}


def mx_report(torch, dev, stream, peak, ms=(1, 8, 16)):
    """Microscaling fp modes on the 5120x5120 layer at the library's choice: us
    per call and GB/s over codes + scale bytes; same chains as configs_report."""
    from quantized_matmul_speculative_gb300 import binding

    N = K = 5120
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    handle = stream.cuda_stream
    out = []
    for fmt, bits, g in (("mxfp4", 4, 32), ("mxfp8", 8, 32), ("nvfp4", 4, 16)):
        q, sc = synth.make_mx(9000 + bits + g, N, K, fmt)
        cb = N * K * bits // 8 + N * K // g
        ncopy = max(2, int(np.ceil(4 * l2 / cb)) + 1)
        wq = torch.from_numpy(binding.pack(q, bits).view(np.int32)).to(dev)
        s8 = torch.from_numpy(sc).to(dev)
        copies = [(wq, s8)] + [(wq.clone(), s8.clone()) for _ in range(ncopy - 1)]
        x = torch.from_numpy(synth.make_x(9000, K).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty((16, N), dtype=torch.bfloat16, device=dev)
        f = binding.MX_FORMATS[fmt][0]
        for M in ms:
            def capture(i, M=M):
                wq_d, s_d = copies[i % ncopy]
                rc = binding.lib().qmm_small_m_mx(x.data_ptr(), wq_d.data_ptr(), s_d.data_ptr(), M, N, K, f,
                                                  y.data_ptr(), binding.OUT_BF16, -1, -1, handle)
                assert rc == 0, rc
            us = graph_us_per_call(torch, stream, capture, 64)
            gbs = cb / (us * 1e-6) / 1e9
            out.append({"format": fmt, "M": M, "bytes_per_call": cb, "us_per_call": round(us, 3),
                        "gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)})
        del copies, wq, s8
        torch.cuda.empty_cache()
    return {"shape": "5120x5120", "per_m": out,
            "note": "library's choice (warp-owned family); one scale byte per 32 codes (E8M0) or per 16 "
                    "(nvfp4: E4M3), no bias"}


def dense_control(torch, dev, stream, ms=(1, 8, 16)):
    """bf16 dense torch.matmul (cuBLAS) on the 5120x5120 layer, for scale only:
    the dense bf16 weights are 4x the bytes of the 4-bit ones."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    N = K = 5120
    ncopy = max(2, int(np.ceil(4 * l2 / (2 * N * K))) + 1)
    g = torch.Generator(device="cpu").manual_seed(7)
    wd = torch.randn((N, K), generator=g).to(torch.bfloat16)
    copies = [wd.to(dev) for _ in range(ncopy)]
    x = torch.randn((16, K), generator=g).to(torch.bfloat16).to(dev)
    y = torch.empty((16, N), dtype=torch.bfloat16, device=dev)
    res = []
    for M in ms:
        def capture(i, M=M):
            torch.matmul(x[:M], copies[i % ncopy].t(), out=y[:M])
        us = graph_us_per_call(torch, stream, capture, 32)
        res.append({"M": M, "us_per_call": round(us, 3), "weight_gbs": round(2 * N * K / (us * 1e-6) / 1e9, 1)})
    del copies
    torch.cuda.empty_cache()
    return {"op": "torch.matmul bf16 dense, 5120x5120", "per_m": res,
            "note": "library call (cuBLAS), for scale only; 2 bytes per weight"}


def run_reference(args, world, rank):
    """The oracle arm: host cores, a bounded sample of the same workload per step.

    The rows per step are sized from a short calibration so that warm-up plus
    the timed steps take about ``--ref-budget`` seconds of CPU work."""
    if rank != 0:
        return 0
    w, sh, p = make_m_sweep_problem()
    ms = list(w.ms)
    nb, dt = cpu_oracle_sample(p, 16, ms)
    per_row = dt / 16
    rows = int(args.ref_budget / max(1, args.steps + args.warmup) / per_row)
    rows = max(1, min(sh.N, rows))
    for _ in range(args.warmup):
        cpu_oracle_sample(p, rows, ms)
    total_b, total_t = 0, 0.0
    for _ in range(args.steps):
        nb, dt = cpu_oracle_sample(p, rows, ms)
        total_b += nb
        total_t += dt
    value = total_b / total_t / 1e9
    sample = (f"each step: M=1..16 over the first {rows} of {sh.N} weight rows of the "
              f"{sh.N}x{sh.K} 4-bit g64 layer, fp64 oracle, 1 thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "N": sh.N, "K": sh.K, "bits": w.bits,
                                        "group_size": w.group_size, "M": "1..16", "rows_sampled": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class StepGraphs:
    """CUDA graphs of the bench step, so that exactly K steps can be replayed.

    A graph of `reps` consecutive steps (the copy index advancing every call,
    enough steps to touch every weight copy) is replayed K // reps times, then a
    graph of K % reps steps once.  Graphs are captured on first use."""

    def __init__(self, torch, stream, issue_step, reps):
        self.torch, self.stream, self.issue_step, self.reps = torch, stream, issue_step, reps
        self.graphs = {}

    def _graph(self, n):
        if n not in self.graphs:
            g = self.torch.cuda.CUDAGraph()
            with self.torch.cuda.graph(g, stream=self.stream):
                for s in range(n):
                    self.issue_step(s)
            self.graphs[n] = g
        return self.graphs[n]

    def run(self, steps):
        """Enqueue exactly `steps` steps on the stream (graphs captured beforehand by prepare())."""
        full, rem = divmod(steps, self.reps)
        with self.torch.cuda.stream(self.stream):
            for _ in range(full):
                self.graphs[self.reps].replay()
            if rem:
                self.graphs[rem].replay()

    def prepare(self, *counts):
        for steps in counts:
            full, rem = divmod(steps, self.reps)
            if full:
                self._graph(self.reps)
            if rem:
                self._graph(rem)
        self.stream.synchronize()

    def release(self):
        self.graphs.clear()


def headline_line(*, value, world, steps, warmup, ms_per_step, workload, shape, ncopy, copy_mb, l2_mb, roofline,
                  per_m, e2e, cpu, launches, clocks):
    """The bench's last stdout line: compact (the driver keeps the tail of
    stdout), every extra report goes out on earlier lines."""
    N, K, bits, gs = shape
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "N": N, "K": K, "bits": bits, "group_size": gs, "M": "1..16",
                   "chain": "dependent", "l2": f"{ncopy} weight copies, {copy_mb:.0f} MB > L2 {l2_mb:.0f} MB",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "per_m_us": [round(r["us_per_call"], 2) for r in per_m],
        "per_m_frac": [round(r["frac_hbm"], 3) for r in per_m],
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clocks,
    }


def emit(report: str, body):
    """One extra report as its own JSON line (before the headline)."""
    print(json.dumps({"report": report, **body}), flush=True)


def per_m_report(torch, stream, call, ms, call_b, peak, ncopy, names, select):
    """us per call at each M: a graph of 64 chained calls at one M over `ncopy`
    rotating weight copies (cold HBM when their total exceeds L2; one copy:
    L2-warm), median of 5 replays."""
    rows = []
    for M in ms:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(64):
                call(M, i % ncopy, i % 2)
        times = []
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            for _ in range(5):
                a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b2.record(stream)
                b2.synchronize()
                times.append(a.elapsed_time(b2) * 1e3 / 64)
        del g
        us = float(np.median(times))
        gbs = call_b / (us * 1e-6) / 1e9
        variant, splits = select(M)
        rows.append({"M": M, "us_per_call": round(us, 3), "weight_gbs": round(gbs, 1),
                     "frac_hbm": round(gbs / peak, 4), "variant": names[variant], "splits": splits,
                     "spread_us": round(max(times) - min(times), 3)})
    return rows


def run_ours(args, world, rank, local):
    import torch

    from quantized_matmul_speculative_gb300 import binding, build

    build.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w, sh, p = make_m_sweep_problem()
    N, K, bits, gs = sh.N, sh.K, w.bits, w.group_size
    ms = list(w.ms)
    call_b = workloads.call_bytes(N, K, bits, gs)
    names = binding.variant_names()

    # weights: distinct copies whose total exceeds 4x L2, so each call reads cold HBM
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ncopy = max(args.min_copies, int(np.ceil(4 * l2 / call_b)) + 1)
    wq_h = torch.from_numpy(binding.pack(p.q, bits).view(np.int32))
    s_h = torch.from_numpy(p.scales.view(np.float16))
    b_h = torch.from_numpy(p.biases.view(np.float16))
    copies = [(wq_h.to(dev), s_h.to(dev), b_h.to(dev)) for _ in range(ncopy)]
    x0 = torch.from_numpy(p.x.view(np.int16)).to(dev).view(torch.bfloat16)
    bufs = [x0.clone(), torch.empty_like(x0)]
    stream = torch.cuda.Stream(dev)
    handle = stream.cuda_stream

    def launch(M, ci, xb, yb):
        wq, s, b = copies[ci % ncopy]
        binding.small_m_ptr(xb.data_ptr(), wq.data_ptr(), s.data_ptr(), b.data_ptr(), M, N, K, bits, gs,
                            yb.data_ptr(), binding.OUT_BF16, -1, -1, handle)

    def call(M, ci, parity):  # the chain ping-pongs between two activation buffers
        launch(M, ci, bufs[parity], bufs[parity ^ 1])

    calls_per_step = len(ms)
    reps = max(1, int(np.ceil(ncopy / calls_per_step)))  # steps until every copy has been read

    def issue_step(s):
        for j, M in enumerate(ms):
            ci = s * calls_per_step + j
            call(M, ci, ci % 2)

    with torch.cuda.stream(stream):
        issue_step(0)  # eager warm-up: kernel attributes, module load, tensor maps
        issue_step(1)
    stream.synchronize()
    graphs = StepGraphs(torch, stream, issue_step, reps)
    graphs.prepare(args.warmup, args.steps)

    # timed region: exactly --steps steps after exactly --warmup steps
    graphs.run(args.warmup)
    stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        start.record(stream)
        graphs.run(args.steps)
        end.record(stream)
        end.synchronize()
        torch.cuda.synchronize(dev)
        barrier(world)
    graphs.release()
    ms_total = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_per_step = ms_total / args.steps
    step_bytes = calls_per_step * call_b
    value = world * step_bytes * args.steps / (ms_total * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    clk = clocks.summary()

    def select(M):
        return binding.select_variant(M, N, K, bits, gs)

    per_m = per_m_report(torch, stream, call, ms, call_b, peak, ncopy, names, select)
    per_m_warm = per_m_report(torch, stream, call, ms, call_b, peak, 1, names, select)
    kernels = sorted({"qmm_own_kernel" if "_own_" in r["variant"] else
                      "qmm_tma_kernel" if r["variant"].startswith("tma") else "qmm_mma_kernel" for r in per_m})
    if rank == 0:
        emit("per_m_cold", {"workload": w.name, "per_m": per_m,
                            "note": f"64 chained calls at one M over {ncopy} rotating weight copies, median of 5"})
        emit("per_m_l2_warm", {"workload": w.name, "per_m": per_m_warm,
                               "note": "L2-WARM: the same chain on one weight copy (14.7 MB stays in L2); "
                                       "not the roofline figure"})

    # e2e: the public API with host buffers.  Every step copies the activations
    # of its 16 calls in from pinned host memory (one copy), runs the calls
    # (each on its own rows), and reads all their outputs back (one copy); the
    # steps are graph-replayed so that the timing is the device's.
    rows = sum(ms)
    x_host = torch.empty((rows, K), dtype=torch.bfloat16).pin_memory()
    r0 = 0
    for M in ms:
        x_host[r0:r0 + M].copy_(torch.from_numpy(p.x[:M].view(np.int16)).view(torch.bfloat16))
        r0 += M
    y_host = torch.empty((rows, N), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((rows, K), dtype=torch.bfloat16, device=dev)
    yd = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
    h2d = 2 * rows * K
    d2h = 2 * rows * N

    def e2e_step(s):
        xd.copy_(x_host, non_blocking=True)
        r = 0
        for j, M in enumerate(ms):
            launch(M, s * calls_per_step + j, xd[r:r + M], yd[r:r + M])
            r += M
        y_host.copy_(yd, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step(0)
    stream.synchronize()
    e2e_graphs = StepGraphs(torch, stream, e2e_step, reps)
    e2e_graphs.prepare(args.warmup, args.steps)
    e2e_graphs.run(args.warmup)
    stream.synchronize()
    barrier(world)
    a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_graphs.run(args.steps)
    b2.record(stream)
    b2.synchronize()
    e2e_graphs.release()
    e2e_ms = max_over_ranks(a.elapsed_time(b2), world, dev)
    e2e_value = world * step_bytes * args.steps / (e2e_ms * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        nb, dt = cpu_oracle_sample(p, args.cpu_rows, ms)
        cpu = {"value": round(nb / dt / 1e9, 5), "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(),
               "kind": "oracle",
               "sample": f"M=1..16, rows 0..{args.cpu_rows - 1} of {N}, 1 thread, {dt:.1f} s"}

    if rank == 0 and not args.no_extra:
        emit("configs", {"per_config": configs_report(torch, dev, stream, peak)})
        emit("verify_step", verify_step_report(torch, dev, stream, peak))
        emit("controls", dense_control(torch, dev, stream))
        emit("residual", residual_report(torch, dev, stream))
        emit("moe", moe_report(torch, dev, stream, peak))
        emit("mx", mx_report(torch, dev, stream, peak))

    if rank == 0:
        achieved = value / world
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": profiled_traffic(w.name),
                    "peak_source": "measured" if peak_kind == "measured" else "fallback",
                    "kernel": ",".join(kernels)}
        e2e = {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        clocks_short = None if clk is None else {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                                                  "reasons": clk["reasons"]}
        line = headline_line(value=value, world=world, steps=args.steps, warmup=args.warmup,
                             ms_per_step=ms_per_step, workload=w.name, shape=(N, K, bits, gs), ncopy=ncopy,
                             copy_mb=ncopy * call_b / 1e6, l2_mb=l2 / 1e6, roofline=roofline, per_m=per_m,
                             e2e=e2e, cpu=cpu, launches=args.steps * calls_per_step, clocks=clocks_short)
        print(json.dumps(line, separators=(",", ":")), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--min-copies", type=int, default=36)
    ap.add_argument("--cpu-rows", type=int, default=5120)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-config, verify-step and dense-control reports")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
    world, rank, local = dist_setup(args)
    try:
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
