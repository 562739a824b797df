"""The C ABI from several host threads at once: a fresh process (so that the
library's one-time initialization, the dispatch table, the planners' caches
and the kernels' shared-memory attributes are first touched concurrently)
starts six threads on a barrier, each issuing a different mix of calls
(plain, residual, gathered, microscaling, the warp-owned whole-tile metadata
path, forced variants) on its own stream.  Every result must be bit-identical
to the same call made afterwards from one thread, and the device status word
must stay clean."""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parents[1]

SCRIPT = textwrap.dedent('''
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    from quantized_matmul_speculative_gb300 import binding, build, synth

    build.build()
    names = binding.variant_names()

    def dev_problem(seed, n, k, bits, gs):
        p = synth.make_problem(seed, n, k, bits, gs)
        wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32)).cuda()
        s = torch.from_numpy(p.scales.view(np.float16)).cuda()
        b = torch.from_numpy(p.biases.view(np.float16)).cuda()
        x = torch.from_numpy(p.x.view(np.int16)).cuda().view(torch.bfloat16)
        return wq, s, b, x, bits, gs

    plain = [dev_problem(11, 5120, 5120, 4, 64), dev_problem(12, 15360, 3840, 4, 64),
             dev_problem(13, 2048, 2048, 8, 64), dev_problem(14, 200, 1920, 2, 32)]
    mp = synth.make_moe(15, 16, 256, 512, 4, 64, 4, 2)
    g_wq = torch.from_numpy(binding.pack(mp.q.reshape(16 * 256, 512), 4).view(np.int32)).reshape(16, 256, -1).cuda()
    g_s = torch.from_numpy(mp.scales.view(np.float16)).cuda()
    g_b = torch.from_numpy(mp.biases.view(np.float16)).cuda()
    g_x = torch.from_numpy(mp.x.view(np.int16)).cuda().view(torch.bfloat16)
    lhs, rhs = (torch.from_numpy(a).cuda() for a in mp.lists())
    q, sc = synth.make_mx(16, 2880, 2880, "mxfp4")
    mx_wq = torch.from_numpy(binding.pack(q, 4).view(np.int32)).cuda()
    mx_s = torch.from_numpy(sc).cuda()
    mx_x = torch.from_numpy(synth.make_x(16, 2880).view(np.int16)).cuda().view(torch.bfloat16)
    torch.cuda.synchronize()

    def calls():
        """(name, function(stream) -> output) for every call of the mix."""
        out = []
        for pi, (wq, s, b, x, bits, gs) in enumerate(plain):
            for m in (1, 5, 9, 16):
                out.append((f"plain{pi}-M{m}", lambda st, wq=wq, s=s, b=b, x=x, bits=bits, gs=gs, m=m:
                            binding.small_m(x[:m].contiguous(), wq, s, b, bits, gs, stream=st)))
            r = torch.ones((3, wq.shape[0]), dtype=torch.float32, device="cuda")
            out.append((f"residual{pi}", lambda st, wq=wq, s=s, b=b, x=x, bits=bits, gs=gs, r=r:
                        binding.small_m(x[:3].contiguous(), wq, s, b, bits, gs, out_dtype=torch.float32,
                                        residual=r, stream=st)))
        for v in ("mma_r2_wn2_wk4", "tma_own_w8_d2_2cta", "tma_w8_2cta"):
            wq, s, b, x, bits, gs = plain[0]
            out.append((f"forced-{v}", lambda st, v=v, wq=wq, s=s, b=b, x=x, bits=bits, gs=gs:
                        binding.small_m(x[:7].contiguous(), wq, s, b, bits, gs, variant=names.index(v), stream=st)))
        out.append(("gather", lambda st: binding.gather_small_m(g_x[:4].contiguous(), g_wq, g_s, g_b, lhs, rhs, 4, 64,
                                                                stream=st)))
        out.append(("mx", lambda st: binding.small_m_mx(mx_x[:6].contiguous(), mx_wq, mx_s, "mxfp4", stream=st)))
        return out

    mix = calls()
    nthreads = 6
    results = [dict() for _ in range(nthreads)]
    errors = []
    barrier = threading.Barrier(nthreads)

    def worker(t):
        try:
            st = torch.cuda.Stream()
            order = list(range(len(mix)))
            np.random.default_rng(t).shuffle(order)
            barrier.wait()
            with torch.cuda.stream(st):
                for rep in range(3):
                    for i in order:
                        name, f = mix[i]
                        results[t][(name, rep)] = f(st)
            st.synchronize()
        except Exception as e:  # reported below
            errors.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    reference = {name: f(torch.cuda.current_stream()) for name, f in mix}
    torch.cuda.synchronize()
    bad = [(t, key) for t in range(nthreads) for key, y in results[t].items()
           if not torch.equal(y, reference[key[0]])]
    assert not bad, bad[:5]
    status = binding.device_status(clear=True)
    assert status == 0, status
    print("threads ok", len(mix), "calls x", nthreads, "threads x 3")
''')


def test_concurrent_calls_from_threads():
    res = subprocess.run([sys.executable, "-c", f"ROOT = {str(ROOT)!r}\n" + SCRIPT], capture_output=True, text=True,
                         timeout=600, cwd=str(ROOT))
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "threads ok" in res.stdout
