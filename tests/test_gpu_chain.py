"""Dependent chains of calls on one stream, the way a verify step issues them:
every call reads the previous call's output as its activations.  Each kernel
starts streaming its weights before the predecessor has finished (programmatic
dependent launch), so these tests check that no activation is read before the
predecessor wrote it and no output is written before the predecessor read the
buffer.

* Every step of a chain with its own output buffer is checked on the
  activations that step actually read: the same call with fp32 output, made
  alone afterwards, must meet the library's bound
  |y - y_ref| <= 2e-3 * sum_k |x w| (+ |r|) + 1e-5 against the oracle, and the
  chain's bf16 output must be exactly its round to nearest even.  The row
  count changes from call to call, so the dispatcher's choices mix the kernel
  families inside one chain; each family is also forced for a whole chain.
* A ping-pong chain (two buffers, each call overwriting the buffer its
  predecessor read) gives bit-identical buffers whether the calls are
  synchronized one by one, issued back to back, or replayed from a CUDA graph.
"""
import numpy as np
import pytest

from oracle import oracle
from qmm_harness import assert_within, check, to_f64
from quantized_matmul_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu

M_SEQ = [1, 5, 16, 8, 3, 12, 2, 9]
SHAPES = [(2048, 4, 64), (5120, 4, 64), (1024, 2, 32), (2048, 8, 64)]  # (N = K, bits, group size)
FAMILIES = ["mma_r2_wn2_wk4", "tma_w8_2cta", "tma_own_w8_d2_2cta"]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_matmul_speculative_gb300 import build

    build.build()
    binding.lib()
    return torch


@pytest.fixture(autouse=True)
def no_device_faults(torch_cuda):
    binding.device_status(clear=True)
    yield
    torch_cuda.cuda.synchronize()
    assert binding.device_status(clear=True) == 0


class Layers:
    """len(M_SEQ) square layers with distinct weights, resident on the GPU."""

    def __init__(self, torch, n, bits, gs):
        self.n, self.bits, self.gs = n, bits, gs
        self.problems = [synth.make_problem(9100 + 17 * i + n + bits + gs, n, n, bits, gs) for i in range(len(M_SEQ))]
        self.dev = []
        for p in self.problems:
            wq = torch.from_numpy(binding.pack(p.q, bits).view(np.int32)).cuda()
            s = torch.from_numpy(p.scales.view(np.float16)).cuda()
            b = torch.from_numpy(p.biases.view(np.float16)).cuda()
            self.dev.append((wq, s, b))
        x0 = self.problems[0].x
        self.x0 = torch.from_numpy(x0.view(np.int16)).cuda().view(torch.bfloat16)

    def call(self, i, x, y, variant, residual=False):
        wq, s, b = self.dev[i]
        r = None
        if residual:  # R = X, widened exactly when the output is fp32
            r = x if y.dtype == x.dtype else x.to(y.dtype)
        binding.small_m(x, wq, s, b, self.bits, self.gs, out=y, variant=variant, residual=r)

    def plans(self, torch, variant):
        """True if the variant takes every row count of the chain on this shape."""
        if variant < 0:
            return True
        y = torch.empty((16, self.n), dtype=torch.bfloat16, device="cuda")
        for m in sorted(set(M_SEQ)):
            try:
                self.call(0, self.x0[:m], y[:m], variant)
            except binding.QmmError as e:
                if e.status == 3:
                    return False
                raise
        torch.cuda.synchronize()
        return True


def bits_of(t):
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def chain_variants():
    names = binding.variant_names()
    return [("default", -1)] + [(f, names.index(f)) for f in FAMILIES]


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("n,bits,gs", SHAPES)
def test_chain_each_step_against_oracle(torch_cuda, n, bits, gs, residual):
    torch = torch_cuda
    layers = Layers(torch, n, bits, gs)
    ol = oracle.load()
    wq_host = [ol.pack(p.q, bits) for p in layers.problems]
    ran = 0
    for name, v in chain_variants():
        if not layers.plans(torch, v):
            continue
        ran += 1
        # buffer i feeds call i; rows a call does not write keep the first activations
        bufs = [layers.x0.clone() for _ in range(len(M_SEQ) + 1)]
        torch.cuda.synchronize()
        for i, m in enumerate(M_SEQ):
            layers.call(i, bufs[i][:m], bufs[i + 1][:m], v, residual)
        torch.cuda.synchronize()
        x0 = bits_of(layers.x0)
        for i, m in enumerate(M_SEQ):
            p = layers.problems[i]
            x_in = bits_of(bufs[i])[:m]
            if residual:
                y_ref, a_ref = ol.qmm_residual(x_in, wq_host[i], p.scales, p.biases, x_in, bits, gs)
            else:
                y_ref, a_ref = ol.qmm(x_in, wq_host[i], p.scales, p.biases, bits, gs)
            what = f"{name} step {i} M={m}"
            y16 = bufs[i + 1][:m]
            y32 = torch.empty((m, n), dtype=torch.float32, device="cuda")
            layers.call(i, bufs[i][:m], y32, v, residual)
            torch.cuda.synchronize()
            assert_within(to_f64(y32), y_ref, a_ref, what + " (fp32, alone)")
            check(y16, y_ref, a_ref, what)
            assert torch.equal(y16, y32.to(torch.bfloat16)), f"{what}: chain output is not RNE of the fp32 result"
            assert np.array_equal(bits_of(bufs[i + 1])[m:], x0[m:]), f"{name} step {i}: rows >= M written"
    assert ran >= 2, "fewer than two chain variants could plan this shape"


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("n,bits,gs", SHAPES[:2])
def test_ping_pong_chain_is_race_free(torch_cuda, n, bits, gs, residual):
    torch = torch_cuda
    layers = Layers(torch, n, bits, gs)
    for name, v in chain_variants():
        if not layers.plans(torch, v):
            continue
        buf = [torch.empty_like(layers.x0), torch.empty_like(layers.x0)]

        def reset():
            buf[0].copy_(layers.x0)
            buf[1].copy_(layers.x0)

        def chain(sync):
            for i, m in enumerate(M_SEQ):
                layers.call(i, buf[i % 2][:m], buf[(i + 1) % 2][:m], v, residual)
                if sync:
                    torch.cuda.synchronize()

        reset()
        torch.cuda.synchronize()
        chain(sync=True)
        ref = [b.clone() for b in buf]
        for _ in range(3):
            reset()
            chain(sync=False)
            torch.cuda.synchronize()
            for k in range(2):
                assert torch.equal(buf[k].view(torch.int16), ref[k].view(torch.int16)), f"{name} back to back"

        stream = torch.cuda.Stream()
        reset()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            chain(sync=False)
        for _ in range(3):
            reset()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            for k in range(2):
                assert torch.equal(buf[k].view(torch.int16), ref[k].view(torch.int16)), f"{name} graph replay"
