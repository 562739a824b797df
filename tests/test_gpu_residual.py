"""GPU parity of the fused residual add, Y = R + X . dequant(W)^T
(qmm_small_m_residual), against the oracle's residual product.

The bound is the library's acceptance bound with |r| added to the scale:
|y - y_ref| <= 2e-3 * (|r| + sum_k |x w|) + 1e-5.  The oracle returns that
scale as its A.  The residual is added to the fp32 result before the single
rounding to Y's dtype.  That rounding is not inside the bound when R dominates
the sum (half a bf16 ulp is up to 2^-8 |y|, and |y| can be close to A), so a
bf16 output is held to the bound plus half a bf16 ulp, and checked bit for bit
as the round to nearest even of the fp32 output of the same variant with R
widened exactly to fp32.
"""
import numpy as np
import pytest

from oracle import oracle
from qmm_harness import DeviceProblem, OracleRef, assert_within, check, sample_positions, to_f64
from quantized_matmul_speculative_gb300 import binding, synth, workloads

pytestmark = pytest.mark.gpu


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


def residual_tensor(torch, r_np, f32: bool):
    if f32:
        return torch.from_numpy(np.ascontiguousarray(r_np)).cuda()
    return torch.from_numpy(np.ascontiguousarray(r_np).view(np.int16)).cuda().view(torch.bfloat16)


def run_residual(torch, dp, M, rt, out, v, s):
    try:
        return binding.small_m(dp.x[:M].contiguous(), dp.wq, dp.s, dp.b, dp.p.bits, dp.p.group_size, out=out,
                               out_dtype=out.dtype, variant=v, splits=s, residual=rt)
    except binding.QmmError as e:
        if e.status == 3:
            return None
        raise


@pytest.mark.parametrize("f32", [False, True], ids=["bf16", "f32"])
def test_residual_every_variant(torch_cuda, f32):
    """Several tiles with a ragged N tail, every variant, M = 1, 8, 9, 16, a
    separate residual buffer and the in-place form (R is Y)."""
    torch = torch_cuda
    N, K, bits, gs = 200, 512, 4, 64
    p = synth.make_problem(9400, N, K, bits, gs)
    dp = DeviceProblem(p)
    ol = oracle.load()
    wq_ref = ol.pack(p.q, bits)
    r_all = synth.make_residual(9400, 16, N, f32=f32)
    dt = torch.float32 if f32 else torch.bfloat16
    ran = set()
    for M in (1, 8, 9, 16):
        r = np.ascontiguousarray(r_all[:M])
        y_ref, a_ref = ol.qmm_residual(p.x_rows(M), wq_ref, p.scales, p.biases, r, bits, gs)
        for v in range(len(binding.variant_names())):
            for s in (1, 2):
                rt = residual_tensor(torch, r, f32)
                out = torch.empty((M, N), dtype=dt, device="cuda")
                y = run_residual(torch, dp, M, rt, out, v, s)
                if y is None:
                    continue
                ran.add(binding.variant_names()[v].split("_")[0])
                what = f"{binding.variant_names()[v]}/{s} M={M}"
                check(y, y_ref, a_ref, what)
                if not f32:  # the same call with fp32 output and R widened exactly
                    y32 = run_residual(torch, dp, M, rt.float(), torch.empty((M, N), dtype=torch.float32,
                                                                             device="cuda"), v, s)
                    assert_within(to_f64(y32), y_ref, a_ref, what + " f32 twin")
                    assert torch.equal(y, y32.to(torch.bfloat16)), f"{what}: bf16 is not RNE of the fp32 result"
                assert torch.equal(rt, residual_tensor(torch, r, f32)), f"{what}: R was modified"
                inplace = residual_tensor(torch, r, f32)
                run_residual(torch, dp, M, inplace, inplace, v, s)
                assert torch.equal(inplace, y), f"{what}: in-place result differs"
    assert {"mma", "tma"} <= ran


def test_residual_bench_shape_sampled(torch_cuda):
    """5120x5120 4-bit g64 through the dispatcher, M = 1, 8, 16, bf16 output:
    sampled outputs against the oracle's product plus R."""
    torch = torch_cuda
    w = workloads.M_SWEEP
    sh = w.shapes[0]
    p = synth.make_problem(workloads.shape_seed(w, 0), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    r_all = synth.make_residual(77, 16, sh.N)
    r64 = synth.bf16_bits_to_f32(r_all).astype(np.float64)
    for M in (1, 8, 16):
        rt = residual_tensor(torch, r_all[:M], False)
        y = binding.small_m(dp.x[:M].contiguous(), dp.wq, dp.s, dp.b, w.bits, w.group_size, residual=rt)
        ms, ns = sample_positions(M, sh.N, 256, seed=M)
        y_ref, a_ref = ref.sampled(M, ms, ns)
        check(y, r64[ms, ns] + y_ref, np.abs(r64[ms, ns]) + a_ref, f"M={M}", at=(ms, ns))


def test_residual_empty_sum_and_validation(torch_cuda):
    """K = 0 gives Y = R (copied, or untouched in place); a partly overlapping
    or missing residual is rejected before launch."""
    torch = torch_cuda
    x = torch.zeros((3, 0), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((5, 0), dtype=torch.int32, device="cuda")
    s = torch.zeros((5, 0), dtype=torch.float16, device="cuda")
    r = torch.arange(15, dtype=torch.float32, device="cuda").view(3, 5)
    y = torch.full((3, 5), 7.0, dtype=torch.float32, device="cuda")
    binding.small_m(x, wq, s, s, 4, 64, out=y, residual=r)
    torch.cuda.synchronize()
    assert torch.equal(y, r)
    binding.small_m(x, wq, s, s, 4, 64, out=r, residual=r)
    torch.cuda.synchronize()
    assert torch.equal(r, torch.arange(15, dtype=torch.float32, device="cuda").view(3, 5))

    p = synth.make_problem(9401, 64, 256, 4, 64)
    dp = DeviceProblem(p)
    buf = torch.full((2 * 64 + 8,), 3.0, dtype=torch.float32, device="cuda")
    yv = buf[:128]
    args = [dp.x.data_ptr(), dp.wq.data_ptr(), dp.s.data_ptr(), dp.b.data_ptr()]
    with pytest.raises(binding.QmmError) as ei:  # residual 4 elements into Y
        binding.small_m_residual_ptr(*args, buf.data_ptr() + 16, 2, 64, 256, 4, 64, yv.data_ptr(), binding.OUT_F32)
    assert ei.value.status == 2
    with pytest.raises(binding.QmmError) as ei:
        binding.small_m_residual_ptr(*args, 0, 2, 64, 256, 4, 64, yv.data_ptr(), binding.OUT_F32)
    assert ei.value.status == 1
    torch.cuda.synchronize()
    assert bool((buf == 3.0).all()), "a rejected call wrote to Y"
