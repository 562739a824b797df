"""GPU parity of the microscaling fp modes (qmm_small_m_mx): mxfp4 (E2M1) and
mxfp8 (E4M3) codes with E8M0 scales per 32, and nvfp4 (E2M1 codes with E4M3
scales per 16), against the oracle, with the
library's bound |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5 on the fp32 output.

The bf16 output is checked as the exact round-to-nearest-even of the fp32
output of the same variant: with E4M3's heavy-tailed weights one product can
dominate a row (|y| close to sum |x w|), and half a bf16 ulp (up to 2^-8 |y|)
then exceeds 2e-3 * sum |x w| by itself."""
import numpy as np
import pytest

from oracle import oracle
from qmm_harness import assert_within, sample_positions, to_f64
from quantized_matmul_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu

FORMATS = [("mxfp4", 4), ("mxfp8", 8), ("nvfp4", 4)]


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


def upload(torch, q, sc, bits):
    wq = torch.from_numpy(binding.pack(q, bits).view(np.int32)).cuda()
    return wq, torch.from_numpy(sc).cuda()


@pytest.mark.parametrize("fmt,bits", FORMATS)
def test_every_code_value(torch_cuda, fmt, bits):
    """Each code of the format in turn (one-hot X picks it out): the GPU
    reproduces the oracle's decoding of every E2M1 and every E4M3 code, the
    two NaN codes (0x7F, 0xFF) included (NaN where the oracle has NaN)."""
    torch = torch_cuda
    ncode = 16 if bits == 4 else 256
    codes = list(range(ncode))
    N, K = len(codes), 64
    q = np.zeros((N, K), dtype=np.uint8)
    q[:, 5] = codes
    # scale 1: E8M0 127, or E4M3 0x38 for nvfp4 (groups of 16)
    sc = np.full((N, K // 16), 0x38, dtype=np.uint8) if fmt == "nvfp4" else np.full((N, K // 32), 127, dtype=np.uint8)
    wq, s = upload(torch, q, sc, bits)
    xb = np.zeros((1, K), dtype=np.uint16)
    xb[0, 5] = 0x3F80  # bf16 1.0
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y = to_f64(binding.small_m_mx(x, wq, s, fmt, out_dtype=torch.float32))
    ref, _ = oracle.load().mx_qmm(fmt, xb, binding.pack(q, bits), sc)
    assert np.array_equal(y[0], ref[0], equal_nan=True)
    if bits == 8:
        assert np.isnan(ref[0][[0x7F, 0xFF]]).all() and np.isfinite(np.delete(ref[0], [0x7F, 0xFF])).all()


@pytest.mark.parametrize("fmt,bits", FORMATS)
def test_nan_encodings(torch_cuda, fmt, bits):
    """NaN encodings planted in the weights: E4M3 NaN codes (mxfp8), E4M3 NaN
    scale bytes (nvfp4) and E8M0 255 scales (mxfp4, mxfp8).  On the default
    and on every variant that takes the shape, bf16 and fp32, the outputs that
    are NaN are exactly the oracle's NaN outputs, and every other output meets
    the bound."""
    torch = torch_cuda
    ol = oracle.load()
    N, K = 200, 512
    q, sc = synth.make_mx(8700 + bits, N, K, fmt)
    rng = np.random.default_rng(8700)
    rows = rng.choice(N, size=12, replace=False)
    for r in rows[:6]:  # NaN scale bytes
        sc[r, rng.integers(sc.shape[1])] = (0x7F | (0x80 * int(rng.integers(2)))) if fmt == "nvfp4" else 255
    if bits == 8:
        for r in rows[6:]:  # NaN codes
            q[r, rng.integers(K)] = 0x7F | (0x80 * int(rng.integers(2)))
    wq, s = upload(torch, q, sc, bits)
    xb = synth.make_x(8700, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = ol.mx_qmm(fmt, xb, binding.pack(q, bits), sc)
    nan_ref = np.isnan(y_ref)
    assert nan_ref[:, rows[:6]].all() and nan_ref.any(axis=0).sum() == (12 if bits == 8 else 6)
    names = binding.variant_names()
    for v in [-1] + list(range(len(names))):
        for M in (1, 9, 16):
            for dt in (torch.float32, torch.bfloat16):
                try:
                    y = to_f64(binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=dt, variant=v))
                except binding.QmmError as e:
                    assert e.status == 3 and names[v].startswith("tma"), names[v]
                    break
                what = f"{fmt} {'default' if v < 0 else names[v]} M={M} {dt}"
                assert np.array_equal(np.isnan(y), nan_ref[:M]), what + ": NaN positions"
                fin = ~nan_ref[:M]
                assert_within(y[fin], y_ref[:M][fin], a_ref[:M][fin], what, bf16=dt == torch.bfloat16)


@pytest.mark.parametrize("fmt,bits", FORMATS)
def test_mx_products(torch_cuda, fmt, bits):
    """Several tiles and a ragged N, M = 1..16, every mma variant with split 1
    and 2, bf16 and fp32; then a 4096x4096 layer at sampled outputs."""
    torch = torch_cuda
    ol = oracle.load()
    N, K = 200, 512
    q, sc = synth.make_mx(8600, N, K, fmt)
    wq, s = upload(torch, q, sc, bits)
    xb = synth.make_x(8600, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = ol.mx_qmm(fmt, xb, binding.pack(q, bits), sc)
    for M in range(1, 17):
        y = binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.float32)
        assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"{fmt} M={M}")
    names = binding.variant_names()
    ran_own = False
    for v in range(len(names)):
        for sp in (1, 2):
            for M in (3, 12):
                try:
                    y32 = binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.float32, variant=v,
                                             splits=sp)
                except binding.QmmError as e:  # tma variants, and warp-owned ones that cannot plan this shape
                    assert e.status == 3 and names[v].startswith("tma"), names[v]
                    continue
                ran_own |= names[v].startswith("tma_own")
                assert_within(to_f64(y32), y_ref[:M], a_ref[:M], f"{fmt} v{v} s{sp} M={M}")
                y16 = binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.bfloat16, variant=v,
                                         splits=sp)
                assert torch.equal(y16, y32.to(torch.bfloat16)), f"{fmt} v{v} s{sp} M={M}: bf16 = RNE(fp32)"
    assert ran_own
    N = K = 4096
    q, sc = synth.make_mx(8601, N, K, fmt)
    wq, s = upload(torch, q, sc, bits)
    xb = synth.make_x(8601, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = ol.mx_qmm(fmt, xb, binding.pack(q, bits), sc)
    for M in (1, 8, 16):
        y = to_f64(binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.float32))
        ms, ns = sample_positions(M, N, 256, seed=M)
        assert_within(y[ms, ns], y_ref[ms, ns], a_ref[ms, ns], f"{fmt} 4096 M={M}")


@pytest.mark.parametrize("fmt,bits", FORMATS)
@pytest.mark.parametrize("N,K", [(72, 256), (71, 256), (64, 2880), (16, 8224)])
def test_mx_unstrided_scale_rows(torch_cuda, fmt, bits, N, K):
    """Scale-byte rows that are not 16-byte strided (K/g not a multiple of 16:
    8 or 90 bytes per row; nvfp4's 16 and 180): the warp-owned family copies
    each tile's scale bytes whole when N * K/g is a multiple of 16 and K/g <=
    256, and refuses otherwise (71 rows; 257 groups), where the default falls
    back to the mma family.  Default, a forced warp-owned and a forced mma
    variant against the oracle."""
    torch = torch_cuda
    q, sc = synth.make_mx(8602 + N + K, N, K, fmt)
    wq, s = upload(torch, q, sc, bits)
    xb = synth.make_x(8602, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = oracle.load().mx_qmm(fmt, xb, binding.pack(q, bits), sc)
    G = K // binding.MX_FORMATS[fmt][2]
    own_ok = (N * G) % 16 == 0 and G <= 256
    names = binding.variant_names()
    for M in (1, 9):
        y = binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.float32)
        assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"{fmt} N={N} K={K} M={M} default")
        for v in (names.index("tma_own_w8_d2_2cta"), names.index("mma_r2_wn2_wk4")):
            try:
                y = binding.small_m_mx(x[:M].contiguous(), wq, s, fmt, out_dtype=torch.float32, variant=v)
            except binding.QmmError as e:
                assert e.status == 3 and names[v].startswith("tma_own") and not own_ok, f"{names[v]}: {e}"
                continue
            assert own_ok or not names[v].startswith("tma_own"), f"{names[v]} took G={G} N={N}"
            assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"{fmt} N={N} K={K} M={M} {names[v]}")
