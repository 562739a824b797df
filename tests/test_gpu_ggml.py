"""ggml Q4_0 / Q4_1 / Q8_0 weights on the GPU: qmm_from_ggml converts the
blocks exactly (the converted matrix dequantizes, in fp64, to exactly the
oracle's decoding of the blocks), and the product through qmm_small_m on the
converted weights matches the oracle's ggml product within the library's
bound |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5."""
import numpy as np
import pytest

from oracle import oracle
from qmm_harness import check, sample_positions
from quantized_matmul_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu

KINDS = ["q4_0", "q4_1", "q8_0"]


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


def convert(torch, blocks, N, K, kind):
    wq, s, b, bits = binding.from_ggml(kind, torch.from_numpy(blocks.reshape(-1)).cuda(), N, K)
    torch.cuda.synchronize()
    return wq, s, b, bits


@pytest.mark.parametrize("kind", KINDS)
def test_conversion_is_exact(torch_cuda, kind):
    torch = torch_cuda
    N, K = 37, 320
    blocks = synth.make_ggml_blocks(8400, N, K, kind)
    wq, s, b, bits = convert(torch, blocks, N, K, kind)
    ol = oracle.load()
    w_conv = ol.dequant(wq.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
                        b.cpu().numpy().view(np.uint16), K, bits, 32)
    assert np.array_equal(w_conv, ol.ggml_dequant(kind, blocks, N, K))


@pytest.mark.parametrize("kind", KINDS)
def test_ggml_product(torch_cuda, kind):
    """Several tiles and a ragged N, M = 1..16 at the dispatcher's choice and
    on every variant at M = 5, bf16 and fp32; then a 4096x4096 layer at
    sampled outputs."""
    torch = torch_cuda
    ol = oracle.load()
    N, K = 200, 512
    blocks = synth.make_ggml_blocks(8500, N, K, kind)
    wq, s, b, bits = convert(torch, blocks, N, K, kind)
    xb = synth.make_x(8500, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = ol.ggml_qmm(kind, xb, blocks, N)
    for M in range(1, 17):
        y = binding.small_m(x[:M].contiguous(), wq, s, b, bits, 32, out_dtype=torch.float32)
        check(y, y_ref[:M], a_ref[:M], f"{kind} M={M}")
    for v in range(len(binding.variant_names())):
        for dt in (torch.float32, torch.bfloat16):
            try:
                y = binding.small_m(x[:5].contiguous(), wq, s, b, bits, 32, out_dtype=dt, variant=v, splits=2)
            except binding.QmmError as e:
                assert e.status == 3
                continue
            check(y, y_ref[:5], a_ref[:5], f"{kind} v{v} {dt}")

    N = K = 4096
    blocks = synth.make_ggml_blocks(8501, N, K, kind)
    wq, s, b, bits = convert(torch, blocks, N, K, kind)
    xb = synth.make_x(8501, K)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y_ref, a_ref = ol.ggml_qmm(kind, xb, blocks, N)
    for M in (1, 8, 16):
        y = binding.small_m(x[:M].contiguous(), wq, s, b, bits, 32)
        ms, ns = sample_positions(M, N, 256, seed=M)
        check(y, y_ref[ms, ns], a_ref[ms, ns], f"{kind} 4096 M={M}", at=(ms, ns))


@pytest.mark.parametrize("kind", KINDS)
def test_conversion_unaligned_buffers(torch_cuda, kind):
    """The conversion's byte-wise staging (a block buffer that starts on an odd
    address) and its word-wise stores (code words 4- but not 16-byte aligned),
    over a partial last CTA of blocks: still exact."""
    torch = torch_cuda
    N, K = 29, 640  # 580 blocks: one full CTA of 512 blocks and a partial one
    blocks = synth.make_ggml_blocks(8700, N, K, kind)
    t, nbytes, bits = binding.GGML_TYPES[kind]
    raw = torch.zeros(blocks.size + 1, dtype=torch.uint8, device="cuda")
    raw[1:] = torch.from_numpy(blocks.reshape(-1)).cuda()
    words = N * K * bits // 32
    wq_buf = torch.zeros(words + 1, dtype=torch.int32, device="cuda")
    s = torch.empty((N, K // 32), dtype=torch.float16, device="cuda")
    b = torch.empty((N, K // 32), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = binding.lib().qmm_from_ggml(t, raw.data_ptr() + 1, N, K, wq_buf.data_ptr() + 4, s.data_ptr(), b.data_ptr(),
                                     stream)
    assert rc == 0
    torch.cuda.synchronize()
    ol = oracle.load()
    w_conv = ol.dequant(wq_buf[1:].cpu().numpy().view(np.uint32).reshape(N, -1), s.cpu().numpy().view(np.uint16),
                        b.cpu().numpy().view(np.uint16), K, bits, 32)
    assert np.array_equal(w_conv, ol.ggml_dequant(kind, blocks, N, K))
    assert int(wq_buf[0]) == 0, "a word before Wq was written"


# |d| at and just past the largest value whose bias -8 d (Q4_0) / -128 d
# (Q8_0) is a finite fp16, and the fp16 maximum: (kind, d, exact)
RANGE_CASES = [("q8_0", 511.75, True), ("q8_0", -511.75, True), ("q8_0", 512.0, False), ("q8_0", -512.0, False),
               ("q8_0", 65504.0, False), ("q4_0", 8188.0, True), ("q4_0", -8188.0, True), ("q4_0", 8192.0, False),
               ("q4_0", 65504.0, False), ("q4_1", 65504.0, True), ("q4_1", -65504.0, True)]


@pytest.mark.parametrize("kind,d,exact", RANGE_CASES, ids=[f"{k}_{d:g}" for k, d, _ in RANGE_CASES])
def test_conversion_range(torch_cuda, kind, d, exact):
    """Blocks with a large scale d: inside the stated range the conversion is
    still exact (the converted matrix dequantizes to the oracle's decoding of
    the blocks) and the status word stays clear; past it, bit 4 of the status
    word is set (the affine layout cannot hold the block)."""
    torch = torch_cuda
    N, K = 5, 96
    blocks = synth.make_ggml_blocks(8800, N, K, kind)
    blocks[7, 0:2] = np.array([d], dtype=np.float16).view(np.uint8)  # row 2, block 1
    if kind == "q4_1":  # m stays in range: fp16(-7.5 d) would overflow for |d| > 8733
        blocks[7, 2:4] = np.array([-0.5 * d], dtype=np.float16).view(np.uint8)
    binding.device_status(clear=True)
    wq, s, b, bits = convert(torch, blocks, N, K, kind)
    status = binding.device_status(clear=True)
    if not exact:
        assert status == 16, f"status {status:#x}"
        return
    assert status == 0, f"status {status:#x}"
    ol = oracle.load()
    w_conv = ol.dequant(wq.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
                        b.cpu().numpy().view(np.uint16), K, bits, 32)
    w_ref = ol.ggml_dequant(kind, blocks, N, K)
    assert np.array_equal(w_conv, w_ref)
    assert np.abs(w_ref[2, 32:64]).max() > 100.0  # the large block is really there
