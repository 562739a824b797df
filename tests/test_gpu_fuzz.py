"""Seeded random shapes through the C ABI against the fp64 oracle: random
bits and group size, N (ragged, 1..700), groups per row (1..48, half of them a
multiple of 8 so the TMA families can plan), M = 1..16, the dispatcher's choice
and every variant with a random split count and output dtype.  Every output
must satisfy |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5; a forced (variant,
splits) pair the shape cannot use must be refused with QMM_ERR_UNSUPPORTED."""
import numpy as np
import pytest

from qmm_harness import DeviceProblem, OracleRef, assert_within, to_f64
from quantized_matmul_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu

BITS_GS = [(4, 32), (4, 64), (4, 128), (2, 32), (2, 64), (2, 128), (8, 32), (8, 64), (8, 128)]


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


def random_case(seed):
    rng = np.random.default_rng(31337 + seed)
    bits, gs = BITS_GS[int(rng.integers(len(BITS_GS)))]
    groups = int(8 * rng.integers(1, 7)) if seed % 2 == 0 else int(rng.integers(1, 49))
    n = int(rng.integers(1, 701))
    m = int(rng.integers(1, 17))
    return rng, bits, gs, n, groups * gs, m


@pytest.mark.parametrize("seed", range(128))
def test_random_shape(torch_cuda, seed):
    torch = torch_cuda
    rng, bits, gs, n, k, m = random_case(seed)
    p = synth.make_problem(60000 + seed, n, k, bits, gs)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(m)
    what = f"seed {seed}: M={m} N={n} K={k} bits={bits} g={gs}"
    assert_within(to_f64(dp.run(m)), y_ref, a_ref, what + " default")
    for v in range(len(binding.variant_names())):
        splits = int(rng.integers(1, 9))
        dt = torch.float32 if rng.integers(2) else torch.bfloat16
        y = dp.run(m, out_dtype=dt, variant=v, splits=splits, allow_unsupported=True)
        if y is None:
            assert binding.variant_names()[v].startswith("tma"), f"{what}: v{v} s{splits} refused"
            continue
        assert_within(to_f64(y), y_ref, a_ref, f"{what} v{v} s{splits} {dt}")
