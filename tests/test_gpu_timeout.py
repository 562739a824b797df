"""A bounded device wait that runs out, without a GPU fault.

Every mbarrier wait in the kernels is bounded in time; one that gives up sets
a bit of the device status word (qmm_device_status) and the kernel carries on,
so that the context stays usable.  The host-side injection
QMM_TEST_INJECT=short_wait makes one wait run out on purpose: the TMA
family's launcher passes a 100 us limit for the waits on tile data, and the
producer of cluster 0 declares 16 bytes more for its first tile than the
copies deliver, so that tile's phase never completes.  The copies themselves
all land (nothing is left in flight at exit), the consumers of that tile give
up after 100 us (status bit 0), the producer's drain gives up on the same
phase (bit 2), and every CTA still passes its cluster barriers and receives
its partners' partial sums with the normal (2 s) limit.  The test checks the
status bits, that the call returned, and that the next, normal call is
correct and leaves the status word clear."""
import numpy as np
import pytest

from qmm_harness import DeviceProblem, OracleRef, check
from quantized_matmul_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_matmul_speculative_gb300 import build

    build.build()
    binding.lib()
    return torch


@pytest.mark.parametrize("variant,splits", [("tma_w8_2cta", 2), ("tma_w4_2cta", 4)])
def test_short_wait_gives_up_and_the_next_call_is_clean(torch_cuda, monkeypatch, variant, splits):
    torch = torch_cuda
    N, K, M = 256, 1024, 4
    p = synth.make_problem(9100, N, K, 4, 64)
    dp = DeviceProblem(p)
    ref = OracleRef(p)
    y_ref, a_ref = ref.full(M)
    v = binding.variant_names().index(variant)
    binding.device_status(clear=True)

    monkeypatch.setenv("QMM_TEST_INJECT", "short_wait")
    y_bad = dp.run(M, out_dtype=torch.float32, variant=v, splits=splits)
    torch.cuda.synchronize()
    status = binding.device_status(clear=True)
    assert status & 1, f"a consumer wait should have given up (status {status:#x})"
    assert status & 4, f"the producer's drain should have given up (status {status:#x})"
    assert status & ~0x7 == 0, f"unexpected status bits {status:#x}"
    assert y_bad.shape == (M, N)

    monkeypatch.delenv("QMM_TEST_INJECT")
    y = dp.run(M, out_dtype=torch.float32, variant=v, splits=splits)
    torch.cuda.synchronize()
    assert binding.device_status(clear=True) == 0
    check(y, y_ref, a_ref, f"{variant} s{splits} after a wait gave up")
    # and the default path as well
    check(dp.run(M, out_dtype=torch.float32), y_ref, a_ref, "default path after a wait gave up")
    assert binding.device_status(clear=True) == 0
