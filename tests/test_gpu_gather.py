"""GPU parity of the gathered (mixture-of-experts) form,
Y[i] = X[lhs[i]] . dequant(W[rhs[i]])^T over an expert stack
(qmm_gather_small_m), against the oracle's gathered product, with the
library's bound |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5."""
import numpy as np
import pytest

from oracle import oracle
from qmm_harness import assert_within, check, to_f64
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


class DeviceStack:
    """A synth.MoeProblem on the GPU (product packing)."""

    def __init__(self, torch, mp: synth.MoeProblem):
        self.mp = mp
        E, N, K = mp.E, mp.N, mp.K
        wq = binding.pack(mp.q.reshape(E * N, K), mp.bits).reshape(E, N, -1)
        self.wq = torch.from_numpy(wq.view(np.int32)).cuda()
        self.s = torch.from_numpy(mp.scales.view(np.float16)).cuda()
        self.b = torch.from_numpy(mp.biases.view(np.float16)).cuda()
        self.x = torch.from_numpy(mp.x.view(np.int16)).cuda().view(torch.bfloat16)

    def run(self, torch, T, lhs, rhs, **kw):
        return binding.gather_small_m(self.x[:T].contiguous(), self.wq, self.s, self.b,
                                      torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(), self.mp.bits,
                                      self.mp.group_size, **kw)


def oracle_ref(mp: synth.MoeProblem, T, lhs, rhs):
    ol = oracle.load()
    E, N, K = mp.E, mp.N, mp.K
    wq = ol.pack(mp.q.reshape(E * N, K), mp.bits).reshape(E, N, -1)
    return ol.gather_qmm(mp.x[:T], wq, mp.scales, mp.biases, lhs, rhs, mp.bits, mp.group_size)


def gather_variants():
    """Every variant: mma (each expert's own entries), tma and warp-owned
    (every token against each expert of the union)."""
    return list(range(len(binding.variant_names())))


@pytest.mark.parametrize("groups", [4, 8], ids=["G4", "G8"])
@pytest.mark.parametrize("bits,gs", [(4, 64), (2, 32), (8, 32), (4, 128)])
def test_gather_small_stacks(torch_cuda, bits, gs, groups):
    """Ragged N, T = 1..16 tokens routed to k = 1..4 distinct experts, every
    variant, split 1 and 2, bf16 and fp32.  With 4 groups per row (scale rows
    not 16-byte strided) the row-stacking TMA variants cannot plan the shape and
    the warp-owned ones take each tile's metadata whole."""
    torch = torch_cuda
    E, N, K = 6, 200, groups * gs
    ran_tma = ran_own = False
    for T, k in ((1, 1), (3, 2), (8, 4), (16, 2), (5, 4)):
        mp = synth.make_moe(8100 + T * 10 + k + bits * 100 + gs + groups, E, N, K, bits, gs, T, k)
        ds = DeviceStack(torch, mp)
        lhs, rhs = mp.lists()
        y_ref, a_ref = oracle_ref(mp, T, lhs, rhs)
        y = ds.run(torch, T, lhs, rhs, out_dtype=torch.float32)  # the library's choice
        assert_within(to_f64(y), y_ref, a_ref, f"T={T} k={k} default")
        for v in gather_variants():
            for s in (1, 2):
                for dt in (torch.float32, torch.bfloat16):
                    try:
                        y = ds.run(torch, T, lhs, rhs, out_dtype=dt, variant=v, splits=s)
                    except binding.QmmError as e:
                        assert e.status == 3 and binding.variant_names()[v].startswith("tma")
                        continue  # a tma / warp-owned variant that cannot plan this shape
                    ran_tma |= binding.variant_names()[v].startswith("tma_w")
                    ran_own |= binding.variant_names()[v].startswith("tma_own")
                    check(y, y_ref, a_ref, f"T={T} k={k} v{v} s{s} {dt}")
    assert ran_own and ran_tma == (groups == 8)


@pytest.mark.parametrize("K", [256, 512], ids=["G4", "G8"])
def test_gather_arbitrary_lists_and_determinism(torch_cuda, K):
    """A hand-made list with a repeated (token, expert) entry, unsorted experts
    and an expert used by one entry only, at the library's choice, on a forced
    mma and warp-owned variant and (8 groups per row) a forced tma variant;
    repeats are bit-identical."""
    torch = torch_cuda
    mp = synth.make_moe(8200, 5, 136, K, 4, 64, 4, 1)
    ds = DeviceStack(torch, mp)
    lhs = np.array([3, 0, 0, 2, 1, 3, 0, 2], dtype=np.int32)
    rhs = np.array([4, 1, 4, 1, 0, 1, 1, 4], dtype=np.int32)
    y_ref, a_ref = oracle_ref(mp, 4, lhs, rhs)
    tma = binding.variant_names().index("tma_w8_2cta")
    own = binding.variant_names().index("tma_own_w8_d2_2cta")
    mma = binding.variant_names().index("mma_r2_wn2_wk4")
    for v in ([-1, mma, tma, own] if K == 512 else [-1, mma, own]):
        first = ds.run(torch, 4, lhs, rhs, out_dtype=torch.float32, variant=v)
        assert_within(to_f64(first), y_ref, a_ref, f"hand-made list v{v}")
        assert torch.equal(first[1], first[6]), "a repeated entry gets the same row"
        for _ in range(3):
            assert torch.equal(first, ds.run(torch, 4, lhs, rhs, out_dtype=torch.float32, variant=v))


@pytest.mark.parametrize("T", [1, 4, 8])
def test_gather_moe_workload_full(torch_cuda, T):
    """The 128-expert top-8 gate+up stack at verify widths: every output, at
    the library's choice and on a forced warp-owned variant."""
    torch = torch_cuda
    w = workloads.MOE_GATE_UP
    mp = synth.make_moe(w.seed, w.E, w.N, w.K, w.bits, w.group_size, T, w.k)
    ds = DeviceStack(torch, mp)
    lhs, rhs = mp.lists()
    y_ref, a_ref = oracle_ref(mp, T, lhs, rhs)
    for v in (-1, binding.variant_names().index("mma_r2_wn2_wk4")):
        y = ds.run(torch, T, lhs, rhs, variant=v)
        check(y, y_ref, a_ref, f"moe T={T} v{v}")


@pytest.mark.parametrize("K", [256, 512], ids=["G4", "G8"])
def test_gather_invalid_index_flagged(torch_cuda, K):
    """An expert index out of range: its row stays unwritten, the others are
    right, and the device status word reports bit 3."""
    torch = torch_cuda
    mp = synth.make_moe(8300, 4, 64, K, 4, 64, 4, 1)
    ds = DeviceStack(torch, mp)
    lhs = np.array([0, 1, 2, 3], dtype=np.int32)
    rhs = np.array([0, 9, 2, 1], dtype=np.int32)
    ok = np.array([0, 2, 3])
    y_ref, a_ref = oracle_ref(mp, 4, lhs[ok], rhs[ok])
    tma = binding.variant_names().index("tma_w8_2cta")
    own = binding.variant_names().index("tma_own_w8_d2_2cta")
    mma = binding.variant_names().index("mma_r2_wn2_wk4")
    for v in ([-1, mma, tma, own] if K == 512 else [-1, mma, own]):
        out = torch.full((4, 64), 5.0, dtype=torch.float32, device="cuda")
        ds.run(torch, 4, lhs, rhs, out=out, variant=v)
        torch.cuda.synchronize()
        assert binding.device_status(clear=True) & 8
        assert bool((out[1] == 5.0).all())
        assert_within(to_f64(out)[ok], y_ref, a_ref, f"valid rows of a list with a bad index v{v}")


def test_gather_too_many_entries_for_one_expert_flagged(torch_cuda):
    """On the mma variants, a ninth entry for one expert with T <= 8 is flagged
    and that expert's rows stay unwritten; the library's choice (warp-owned)
    and the row-stacking variants (8 groups per row) take the same list."""
    torch = torch_cuda
    names = binding.variant_names()
    mp = synth.make_moe(8301, 4, 64, 256, 4, 64, 4, 1)
    ds = DeviceStack(torch, mp)
    lhs9 = np.array([0, 1, 2, 3, 0, 1, 2, 3, 0], dtype=np.int32)
    rhs9 = np.zeros(9, dtype=np.int32)
    out9 = torch.full((9, 64), 5.0, dtype=torch.float32, device="cuda")
    ds.run(torch, 4, lhs9, rhs9, out=out9, variant=names.index("mma_r2_wn2_wk4"))
    torch.cuda.synchronize()
    assert binding.device_status(clear=True) & 8
    assert bool((out9 == 5.0).all())
    y_ref, a_ref = oracle_ref(mp, 4, lhs9, rhs9)
    y = ds.run(torch, 4, lhs9, rhs9, out_dtype=torch.float32)
    assert_within(to_f64(y), y_ref, a_ref, "nine entries for one expert, 4 groups per row, default")
    mp8 = synth.make_moe(8302, 4, 64, 512, 4, 64, 4, 1)
    ds8 = DeviceStack(torch, mp8)
    y_ref, a_ref = oracle_ref(mp8, 4, lhs9, rhs9)
    for v in (-1, names.index("tma_w8_2cta")):
        y = ds8.run(torch, 4, lhs9, rhs9, out_dtype=torch.float32, variant=v)
        assert_within(to_f64(y), y_ref, a_ref, f"nine entries for one expert, v{v}")
