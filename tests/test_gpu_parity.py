"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every output must satisfy |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5.  Small
shapes are checked element by element against the full oracle; full-size
workload shapes are checked on sampled outputs the oracle computes one by one,
in the same launch configuration the benchmark uses (the dispatcher's choice).
"""
import pytest

from qmm_harness import DeviceProblem, OracleRef, assert_within, check, sample_positions, to_f64
from quantized_matmul_speculative_gb300 import binding, synth, workloads

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


def variants():
    return list(range(len(binding.variant_names())))


def is_tma(v):
    return binding.variant_names()[v].startswith("tma")


@pytest.fixture(autouse=True)
def no_device_faults(torch_cuda):
    """Every GPU test ends with a clean device status word (no bounded wait gave up)."""
    binding.device_status(clear=True)
    yield
    torch_cuda.cuda.synchronize()
    assert binding.device_status(clear=True) == 0


# ------------------------------------------------------------- small shapes
@pytest.mark.parametrize("bits,gs", BITS_GS)
def test_small_shapes_all_m(torch_cuda, bits, gs):
    """Several tiles and a ragged N tail, M = 1..16, every variant, split 1 and 2."""
    torch = torch_cuda
    N, K = 200, 8 * gs
    p = synth.make_problem(7000 + bits * 1000 + gs, N, K, bits, gs)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(16)
    ran_tma = False
    for v in variants():
        for splits in ((1, 2, 4) if is_tma(v) else (1, 2)):
            for M in range(1, 17):
                y = dp.run(M, out_dtype=torch.float32, variant=v, splits=splits, allow_unsupported=is_tma(v))
                if y is None:
                    break
                ran_tma |= is_tma(v)
                assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"v{v} s{splits} M={M} f32")
            y = dp.run(16, variant=v, splits=splits, allow_unsupported=is_tma(v))
            if y is not None:
                check(y, y_ref, a_ref, f"v{v} s{splits} M=16 bf16")
    assert ran_tma, "no TMA variant ran on this shape"


@pytest.mark.parametrize("N", [1, 7, 15, 17, 129])
@pytest.mark.parametrize("bits,gs", [(4, 64), (2, 32), (4, 128), (8, 64)])
def test_ragged_n_and_one_group(torch_cuda, N, bits, gs):
    torch = torch_cuda
    for K in (gs, 2 * gs, 8 * gs):
        p = synth.make_problem(8000 + N + K, N, K, bits, gs)
        dp, ref = DeviceProblem(p), OracleRef(p)
        y_ref, a_ref = ref.full(16)
        for v in variants():
            for M in (1, 8, 9, 16):
                for splits in (1, 3):
                    y = dp.run(M, out_dtype=torch.float32, variant=v, splits=splits, allow_unsupported=is_tma(v))
                    if y is None:
                        continue
                    assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"N={N} K={K} v{v} M={M} s{splits}")


def test_single_layer_workload_full(torch_cuda):
    """1024x1024 4-bit g64 at M=4: every output, every variant and split 1..8, both dtypes."""
    torch = torch_cuda
    w = workloads.SINGLE_LAYER
    sh = w.shapes[0]
    p = synth.make_problem(workloads.shape_seed(w, 0), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(4)
    y = dp.run(4)
    check(y, y_ref, a_ref, "dispatcher")
    for v in variants():
        for splits in (1, 2, 4, 8):
            for dt in (torch.bfloat16, torch.float32):
                y = dp.run(4, out_dtype=dt, variant=v, splits=splits, allow_unsupported=is_tma(v))
                if y is not None:
                    check(y, y_ref, a_ref, f"v{v} s{splits} {dt}")


def test_m_sweep_5120_full(torch_cuda):
    """5120x5120 4-bit g64, M = 1..16 through the dispatcher: every output."""
    w = workloads.M_SWEEP
    sh = w.shapes[0]
    p = synth.make_problem(workloads.shape_seed(w, 0), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(16)
    for M in w.ms:
        y = dp.run(M)
        check(y, y_ref[:M], a_ref[:M], f"M={M}")


@pytest.mark.parametrize("shape_index", range(4))
def test_dense27b_layer_sampled(torch_cuda, shape_index):
    w = workloads.DENSE_27B_LAYER
    sh = w.shapes[shape_index]
    p = synth.make_problem(workloads.shape_seed(w, shape_index), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    for M in w.ms:
        y = dp.run(M)
        ms, ns = sample_positions(M, sh.N, 192, seed=M)
        y_ref, a_ref = ref.sampled(M, ms, ns)
        check(y, y_ref, a_ref, f"{sh.name} M={M}", at=(ms, ns))


@pytest.mark.parametrize("bits,gs", workloads.GROUP_BIT_SWEEP.variants)
def test_group_bit_sweep_sampled(torch_cuda, bits, gs):
    w = workloads.GROUP_BIT_SWEEP
    sh = w.shapes[0]
    p = synth.make_problem(workloads.shape_seed(w, 0, bits=bits, group_size=gs), sh.N, sh.K, bits, gs)
    dp, ref = DeviceProblem(p), OracleRef(p)
    for M in w.ms:
        y = dp.run(M)
        ms, ns = sample_positions(M, sh.N, 96, seed=M)
        y_ref, a_ref = ref.sampled(M, ms, ns)
        check(y, y_ref, a_ref, f"{bits}b g{gs} M={M}", at=(ms, ns))


@pytest.mark.parametrize("shape_index", range(4))
def test_verify_step_shapes_sampled(torch_cuda, shape_index):
    w = workloads.VERIFY_STEP
    sh = w.shapes[shape_index]
    p = synth.make_problem(workloads.shape_seed(w, shape_index), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    for M in w.ms:
        y = dp.run(M)
        ms, ns = sample_positions(M, sh.N, 96, seed=M)
        y_ref, a_ref = ref.sampled(M, ms, ns)
        check(y, y_ref, a_ref, f"{sh.name} M={M}", at=(ms, ns))


@pytest.mark.parametrize("wname,shape_index", [("int8_affine_8b_g64", 0), ("int8_affine_8b_g64", 1),
                                               ("qmv_wide_gate_up_15360x3840_4b_g64", 0)])
def test_int8_and_qmv_wide_sampled(torch_cuda, wname, shape_index):
    """M = 1..16 through the dispatcher: 8-bit affine g64 on 5120x5120 and on
    the 15360x3840 gate/up shape, and that shape at 4 bits (60 groups per row:
    scale rows that are not 16-byte strided)."""
    w = workloads.BY_NAME[wname]
    sh = w.shapes[shape_index]
    p = synth.make_problem(workloads.shape_seed(w, shape_index), sh.N, sh.K, w.bits, w.group_size)
    dp, ref = DeviceProblem(p), OracleRef(p)
    for M in w.ms:
        y = dp.run(M)
        ms, ns = sample_positions(M, sh.N, 128, seed=M)
        y_ref, a_ref = ref.sampled(M, ms, ns)
        check(y, y_ref, a_ref, f"{w.name} {sh.name} M={M}", at=(ms, ns))


# ------------------------------------- scale rows that are not 16-byte strided
# (bits, group size, groups per row G, N): G % 8 != 0, so a [N, G] fp16 row is
# not a 16-byte multiple; N * G % 8 == 0 except in the last two, and the last
# has G > 128.
UNSTRIDED = [(4, 64, 60, 200), (4, 64, 45, 64), (8, 64, 60, 48), (2, 32, 30, 96), (4, 128, 30, 32),
             (4, 64, 84, 160), (4, 32, 100, 64), (4, 64, 1, 16), (4, 64, 3, 40), (4, 64, 12, 18),
             (4, 64, 60, 17), (4, 32, 130, 16)]


@pytest.mark.parametrize("bits,gs,G,N", UNSTRIDED)
def test_unstrided_scale_rows(torch_cuda, bits, gs, G, N):
    """The warp-owned variants take such shapes (each stage holds its tile's
    metadata for every group) when N * G is a multiple of 8 and G <= 128, and
    refuse the others; the row-stacking TMA variants never run them.  Every
    variant that runs, split 1..4, M = 1, 8, 9, 16, against the oracle; at
    M = 1 the dispatcher falls back to a warp-owned variant exactly when one of
    its two warp-owned defaults can plan the shape (the whole-tile metadata
    takes 64 G bytes of every stage, so large G can run out of shared memory)."""
    torch = torch_cuda
    K = G * gs
    p = synth.make_problem(9700 + G + N + bits, N, K, bits, gs)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(16)
    names = binding.variant_names()
    own_ok = N * G % 8 == 0 and G <= 128
    defaults = {"tma_own_w8_d2_2cta", "tma_own_w16_d2_1cta"}  # the dispatcher's warp-owned fallbacks
    ran_own = default_ran_m1 = False
    for v in variants():
        for splits in (1, 2, 3, 4):
            for M in (1, 8, 9, 16):
                y = dp.run(M, out_dtype=torch.float32, variant=v, splits=splits, allow_unsupported=is_tma(v))
                if y is None:  # (a warp-owned variant may also refuse for shared memory or G % splits)
                    continue
                assert not names[v].startswith("tma_w"), f"{names[v]} planned G={G}"
                assert own_ok or not names[v].startswith("tma_own"), f"{names[v]} took N*G % 8 != 0 or G > 128"
                ran_own |= names[v].startswith("tma_own")
                default_ran_m1 |= M == 1 and names[v] in defaults
                assert_within(to_f64(y), y_ref[:M], a_ref[:M], f"G={G} N={N} {names[v]}/{splits} M={M}")
    assert ran_own == own_ok
    v, s = binding.select_variant(1, N, K, bits, gs)
    assert names[v].startswith("tma_own") == default_ran_m1, f"dispatcher chose {names[v]} for G={G} M=1"
    for M in (1, 9, 16):
        check(dp.run(M), y_ref[:M], a_ref[:M], f"G={G} N={N} dispatcher M={M}")


# ------------------------------------------------------------- properties
def test_determinism_and_batch_invariance(torch_cuda):
    torch = torch_cuda
    p = synth.make_problem(9100, 777, 2048, 4, 64)
    dp, ref = DeviceProblem(p), OracleRef(p)
    y_ref, a_ref = ref.full(16)
    for v in variants():
        first = dp.run(16, out_dtype=torch.float32, variant=v, splits=4, allow_unsupported=is_tma(v))
        if first is None:
            continue
        for _ in range(4):
            again = dp.run(16, out_dtype=torch.float32, variant=v, splits=4)
            assert torch.equal(first, again), f"variant {v} not deterministic"
        assert_within(to_f64(first), y_ref, a_ref, f"variant {v} M=16")
        # each row of the 16-row call against a 1-row call on that row alone
        for m in (0, 5, 15):
            x1 = dp.x[m:m + 1].contiguous()
            single = binding.small_m(x1, dp.wq, dp.s, dp.b, 4, 64, out_dtype=torch.float32, variant=v, splits=4)
            assert_within(to_f64(single)[0], y_ref[m], a_ref[m], f"variant {v} row {m} alone")
            bitwise = torch.equal(single[0], first[m])
            print(f"variant {v} row {m}: bit-identical across M: {bitwise}")


def test_output_guard_bands(torch_cuda):
    """Writes stay inside Y: canaries around the output are untouched."""
    torch = torch_cuda
    p = synth.make_problem(9200, 129, 512, 4, 64)
    dp = DeviceProblem(p)
    for M in (1, 7, 16):
        for dt in (torch.bfloat16, torch.float32):
            pad = 64
            buf = torch.full((M * 129 + 2 * pad,), -12345.0, dtype=dt, device="cuda")
            out = buf[pad:pad + M * 129].view(M, 129)
            for v in variants():
                dp.run(M, out_dtype=dt, variant=v, splits=2, out=out, allow_unsupported=is_tma(v))
                torch.cuda.synchronize()
                assert bool((buf[:pad] == -12345.0).all()) and bool((buf[-pad:] == -12345.0).all())


def test_empty_and_degenerate(torch_cuda):
    torch = torch_cuda
    dev = "cuda"
    x = torch.zeros((4, 0), dtype=torch.bfloat16, device=dev)
    wq = torch.zeros((5, 0), dtype=torch.int32, device=dev)
    s = torch.zeros((5, 0), dtype=torch.float16, device=dev)
    y = torch.full((4, 5), 7.0, dtype=torch.float32, device=dev)
    binding.small_m(x, wq, s, s, 4, 64, out=y)  # K = 0: empty sum
    assert bool((y == 0).all())
    # M = 0 and N = 0 launch nothing and succeed
    binding.small_m_ptr(0, 0, 0, 0, 0, 5, 64, 4, 64, 0)
    binding.small_m_ptr(0, 0, 0, 0, 3, 0, 64, 4, 64, 0)


def test_error_paths_launch_nothing(torch_cuda, monkeypatch):
    torch = torch_cuda
    p = synth.make_problem(9300, 64, 256, 4, 64)
    dp = DeviceProblem(p)
    y = torch.full((2, 64), 3.0, dtype=torch.float32, device="cuda")
    x = dp.x[:2].contiguous()
    args = [x.data_ptr(), dp.wq.data_ptr(), dp.s.data_ptr(), dp.b.data_ptr(), 2, 64, 256, 4, 64, y.data_ptr()]
    cases = {
        "misaligned X": (dict(idx=0, delta=2), 4),
        "misaligned Wq": (dict(idx=1, delta=4), 4),
    }
    for name, (mod, code) in cases.items():
        a = list(args)
        a[mod["idx"]] += mod["delta"]
        with pytest.raises(binding.QmmError) as ei:
            binding.small_m_ptr(*a, out_dtype=binding.OUT_F32)
        assert ei.value.status == code, name
    for bad, code in (({"M": 17}, 2), ({"bits": 3}, 3), ({"gs": 48}, 3), ({"K": 96}, 2)):
        a = list(args)
        key = {"M": 4, "bits": 7, "gs": 8, "K": 6}[next(iter(bad))]
        a[key] = next(iter(bad.values()))
        with pytest.raises(binding.QmmError) as ei:
            binding.small_m_ptr(*a, out_dtype=binding.OUT_F32)
        assert ei.value.status == code, bad
    monkeypatch.setenv("QMM_TEST_INJECT", "launch_fail")
    with pytest.raises(binding.QmmError) as ei:
        binding.small_m_ptr(*args, out_dtype=binding.OUT_F32)
    assert ei.value.status == 5
    monkeypatch.delenv("QMM_TEST_INJECT")
    torch.cuda.synchronize()
    assert bool((y == 3.0).all()), "a rejected call wrote to Y"
    # the context is still healthy
    binding.small_m_ptr(*args, out_dtype=binding.OUT_F32)
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_repack_round_trip_and_use(torch_cuda):
    """qmm_repack / qmm_unrepack are bit-exact inverses, and a repacked matrix
    gives the oracle's result through the normal entry point."""
    import torch

    p = synth.make_problem(91, 200, 1024, 4, 64)
    dp = DeviceProblem(p)
    native = binding.repack(dp.wq, 4)
    back = binding.repack(native, 4, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(native, dp.wq) and torch.equal(back, dp.wq)
    ref = OracleRef(p)
    y_ref, a_ref = ref.full(5)
    y = binding.small_m(dp.x[:5].contiguous(), native, dp.s, dp.b, 4, 64, out_dtype=torch.float32)
    assert_within(to_f64(y), y_ref, a_ref, "repacked weights")



# ------------------------------------------------------------- large extents
@pytest.mark.parametrize("N,K,bits,gs,M", [(64, 65536, 4, 128, 16), (262144, 256, 4, 64, 3), (96, 32768, 8, 32, 9)],
                         ids=["K65536", "N262144", "K32768_8bit"])
def test_large_extents(torch_cuda, N, K, bits, gs, M):
    """A very long K (the activations no longer fit one CTA's shared memory
    unless K is split) and a very tall N, on every variant that takes the
    shape, against the oracle (full for long K, sampled for tall N)."""
    torch = torch_cuda
    p = synth.make_problem(9500 + N % 1000 + K % 997, N, K, bits, gs)
    dp, ref = DeviceProblem(p), OracleRef(p)
    full = N * K <= 64 * 65536
    if full:
        y_ref, a_ref = ref.full(M)
    ms, ns = sample_positions(M, N, 256, seed=7)
    if not full:
        y_ref_s, a_ref_s = ref.sampled(M, ms, ns)
    ran = 0
    for v in [-1] + variants():
        y = dp.run(M, out_dtype=torch.float32, variant=v, allow_unsupported=True)
        if y is None:
            continue
        ran += 1
        y = to_f64(y)
        if full:
            assert_within(y, y_ref, a_ref, f"N={N} K={K} v{v}")
        else:
            assert_within(y[ms, ns], y_ref_s, a_ref_s, f"N={N} K={K} v{v}")
    assert ran >= 2
