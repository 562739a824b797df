"""The C ABI without a GPU: the library loads, exports every declared symbol,
packs bit-exactly like the oracle's packer, and rejects bad arguments on the
host before touching the device."""
import ctypes
import os
import re
from pathlib import Path

import numpy as np
import pytest

from oracle import oracle
from quantized_matmul_speculative_gb300 import binding, build

HEADER = Path(__file__).resolve().parents[1] / "include" / "qmm.h"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "qmm_small_m" in names and "qmm_pack" in names
    raw = ctypes.CDLL(str(binding.LIBRARY))
    for name in names:
        assert hasattr(raw, name), f"{name} declared in qmm.h but not exported"
    assert set(names) == set(binding.SIGNATURES), "binding signatures out of sync with qmm.h"


def test_pack_matches_oracle_bit_exact(lib):
    ol = oracle.load()
    rng = np.random.default_rng(11)
    for bits in (2, 4, 8):
        for N, K in ((1, 32), (3, 64), (17, 256), (64, 1024)):
            q = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
            ours = binding.pack(q, bits)
            assert np.array_equal(ours, ol.pack(q, bits)), (bits, N, K)
            assert np.array_equal(binding.unpack(ours, K, bits), q)
    assert int(binding.pack(np.arange(8, dtype=np.uint8).reshape(1, 8), 4)[0, 0]) == 0x76543210
    assert int(binding.pack(np.tile(np.arange(4, dtype=np.uint8), 4).reshape(1, 16), 2)[0, 0]) == 0xE4E4E4E4


def test_pack_rejects_bad_input(lib):
    with pytest.raises(binding.QmmError):
        binding.pack(np.full((1, 8), 16, dtype=np.uint8), 4)  # code out of range
    with pytest.raises(binding.QmmError):
        binding.pack(np.zeros((1, 12), dtype=np.uint8), 4)  # K does not fill whole words
    assert binding.packed_words(10, 64, 4) == 80
    assert binding.packed_words(10, 64, 3) == 0


def test_validation_before_launch(lib):
    call = lib.qmm_small_m_ex
    # (X, Wq, S, B, M, N, K, bits, gs, Y, out, variant, splits, stream); bogus but aligned pointers
    p = 0x10000
    base = [p, p, p, p, 4, 64, 256, 4, 64, p, 0, -1, -1, None]

    def rc(**kw):
        a = list(base)
        pos = {"M": 4, "N": 5, "K": 6, "bits": 7, "gs": 8, "out": 10, "variant": 11, "splits": 12,
               "X": 0, "Wq": 1, "Y": 9}
        for k, v in kw.items():
            a[pos[k]] = v
        return call(*a)

    assert rc(M=17) == 2 and rc(M=-1) == 2 and rc(N=-3) == 2
    assert rc(bits=3) == 3 and rc(bits=16) == 3 and rc(gs=48) == 3 and rc(gs=256) == 3
    assert rc(K=96) == 2
    assert rc(out=2) == 3 and rc(variant=lib.qmm_num_variants()) == 3 and rc(splits=0) == 3 and rc(splits=17) == 3
    assert rc(X=None) == 1 and rc(Wq=None) == 1 and rc(Y=None) == 1
    assert rc(X=p + 2) == 4 and rc(Wq=p + 8) == 4 and rc(Y=p + 1) == 4
    assert rc(M=0) == 0 and rc(N=0) == 0  # nothing to compute


def test_residual_validation_before_launch(lib):
    """qmm_small_m_residual rejects a missing, misaligned or partly overlapping
    residual before any CUDA call (the pointers are never dereferenced)."""
    call = lib.qmm_small_m_residual
    p, r, y = 0x10000, 0x200000, 0x400000
    # (X, Wq, S, B, R, M, N, K, bits, gs, Y, out, variant, splits, stream)
    base = [p, p, p, p, r, 4, 64, 256, 4, 64, y, 0, -1, -1, None]

    def rc(**kw):
        a = list(base)
        pos = {"R": 4, "M": 5, "N": 6, "Y": 10, "out": 11}
        for k, v in kw.items():
            a[pos[k]] = v
        return call(*a)

    assert rc(R=None) == 1
    assert rc(R=r + 1) == 4 and rc(R=r + 2, out=1) == 4      # bf16 needs 2-byte, fp32 4-byte alignment
    assert rc(R=y + 2) == 2 and rc(R=y - 2) == 2              # partly overlaps Y
    assert rc(R=None, M=0) == 0 and rc(R=None, N=0) == 0      # nothing to compute
    assert rc(M=17) == 2


def test_gather_validation_before_launch(lib):
    """qmm_gather_small_m rejects bad sizes, widths, variants, null and
    misaligned pointers before any CUDA call."""
    call = lib.qmm_gather_small_m
    p = 0x10000
    # (X, Wq, S, B, lhs, rhs, P, T, E, N, K, bits, gs, Y, out, variant, splits, stream)
    base = [p, p, p, p, p, p, 8, 4, 16, 64, 256, 4, 64, p, 0, -1, -1, None]
    pos = {"X": 0, "lhs": 4, "rhs": 5, "P": 6, "T": 7, "E": 8, "N": 9, "K": 10, "bits": 11, "gs": 12, "Y": 13,
           "out": 14, "variant": 15, "splits": 16}

    def rc(**kw):
        a = list(base)
        for k, v in kw.items():
            a[pos[k]] = v
        return call(*a)

    assert rc(P=257) == 2 and rc(P=-1) == 2 and rc(T=0) == 2 and rc(E=0) == 2 and rc(K=96) == 2
    assert rc(bits=3) == 3 and rc(gs=16) == 3 and rc(out=2) == 3 and rc(splits=0) == 3
    own = next(i for i, n in enumerate(binding.variant_names()) if n.startswith("tma_own"))
    assert rc(variant=own, T=17) == 3  # the row-stacking variants take at most 16 token rows
    assert rc(lhs=None) == 1 and rc(rhs=None) == 1 and rc(Y=None) == 1
    assert rc(lhs=p + 2) == 4 and rc(X=p + 8) == 4
    assert rc(P=0) == 0 and rc(N=0) == 0


def test_from_ggml_validates_on_the_host(lib):
    fake = 0x1000
    assert lib.qmm_from_ggml(3, fake, 4, 64, fake, fake, fake, None) == 3     # unknown type
    assert lib.qmm_from_ggml(0, fake, 4, 48, fake, fake, fake, None) == 2     # K not a multiple of 32
    assert lib.qmm_from_ggml(0, None, 4, 64, fake, fake, fake, None) == 1     # null input
    assert lib.qmm_from_ggml(1, fake, 4, 64, fake + 2, fake, fake, None) == 4  # misaligned Wq
    assert lib.qmm_from_ggml(2, None, 0, 64, None, None, None, None) == 0     # empty


def test_mx_validation_before_launch(lib):
    call = lib.qmm_small_m_mx
    p = 0x10000
    # (X, Wq, scales, M, N, K, format, Y, out, variant, splits, stream)
    base = [p, p, p, 4, 64, 256, 0, p, 0, -1, -1, None]
    pos = {"X": 0, "Wq": 1, "S": 2, "M": 3, "N": 4, "K": 5, "fmt": 6, "Y": 7, "out": 8, "variant": 9, "splits": 10}

    def rc(**kw):
        a = list(base)
        for k, v in kw.items():
            a[pos[k]] = v
        return call(*a)

    assert rc(M=17) == 2 and rc(K=48) == 2 and rc(fmt=3) == 3 and rc(out=3) == 3 and rc(splits=0) == 3
    tma = next(i for i, n in enumerate(binding.variant_names()) if n.startswith("tma") and "own" not in n)
    assert rc(variant=tma) == 3
    assert rc(X=None) == 1 and rc(S=None) == 1 and rc(Y=None) == 1
    assert rc(X=p + 2) == 4 and rc(Wq=p + 4) == 4
    assert rc(M=0) == 0 and rc(N=0) == 0


def test_bad_table_injection_returns_table_error(lib, monkeypatch):
    """A corrupt table entry (host-side injection) is a table error, found before
    any CUDA call (the pointers are never dereferenced)."""
    p = 0x10000
    v, s = binding.select_variant(4, 5120, 5120, 4, 64)
    assert v is not None
    monkeypatch.setenv("QMM_TEST_INJECT", "bad_table")
    assert lib.qmm_select_variant(4, 5120, 5120, 4, 64, None) == -1
    assert lib.qmm_small_m_ex(p, p, p, p, 4, 5120, 5120, 4, 64, p, 0, -1, -1, None) == 6


def test_runtime_table_file(tmp_path):
    """QMM_TABLE replaces the compiled-in table (read once per process, so the
    check runs in fresh processes); an unreadable file is a table error."""
    import subprocess
    import sys

    names = binding.variant_names()
    mma = names.index("mma_r1_wn2_wk4")
    table = tmp_path / "table.inc"
    table.write_text(f"// a one-entry table\n{{4, 5120, 5120, 4, 64, {mma}, 3}},  // forced for the test\n")
    code = ("import sys; sys.path.insert(0, {root!r}); from quantized_matmul_speculative_gb300 import binding; "
            "print(binding.select_variant(4, 5120, 5120, 4, 64), binding.select_variant(4, 4096, 4096, 4, 64))")
    root = str(Path(__file__).resolve().parents[1])
    env = dict(os.environ, QMM_TABLE=str(table))
    out = subprocess.run([sys.executable, "-c", code.format(root=root)], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    first, second = out.stdout.strip().split(") (")
    assert first == f"({mma}, 3"
    assert second.rstrip(")").split(", ")[0] != "None"  # not in the file: the rule's choice
    env["QMM_TABLE"] = str(tmp_path / "missing.inc")
    out = subprocess.run([sys.executable, "-c", code.format(root=root)], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "(None, None) (None, None)"


def test_variant_registry(lib):
    names = binding.variant_names()
    assert len(names) == lib.qmm_num_variants() >= 1
    assert lib.qmm_variant_name(len(names)) is None
    v, s = binding.select_variant(4, 5120, 5120, 4, 64)
    assert 0 <= v < len(names) and 1 <= s <= 16
    assert binding.select_variant(17, 5120, 5120, 4, 64) == (None, None)
    assert lib.qmm_status_string(4) == b"misaligned pointer"


def test_repack_validates_on_the_host(lib):
    """qmm_repack / qmm_unrepack reject bad arguments before any CUDA call (the
    pointers below are never dereferenced)."""
    fake = 0x1000  # not a valid device pointer: must not be touched on the error paths
    for fn in (lib.qmm_repack, lib.qmm_unrepack):
        assert fn(fake, 4, 64, 3, fake + 256, None) == 3      # bits not in {2,4,8}
        assert fn(fake, 4, 4, 4, fake + 256, None) == 2       # K*bits not a multiple of 32
        assert fn(fake, -1, 64, 4, fake + 256, None) == 2     # negative N
        assert fn(None, 4, 64, 4, fake, None) == 1            # null source, non-empty matrix
        assert fn(fake, 4, 64, 4, None, None) == 1            # null destination
        assert fn(None, 0, 64, 4, None, None) == 0            # empty: nothing to do
        assert fn(fake, 4, 64, 4, fake, None) == 0            # in place: the layouts coincide


def test_mx_table_names_warp_owned_choices():
    """The compiled-in microscaling table (generated from the committed
    mx_sweep) names warp-owned variants with valid split counts, its comments
    agree with the variant ids, and the 5120x5120 layer the bench times has an
    entry for every format in both activation-tile classes."""
    inc = Path(__file__).resolve().parents[1] / "quantized_matmul_speculative_gb300" / "csrc" / "qmm_mx_table.inc"
    names = binding.variant_names()
    have = set()
    for line in inc.read_text().splitlines():
        m = re.match(r"\{(\d+), (\d+), (\d+), (\d+), (-?\d+), (-?\d+)\},\s*//\s*(\S+)", line)
        if not m:
            continue
        f, M, N, K, v, s = (int(m.group(i)) for i in range(1, 7))
        assert f in (0, 1, 2) and M >= 1, line
        assert 0 <= v < len(names) and names[v].startswith("tma_own") and 1 <= s <= 16, line
        assert names[v] == m.group(7), f"table comment {m.group(7)} != variant {v} ({names[v]})"
        have.add((f, N, K, M <= 8))
    for f in (0, 1, 2):
        for small in (True, False):
            assert (f, 5120, 5120, small) in have, f"no entry for format {f}, 5120x5120, M<=8={small}"


def test_dispatch_table_covers_every_workload():
    """The compiled-in table (generated from the committed sweep) names real
    variants with valid split counts, its comments agree with the variant ids,
    and every workload shape has an entry for each activation-tile class it is
    run at (the dispatcher takes the nearest measured M of the same class)."""
    from quantized_matmul_speculative_gb300 import workloads

    inc = Path(__file__).resolve().parents[1] / "quantized_matmul_speculative_gb300" / "csrc" / "qmm_dispatch_table.inc"
    names = binding.variant_names()
    entries = {}
    for line in inc.read_text().splitlines():
        m = re.match(r"\{(-?\d+), (\d+), (\d+), (\d+), (\d+), (-?\d+), (-?\d+)\},\s*//\s*(\S+)", line)
        if not m:
            continue
        M, N, K, bits, gs, v, s = (int(m.group(i)) for i in range(1, 8))
        if v < 0:
            continue  # the sentinel
        assert 0 <= v < len(names) and 1 <= s <= 16, line
        assert names[v] == m.group(8), f"table comment {m.group(8)} != variant {v} ({names[v]})"
        entries.setdefault((N, K, bits, gs), set()).add(M <= 8)
    for w in workloads.ALL:
        for sh in w.shapes:
            for bits, gs in (w.variants or ((w.bits, w.group_size),)):
                classes = {M <= 8 for M in w.ms}
                have = entries.get((sh.N, sh.K, bits, gs), set())
                assert classes <= have, f"{w.name} {sh.name} {bits}b g{gs}: table lacks M classes {classes - have}"
                for M in w.ms:
                    v, s = binding.select_variant(M, sh.N, sh.K, bits, gs)
                    assert v is not None and 1 <= s <= 16
