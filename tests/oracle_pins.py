"""Pins that tie the fp64 oracle to things other than itself.

Each ``pin_*`` takes an ``OracleLib`` and raises ``AssertionError`` when the
oracle disagrees with what the mathematics or the stated layout fixes:

* exhaustive decoders: every fp16 / bf16 bit pattern against numpy's own
  float16 / float32 conversion;
* the documented pack words (4-bit 0..7 -> 0x76543210, 2-bit 0,1,2,3 repeated
  -> 0xE4E4E4E4) and pack/unpack round trips;
* exact rational brute force (``fractions.Fraction``) on tiny shapes, written
  here from the definition w = s*q + b, y = sum_k x*w, with the codes taken
  from the generator rather than from the packed words;
* closed forms: all-zero codes, one-hot X, X = 1, saturated codes;
* the scale = 1 / bias = 0 special case against numpy's float64 matmul;
* invariants: batch invariance, exact scaling by 2, additivity over disjoint
  supports, permutation of the rows of W;
* the sampled entry point against the full one.

The same functions run against deliberately broken builds of the oracle in
``test_oracle_mutants.py``, which checks that each planted mistake trips at
least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from quantized_matmul_speculative_gb300 import synth

BF16_ONE = 0x3F80
FP16_ONE = 0x3C00


# ---------------------------------------------------------------- helpers
def frac_half(bits: int) -> Fraction:
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


def frac_bf16(bits: int) -> Fraction:
    return Fraction(float(synth.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0]))


def f64_half(a):
    return np.asarray(a, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_bf16(a):
    return synth.bf16_bits_to_f32(np.asarray(a, dtype=np.uint16)).astype(np.float64)


def close(y, ref, a, rel=1e-12, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    bad = np.abs(y - ref) > rel * np.abs(a) + 1e-300
    assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, first at {np.argwhere(bad)[0]}: {y[bad][0]} vs {ref[bad][0]}"


TINY_CASES = [
    # (M, N, K, bits, g)
    (3, 5, 64, 4, 32),
    (2, 4, 128, 4, 64),
    (1, 3, 256, 4, 128),
    (3, 4, 64, 2, 32),
    (2, 3, 128, 2, 64),
    (2, 2, 256, 2, 128),
    (2, 3, 64, 8, 32),
    (3, 2, 128, 8, 64),
    (1, 2, 256, 8, 128),
]


# ---------------------------------------------------------------- pins
def pin_decoders(lib):
    # every fp16 pattern against numpy's float16
    for h in range(0, 1 << 16, 1):
        ref = float(np.array([h], dtype=np.uint16).view(np.float16)[0])
        got = lib.half_to_double(h)
        if np.isnan(ref):
            assert np.isnan(got), f"fp16 {h:#06x}"
        else:
            assert got == ref, f"fp16 {h:#06x}: {got} vs {ref}"
    # every bf16 pattern against float32 widening
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    refs = synth.bf16_bits_to_f32(pats).astype(np.float64)
    for h in range(0, 1 << 16, 1):
        got = lib.bf16_to_double(h)
        ref = refs[h]
        if np.isnan(ref):
            assert np.isnan(got), f"bf16 {h:#06x}"
        else:
            assert got == ref, f"bf16 {h:#06x}: {got} vs {ref}"


def pin_pack_words(lib):
    q4 = np.arange(8, dtype=np.uint8).reshape(1, 8)
    assert int(lib.pack(q4, 4)[0, 0]) == 0x76543210
    q2 = np.tile(np.arange(4, dtype=np.uint8), 4).reshape(1, 16)
    assert int(lib.pack(q2, 2)[0, 0]) == 0xE4E4E4E4
    q8 = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    assert int(lib.pack(q8, 8)[0, 0]) == 0x04030201
    rng = np.random.default_rng(7)
    for bits in (2, 4, 8):
        q = rng.integers(0, 1 << bits, size=(5, 96), dtype=np.uint8)
        wq = lib.pack(q, bits)
        assert wq.shape == (5, 96 * bits // 32)
        assert np.array_equal(lib.unpack(wq, 96, bits), q)
        # the row-major word order: row 1 starts right after row 0
        flat = lib.pack(q.reshape(1, -1)[:, : 96], bits)
        assert np.array_equal(flat[0], wq[0])


def exact_product(p: synth.Problem, M: int):
    """y[m][n] and a[m][n] as Fractions, from the codes, fp16 and bf16 values."""
    g = p.group_size
    s = [[frac_half(v) for v in row] for row in p.scales]
    b = [[frac_half(v) for v in row] for row in p.biases]
    x = [[frac_bf16(v) for v in row] for row in p.x[:M]]
    ys, as_ = [], []
    for m in range(M):
        yrow, arow = [], []
        for n in range(p.N):
            acc = Fraction(0)
            mag = Fraction(0)
            for k in range(p.K):
                w = s[n][k // g] * int(p.q[n, k]) + b[n][k // g]
                t = x[m][k] * w
                acc += t
                mag += abs(t)
            yrow.append(acc)
            arow.append(mag)
        ys.append(yrow)
        as_.append(arow)
    return ys, as_


def pin_brute_force(lib):
    for i, (M, N, K, bits, g) in enumerate(TINY_CASES):
        p = synth.make_problem(900 + i, N, K, bits, g, rows=M)
        wq = lib.pack(p.q, bits)
        y, a = lib.qmm(p.x_rows(M), wq, p.scales, p.biases, bits, g)
        ye, ae = exact_product(p, M)
        for m in range(M):
            for n in range(N):
                err = abs(Fraction(float(y[m, n])) - ye[m][n])
                assert err <= Fraction(1, 10**12) * ae[m][n], f"case {i} y[{m},{n}] off by {float(err)}"
                assert abs(Fraction(float(a[m, n])) - ae[m][n]) <= Fraction(1, 10**12) * ae[m][n], f"case {i} a[{m},{n}]"


def pin_closed_forms(lib):
    for bits, g in ((4, 64), (4, 32), (2, 64), (4, 128), (8, 64), (8, 32)):
        M, N, K = 3, 6, 4 * g
        G = K // g
        p = synth.make_problem(950 + bits * 10 + g, N, K, bits, g, rows=M)
        x = f64_bf16(p.x_rows(M))
        s = f64_half(p.scales)
        b = f64_half(p.biases)
        xs = x.reshape(M, G, g).sum(axis=2)  # per-group sums of x
        # all codes zero: y = sum_g b[n,g] * sum_{k in g} x[m,k]
        q0 = np.zeros_like(p.q)
        y, a = lib.qmm(p.x_rows(M), lib.pack(q0, bits), p.scales, p.biases, bits, g)
        close(y, xs @ b.T, a, 1e-12, "all-zero codes")
        # saturated codes: w = (2^bits-1) s + b
        qs = np.full_like(p.q, (1 << bits) - 1)
        y, a = lib.qmm(p.x_rows(M), lib.pack(qs, bits), p.scales, p.biases, bits, g)
        close(y, xs @ (((1 << bits) - 1) * s + b).T, a, 1e-12, "saturated codes")
        # one-hot X picks column k0 of dequant(W)
        for k0 in (0, 1, g - 1, g, K - 1):
            xo = np.zeros((1, K), dtype=np.uint16)
            xo[0, k0] = BF16_ONE
            y, _ = lib.qmm(xo, lib.pack(p.q, bits), p.scales, p.biases, bits, g)
            col = s[:, k0 // g] * p.q[:, k0].astype(np.float64) + b[:, k0 // g]
            assert np.array_equal(y[0], col), f"one-hot k0={k0}"
        # X = 1: y = sum_k w[n,k] = sum_g (s * sum q + g * b)
        x1 = np.full((2, K), BF16_ONE, dtype=np.uint16)
        y, a = lib.qmm(x1, lib.pack(p.q, bits), p.scales, p.biases, bits, g)
        qsum = p.q.astype(np.float64).reshape(N, G, g).sum(axis=2)
        ref = (s * qsum + g * b).sum(axis=1)
        close(y[0], ref, a[0], 1e-12, "x = 1")
        close(y[1], ref, a[1], 1e-12, "x = 1")


def pin_integer_special_case(lib):
    # scale 1, bias 0: y = X @ Q^T, an integer-matrix times bf16 product
    for bits, g in ((4, 64), (2, 32), (8, 64)):
        M, N, K = 4, 7, 256
        p = synth.make_problem(970 + bits, N, K, bits, g, rows=M)
        ones = np.full(p.scales.shape, FP16_ONE, dtype=np.uint16)
        zeros = np.zeros(p.biases.shape, dtype=np.uint16)
        y, a = lib.qmm(p.x_rows(M), lib.pack(p.q, bits), ones, zeros, bits, g)
        ref = f64_bf16(p.x_rows(M)) @ p.q.astype(np.float64).T
        close(y, ref, a, 1e-12, "integer special case")


def pin_invariants(lib):
    M, N, K, bits, g = 5, 9, 320, 4, 64
    p = synth.make_problem(990, N, K, bits, g, rows=M)
    wq = lib.pack(p.q, bits)
    y, a = lib.qmm(p.x_rows(M), wq, p.scales, p.biases, bits, g)
    # batch invariance: row m of an M-row call equals the 1-row call on that row
    for m in range(M):
        y1, _ = lib.qmm(p.x[m:m + 1], wq, p.scales, p.biases, bits, g)
        assert np.array_equal(y1[0], y[m]), f"batch invariance row {m}"
    # scaling X by 2 is exact in bf16 and in the product
    x2 = (f64_bf16(p.x_rows(M)) * 2).astype(np.float32)
    y2, _ = lib.qmm(synth.f32_to_bf16_bits(x2), wq, p.scales, p.biases, bits, g)
    assert np.array_equal(y2, 2 * y), "scaling by 2"
    # additivity over disjoint supports
    xe = p.x_rows(M).copy()
    xe[:, 1::2] = 0
    xo = p.x_rows(M).copy()
    xo[:, 0::2] = 0
    ye, _ = lib.qmm(xe, wq, p.scales, p.biases, bits, g)
    yo, _ = lib.qmm(xo, wq, p.scales, p.biases, bits, g)
    close(ye + yo, y, a, 1e-13, "additivity")
    # permuting the rows of W permutes the columns of Y
    perm = np.random.default_rng(3).permutation(N)
    yp, _ = lib.qmm(p.x_rows(M), lib.pack(p.q[perm], bits), p.scales[perm], p.biases[perm], bits, g)
    assert np.array_equal(yp, y[:, perm]), "row permutation"


def pin_residual(lib):
    """Y = R + X . W^T: exact rational sums for bf16 and fp32 residuals, X = 0
    gives R exactly, R = 0 gives the plain product bit for bit."""
    M, N, K, bits, g = 2, 5, 128, 4, 32
    p = synth.make_problem(996, N, K, bits, g, rows=M)
    wq = lib.pack(p.q, bits)
    ye, ae = exact_product(p, M)
    for f32 in (False, True):
        r = synth.make_residual(996, M, N, f32=f32)
        rf = [[Fraction(float(v)) for v in row] for row in (r if f32 else synth.bf16_bits_to_f32(r))]
        y, a = lib.qmm_residual(p.x_rows(M), wq, p.scales, p.biases, r, bits, g)
        for m in range(M):
            for n in range(N):
                ref, mag = rf[m][n] + ye[m][n], abs(rf[m][n]) + ae[m][n]
                assert abs(Fraction(float(y[m, n])) - ref) <= Fraction(1, 10**12) * mag, f"residual y[{m},{n}]"
                assert abs(Fraction(float(a[m, n])) - mag) <= Fraction(1, 10**12) * mag, f"residual a[{m},{n}]"
        x0 = np.zeros_like(p.x_rows(M))
        y0, _ = lib.qmm_residual(x0, wq, p.scales, p.biases, r, bits, g)
        rr = r.astype(np.float64) if f32 else synth.bf16_bits_to_f32(r).astype(np.float64)
        assert np.array_equal(y0, rr), "X = 0 must give R"
    zero = np.zeros((M, N), dtype=np.float32)
    yz, az = lib.qmm_residual(p.x_rows(M), wq, p.scales, p.biases, zero, bits, g)
    yp, ap = lib.qmm(p.x_rows(M), wq, p.scales, p.biases, bits, g)
    assert np.array_equal(yz, yp) and np.array_equal(az, ap), "R = 0 must give the plain product"


def pin_gather(lib):
    """Y[i] = X[lhs[i]] . W[rhs[i]]^T: exact rational sums on a tiny stack with a
    repeated entry; relabelling the experts leaves Y unchanged; an index out of
    range is an error."""
    E, N, K, bits, g, T = 3, 4, 64, 4, 32, 3
    mp = synth.make_moe(997, E, N, K, bits, g, T, 2)
    wq = np.stack([lib.pack(mp.q[e], bits) for e in range(E)])
    lhs = np.array([0, 2, 1, 2, 0, 1], dtype=np.int32)
    rhs = np.array([2, 0, 1, 2, 1, 2], dtype=np.int32)
    y, a = lib.gather_qmm(mp.x[:T], wq, mp.scales, mp.biases, lhs, rhs, bits, g)
    s = [[[frac_half(v) for v in row] for row in mp.scales[e]] for e in range(E)]
    b = [[[frac_half(v) for v in row] for row in mp.biases[e]] for e in range(E)]
    x = [[frac_bf16(v) for v in row] for row in mp.x[:T]]
    for i in range(len(lhs)):
        t, e = int(lhs[i]), int(rhs[i])
        for n in range(N):
            acc, mag = Fraction(0), Fraction(0)
            for k in range(K):
                term = x[t][k] * (s[e][n][k // g] * int(mp.q[e, n, k]) + b[e][n][k // g])
                acc += term
                mag += abs(term)
            assert abs(Fraction(float(y[i, n])) - acc) <= Fraction(1, 10**12) * mag, f"gather y[{i},{n}]"
            assert abs(Fraction(float(a[i, n])) - mag) <= Fraction(1, 10**12) * mag, f"gather a[{i},{n}]"
    perm = np.array([2, 0, 1])  # new expert j is old expert perm[j]
    inv = np.argsort(perm).astype(np.int32)
    y2, _ = lib.gather_qmm(mp.x[:T], wq[perm], mp.scales[perm], mp.biases[perm], lhs, inv[rhs], bits, g)
    assert np.array_equal(y2, y), "relabelled experts"
    bad = rhs.copy()
    bad[3] = E
    try:
        lib.gather_qmm(mp.x[:T], wq, mp.scales, mp.biases, lhs, bad, bits, g)
    except Exception:
        pass
    else:
        raise AssertionError("an expert index out of range must be an error")


def pin_ggml(lib):
    """ggml blocks decoded per the format: constructed blocks whose weights are
    known by construction (nibble order, the Q4_0 offset 8, Q4_1's m, Q8_0's
    sign), the row-major block order, and the product against the dequantized
    matrix (one-hot X picks a column, X = 1 sums a row)."""
    j = np.arange(16)
    qs4 = (j | ((15 - j) << 4)).astype(np.uint8)         # element e<16: e; element 16+e: 15-e
    codes = np.concatenate([j, 15 - j]).astype(np.float64)
    one, half, m2, quarter = (np.array([v], dtype=np.float16).view(np.uint8) for v in (1.0, 0.5, -2.0, 0.25))
    b40 = np.concatenate([one, qs4])
    assert np.array_equal(lib.ggml_dequant("q4_0", b40, 1, 32)[0], codes - 8), "Q4_0"
    b41 = np.concatenate([half, m2, qs4])
    assert np.array_equal(lib.ggml_dequant("q4_1", b41, 1, 32)[0], 0.5 * codes - 2.0), "Q4_1"
    q8 = (np.arange(32) * 8 - 128).astype(np.int8)
    b80 = np.concatenate([quarter, q8.view(np.uint8)])
    assert np.array_equal(lib.ggml_dequant("q8_0", b80, 1, 32)[0], 0.25 * q8.astype(np.float64)), "Q8_0"
    # two rows of two blocks: block (n, b) is the (2n + b)-th, its d = 2^(2n + b)
    blocks = []
    for i in range(4):
        d = np.array([2.0 ** i], dtype=np.float16).view(np.uint8)
        blocks.append(np.concatenate([d, q8.view(np.uint8)]))
    w = lib.ggml_dequant("q8_0", np.concatenate(blocks), 2, 64)
    for n in range(2):
        for b in range(2):
            assert np.array_equal(w[n, 32 * b:32 * b + 32], 2.0 ** (2 * n + b) * q8), f"block order ({n},{b})"
    for kind in ("q4_0", "q4_1", "q8_0"):
        N, K = 5, 96
        blk = synth.make_ggml_blocks(998, N, K, kind)
        W = lib.ggml_dequant(kind, blk, N, K)
        for k0 in (0, 15, 16, 31, 32, 95):
            xo = np.zeros((1, K), dtype=np.uint16)
            xo[0, k0] = BF16_ONE
            y, _ = lib.ggml_qmm(kind, xo, blk, N)
            assert np.array_equal(y[0], W[:, k0]), f"{kind} one-hot {k0}"
        y, a = lib.ggml_qmm(kind, np.full((1, K), BF16_ONE, dtype=np.uint16), blk, N)
        close(y[0], W.sum(axis=1), a[0], 1e-12, f"{kind} x = 1")


def pin_mx(lib):
    """Microscaling decoders against the OCP tables and independent rational
    formulas; the product against exact rational sums; one-hot X."""
    f4, f8, e8 = lib.mx_decoders()
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        ref = e2m1[c & 7] * (-1.0 if c & 8 else 1.0)
        assert f4(c) == ref and np.signbit(f4(c)) == bool(c & 8), f"e2m1 {c}"
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(f8(c)), f"e4m3 {c:#x} is NaN"
            continue
        mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(f8(c)) == (-mag if s else mag), f"e4m3 {c:#x}"
    assert f8(0x7E) == 448.0 and f8(0x01) == 2.0 ** -9 and f8(0x08) == 2.0 ** -6 and f8(0x38) == 1.0
    assert e8(127) == 1.0 and e8(0) == 2.0 ** -127 and e8(254) == 2.0 ** 127 and np.isnan(e8(255))
    for fmt, bits in (("mxfp4", 4), ("mxfp8", 8), ("nvfp4", 4)):
        M, N, K = 2, 3, 64
        q, sc = synth.make_mx(999, N, K, fmt)
        wq = lib.pack(q, bits)
        xb = synth.make_x(999, K, rows=M)
        y, a = lib.mx_qmm(fmt, xb, wq, sc)
        dec = f8 if fmt == "mxfp8" else f4
        g = 16 if fmt == "nvfp4" else 32

        def scale(n, k):
            b = int(sc[n, k // g])
            if fmt != "nvfp4":
                return Fraction(2) ** (b - 127)
            return (1 + Fraction(b & 7, 8)) * Fraction(2) ** (((b >> 3) & 15) - 7)  # normal, positive by draw

        xs = [[frac_bf16(v) for v in row] for row in xb]
        for m in range(M):
            for n in range(N):
                acc, mag = Fraction(0), Fraction(0)
                for k in range(K):
                    t = xs[m][k] * scale(n, k) * Fraction(dec(int(q[n, k])))
                    acc += t
                    mag += abs(t)
                assert abs(Fraction(float(y[m, n])) - acc) <= Fraction(1, 10**12) * mag, f"{fmt} y[{m},{n}]"
                assert abs(Fraction(float(a[m, n])) - mag) <= Fraction(1, 10**12) * mag, f"{fmt} a[{m},{n}]"
        W = lib.mx_dequant(fmt, wq, sc, K)
        for k0 in (0, 31, 32, 63):
            xo = np.zeros((1, K), dtype=np.uint16)
            xo[0, k0] = BF16_ONE
            yo, _ = lib.mx_qmm(fmt, xo, wq, sc)
            assert np.array_equal(yo[0], W[:, k0]), f"{fmt} one-hot {k0}"


def pin_dequant(lib):
    """oracle_dequant against the definition w[n, k] = s[n, k/g] * q[n, k] + b[n, k/g]
    written out with exact rationals from the generator's codes (not the packed
    words), on shapes with N != K so that a transposed or mis-strided write shows;
    and each column of it against the one-hot product of oracle_qmm."""
    for i, (bits, g, N, K) in enumerate(((4, 64, 3, 128), (4, 32, 5, 96), (2, 64, 4, 192), (8, 32, 2, 64),
                                         (4, 128, 7, 256))):
        p = synth.make_problem(1100 + i, N, K, bits, g, rows=1)
        W = lib.dequant(lib.pack(p.q, bits), p.scales, p.biases, K, bits, g)
        assert W.shape == (N, K), f"dequant shape {W.shape}"
        for n in range(N):
            for k in range(K):
                exact = frac_half(int(p.scales[n, k // g])) * int(p.q[n, k]) + frac_half(int(p.biases[n, k // g]))
                assert Fraction(float(W[n, k])) == exact, f"dequant ({bits}-bit g{g}) w[{n},{k}]"
        wq = lib.pack(p.q, bits)
        for k0 in (0, g - 1, g, K - 1):
            xo = np.zeros((1, K), dtype=np.uint16)
            xo[0, k0] = BF16_ONE
            y, _ = lib.qmm(xo, wq, p.scales, p.biases, bits, g)
            assert np.array_equal(y[0], W[:, k0]), f"dequant column {k0} vs one-hot product"
    # hand-built: codes 0..7 along one 4-bit row, scale 2, bias -1 -> w = 2q - 1
    q = np.arange(64, dtype=np.uint8).reshape(1, 64) % 16
    s = np.full((1, 1), 0x4000, dtype=np.uint16)   # fp16 2.0
    b = np.full((1, 1), 0xBC00, dtype=np.uint16)   # fp16 -1.0
    W = lib.dequant(lib.pack(q, 4), s, b, 64, 4, 64)
    assert np.array_equal(W[0], 2.0 * q[0].astype(np.float64) - 1.0), "hand-built dequant row"


def pin_sampled(lib):
    M, N, K, bits, g = 4, 11, 192, 2, 64
    p = synth.make_problem(995, N, K, bits, g, rows=M)
    wq = lib.pack(p.q, bits)
    y, a = lib.qmm(p.x_rows(M), wq, p.scales, p.biases, bits, g)
    ms = np.array([0, 3, 1, 2, 3])
    ns = np.array([0, 10, 5, 7, 0])
    ys, as_ = lib.qmm_sampled(p.x_rows(M), wq, p.scales, p.biases, bits, g, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


# Pins that run fast enough for the mutation test (the exhaustive decoder pin
# is run once against the real oracle only).
FAST_PINS = (pin_pack_words, pin_brute_force, pin_closed_forms, pin_integer_special_case,
             pin_invariants, pin_dequant, pin_residual, pin_gather, pin_ggml, pin_mx, pin_sampled)
ALL_PINS = (pin_decoders,) + FAST_PINS
