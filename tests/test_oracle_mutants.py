"""Plant plausible mistakes in copies of the oracle source and check that the
pins catch every one of them (CPU only; the real oracle is never modified)."""
import pytest

import oracle_pins
from oracle import oracle

# (name, text in the oracle source, replacement): a wrong sign, a dropped
# term, swapped operands, a reversed code order, a wrong group index, a
# reversed k index, a dropped absolute value, an off-by-one in the decoders.
MUTANTS = [
    ("bias_sign", "return s * q + b;", "return s * q - b;"),
    ("bias_dropped", "return s * q + b;", "return s * q;"),
    ("scale_bias_swapped", "return s * q + b;", "return b * q + s;"),
    ("code_order_reversed", "bits * (k % per_word)", "bits * (per_word - 1 - k % per_word)"),
    ("group_index", "S[n * groups + k / g]", "S[n * groups + (k / g + 1) % groups]"),
    ("k_reversed", "xm[k] * w[k]", "xm[k] * w[K - 1 - k]"),
    ("abs_dropped", "a += std::fabs(p);\n      }\n      Y[m * N + n] = y;", "a += p;\n      }\n      Y[m * N + n] = y;"),
    ("half_bias", "expo - 25", "expo - 24"),
    ("bf16_frac", "128 + frac), expo - 134", "127 + frac), expo - 134"),
    ("residual_sign", "Y[i] = r + Y[i];", "Y[i] = Y[i] - r;"),
    ("residual_dropped_from_scale", "A[i] = std::fabs(r) + A[i];", "A[i] = A[i];"),
    ("gather_rhs_ignored", "const int64_t t = lhs[i], e = rhs[i];", "const int64_t t = lhs[i], e = 0;"),
    ("gather_lhs_ignored", "const int64_t t = lhs[i], e = rhs[i];", "const int64_t t = i % T, e = rhs[i];"),
    ("ggml_nibble_order", "(e < 16) ? (qs[e] & 15) : (qs[e - 16] >> 4)", "(e < 16) ? (qs[e] >> 4) : (qs[e - 16] & 15)"),
    ("ggml_q4_0_offset", "w = d * static_cast<double>(c - 8);", "w = d * static_cast<double>(c);"),
    ("ggml_q8_sign", "static_cast<int8_t>(blk[2 + e])", "static_cast<uint8_t>(blk[2 + e])"),
    ("e2m1_exponent_bias", "std::ldexp(1.0 + 0.5 * m, e - 1)", "std::ldexp(1.0 + 0.5 * m, e - 2)"),
    ("e4m3_subnormal", "std::ldexp(m / 8.0, -6)", "std::ldexp(m / 8.0, -7)"),
    ("e8m0_bias", "static_cast<int>(e) - 127", "static_cast<int>(e) - 128"),
    ("nvfp4_group", "const int64_t g = format == 2 ? 16 : 32;", "const int64_t g = 32;"),
    ("dequant_transposed", "W[n * K + k] = weight_at(Wq, S, B, K, bits, g, n, k);",
     "W[k * N + n] = weight_at(Wq, S, B, K, bits, g, n, k);"),
    ("gather_expert_stride", "const int64_t words_per_matrix = N * (K * bits / 32);",
     "const int64_t words_per_matrix = K * bits / 32;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = oracle.SOURCE.read_text()
    assert old in src, f"mutation site for {name} not found"
    mutant = tmp_path / f"mutant_{name}.cpp"
    mutant.write_text(src.replace(old, new, 1))
    lib = oracle.OracleLib(oracle.compile_source(mutant, tmp_path / f"lib_{name}.so"))
    caught = []
    for pin in oracle_pins.FAST_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception as exc:  # an error return from the mutant also counts as caught
            caught.append(f"{pin.__name__}:{type(exc).__name__}")
    assert caught, f"mutant {name} passed every pin"
