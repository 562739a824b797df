// Oracle for the small-M affine-quantized matrix multiply
//     Y[M,N] = X[M,K] · dequant(Wq, scales, biases)[N,K]^T
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
// definition that the CUDA library is checked against.  Only the tests, the
// smoke check and the benchmark's CPU-baseline leg may build, load or call it.
// It shares no code, header, table or helper with the CUDA library, and the
// library never calls it: there is no CPU fallback anywhere in the product.
//
// Arithmetic: IEEE binary64, single thread, every sum over k in ascending
// order, compiled with -O2 -ffp-contract=off (no fused multiply-add, no
// fast-math).
//
// What is computed, and where the pages say so:
//  * Affine group quantization, w = scale * q + bias, one fp16 scale and one
//    fp16 bias per group of `group_size` weights along K.
//      - "MLX quantized_matmul small-M verify kernels", fact "Fix family 1"
//        (the affine mode of qmv_wide) and fact "Group-size mechanism" (4 B of
//        scale+bias per group: 2 B fp16 scale + 2 B fp16 bias).
//  * W is stored [N,K] and the product is X · W^T:
//      - same page, fact "Microbench": (M,5120)@(17408,5120)^T.
//  * bf16 activations:
//      - same page, facts "qmv_wide speedup" ("bf16 act") and "Fix family 2"
//        ("load A straight from device bf16").
//  * Packing of q into 32-bit words.  The pages print no bit layout.  The
//    reading adopted is the plainest one: little-endian uint32 words, rows of
//    W contiguous along K, codes low-bits-first inside each word, i.e. for
//    b-bit codes word j of row n holds k = j*(32/b) ... j*(32/b) + 32/b - 1 and
//    code k sits at bit offset b * (k mod (32/b)).
//  * Unsigned codes 0 .. 2^b - 1; "affine" adds the bias, there is no other
//    zero point.
//  * Code widths b = 2, 4 and 8.  The 8-bit affine mode is the same
//    definition with four codes per word:
//      - "MLX quantized_matmul small-M verify kernels", facts "qmv_wide
//        speedup" (int8 at M=8) and "mlx-dspark skinny_qmm" (widths 6-16 at
//        8-bit).
//  * Fused residual add (oracle_qmm_residual): Y = R + X · W^T, the sum that
//    a MUL_MAT + ADD fusion writes from the matmul's store.
//      - "metal : few-row MMA mat-mul and batched copies for speculative
//        decoding" (llama.cpp PR #29869), Overview: the fusion-table entry
//        MUL_MAT + ADD.
//  * Gathered product (oracle_gather_qmm), the MoE form of the op at verify
//    widths: entry i of a list pairs activation row lhs[i] with expert matrix
//    rhs[i] of a stack W[E][N][K]: Y[i, n] = sum_k x[lhs[i], k] * w[rhs[i], n, k].
//      - "MLX quantized_matmul small-M verify kernels", the open question on
//        "dense and MoE (gather_qmm) verify" and the "expert-union cost per
//        verify row".
//  * ggml block formats Q4_0, Q4_1 and Q8_0 (oracle_ggml_dequant, _qmm): blocks
//    of 32 weights along K, each row of W a run of K/32 blocks.  The pages name
//    the formats without their byte layout ("metal : few-row MMA mat-mul ...",
//    Overview: Q4_0, Q8_0 and Q4_1 kernels); the reading used is the public
//    ggml layout:
//      Q4_0, 18 bytes: fp16 d, then 16 bytes of 4-bit codes c; byte j holds
//            element j in its low nibble and element j + 16 in its high one;
//            w = d * (c - 8).
//      Q4_1, 20 bytes: fp16 d, fp16 m, then the 16 code bytes as in Q4_0;
//            w = d * c + m.
//      Q8_0, 34 bytes: fp16 d, then 32 signed bytes q; w = d * q.
//  * Microscaling fp modes (oracle_mx_dequant, _qmm): groups of 32 codes
//    along K share one 8-bit power-of-two scale.  The pages list the modes
//    ("MLX quantized_matmul small-M verify kernels", facts "Fix family 1" and
//    "qmv_wide covers affine, nvfp4, mxfp4, mxfp8"); the element and scale
//    encodings are the OCP microscaling ones:
//      codes  mxfp4: FP4 E2M1, 4 bits (sign, 2 exponent bits with bias 1, 1
//             mantissa bit): 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives;
//             packed 8 per word like the 4-bit affine codes.
//             mxfp8: FP8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa
//             bits; exponent 0 is subnormal; S.1111.111 is NaN, no infinity);
//             packed 4 per word like the 8-bit affine codes.
//      scale  E8M0, one byte per (row, group of 32): 2^(E - 127), 255 = NaN;
//             stored [N, K/32].
//    nvfp4: FP4 E2M1 codes as mxfp4, groups of 16 with an FP8 E4M3 scale
//    byte each, stored [N, K/16] (a per-tensor scale, where a model has one,
//    is left to the caller).
//    w = scale * value(code).
//
// Parity pins (tests/test_oracle_pins.py): exact rational brute force on tiny
// shapes (2-, 4- and 8-bit), closed forms (all-zero codes, one-hot X, X = 1,
// saturated codes), the scale=1/bias=0 special case against numpy's integer
// matmul, linearity, row-permutation and batch invariance, the documented
// pack words, and the residual form.

#include <cmath>
#include <cstdint>
#include <vector>

namespace {

// binary16 -> binary64, written out from the IEEE 754 binary16 format:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double half_bits_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1F;
  const int frac = h & 0x3FF;
  double mag;
  if (expo == 0) {
    mag = std::ldexp(static_cast<double>(frac), -24);              // subnormal: frac * 2^-24
  } else if (expo == 31) {
    mag = frac == 0 ? INFINITY : NAN;
  } else {
    mag = std::ldexp(static_cast<double>(1024 + frac), expo - 25); // (1 + frac/1024) * 2^(expo-15)
  }
  return sign ? -mag : mag;
}

// bfloat16 -> binary64: bfloat16 is the upper half of a binary32 pattern
// (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits).
double bf16_bits_to_double(uint16_t b) {
  const int sign = (b >> 15) & 1;
  const int expo = (b >> 7) & 0xFF;
  const int frac = b & 0x7F;
  double mag;
  if (expo == 0) {
    mag = std::ldexp(static_cast<double>(frac), -133);              // frac * 2^-7 * 2^-126
  } else if (expo == 255) {
    mag = frac == 0 ? INFINITY : NAN;
  } else {
    mag = std::ldexp(static_cast<double>(128 + frac), expo - 134);  // (1 + frac/128) * 2^(expo-127)
  }
  return sign ? -mag : mag;
}

bool bits_ok(int bits) { return bits == 2 || bits == 4 || bits == 8; }

// Code k of row n, read straight from the packed words.
inline unsigned code_at(const uint32_t* Wq, int64_t words_per_row, int64_t n, int64_t k, int bits) {
  const int64_t per_word = 32 / bits;
  const uint32_t word = Wq[n * words_per_row + k / per_word];
  const unsigned shift = static_cast<unsigned>(bits * (k % per_word));
  const uint32_t mask = (1u << bits) - 1u;
  return (word >> shift) & mask;
}

// Dequantized weight w[n,k] = scale[n, k/g] * q[n,k] + bias[n, k/g].
inline double weight_at(const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
                        int64_t K, int bits, int64_t g, int64_t n, int64_t k) {
  const int64_t words_per_row = K * bits / 32;
  const int64_t groups = K / g;
  const double s = half_bits_to_double(S[n * groups + k / g]);
  const double b = half_bits_to_double(B[n * groups + k / g]);
  const double q = static_cast<double>(code_at(Wq, words_per_row, n, k, bits));
  return s * q + b;
}

int check_shape(int64_t M, int64_t N, int64_t K, int bits, int64_t g) {
  if (M < 0 || N < 0 || K < 0) return 2;
  if (!bits_ok(bits)) return 3;
  if (g <= 0) return 3;
  if (K % g != 0) return 2;
  if ((K * bits) % 32 != 0) return 2;
  return 0;
}

}  // namespace

extern "C" {

double oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }
double oracle_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

// Pack codes q[N,K] (one code per byte, each < 2^bits) into words Wq[N, K*bits/32].
// Returns 0, or non-zero for an unsupported bit width / shape / out-of-range code.
int oracle_pack(const uint8_t* q, int64_t N, int64_t K, int bits, uint32_t* Wq) {
  if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 32 != 0) return 2;
  const int64_t per_word = 32 / bits;
  const int64_t words_per_row = K / per_word;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < words_per_row; ++j) {
      uint32_t word = 0;
      for (int64_t i = 0; i < per_word; ++i) {
        const uint32_t code = q[n * K + j * per_word + i];
        if (code >> bits) return 3;
        word |= code << (bits * i);
      }
      Wq[n * words_per_row + j] = word;
    }
  }
  return 0;
}

// Inverse of oracle_pack.
int oracle_unpack(const uint32_t* Wq, int64_t N, int64_t K, int bits, uint8_t* q) {
  if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 32 != 0) return 2;
  const int64_t words_per_row = K * bits / 32;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      q[n * K + k] = static_cast<uint8_t>(code_at(Wq, words_per_row, n, k, bits));
  return 0;
}

// Full product.  X: bf16 bit patterns [M,K]; Wq: packed [N, K*bits/32];
// S, B: fp16 bit patterns [N, K/g].  Writes Y[M,N] = sum_k x*w and
// A[M,N] = sum_k |x*w| (the scale the tolerance is stated against), both fp64.
// A may be null.  Each row of W is dequantized once into fp64 and reused for
// all M rows of X; every sum still runs over k in ascending order.
int oracle_qmm(const uint16_t* X, const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
               int64_t M, int64_t N, int64_t K, int bits, int64_t g, double* Y, double* A) {
  const int rc = check_shape(M, N, K, bits, g);
  if (rc) return rc;
  std::vector<double> x(static_cast<size_t>(M * K));
  for (int64_t i = 0; i < M * K; ++i) x[i] = bf16_bits_to_double(X[i]);
  std::vector<double> w(static_cast<size_t>(K));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) w[k] = weight_at(Wq, S, B, K, bits, g, n, k);
    for (int64_t m = 0; m < M; ++m) {
      const double* xm = x.data() + m * K;
      double y = 0.0, a = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = xm[k] * w[k];
        y += p;
        a += std::fabs(p);
      }
      Y[m * N + n] = y;
      if (A) A[m * N + n] = a;
    }
  }
  return 0;
}

// Y = R + X · dequant(W)^T.  R[M,N] is given as bf16 bit patterns (r_is_f32 = 0,
// uint16) or as binary32 values (r_is_f32 = 1, float).  The product is the
// sum over k in ascending order as in oracle_qmm, then r is added; A = |r| +
// sum_k |x*w| (the tolerance scale of the rounded sum).
int oracle_qmm_residual(const uint16_t* X, const uint32_t* Wq, const uint16_t* S, const uint16_t* B, const void* R,
                        int r_is_f32, int64_t M, int64_t N, int64_t K, int bits, int64_t g, double* Y, double* A) {
  const int rc = oracle_qmm(X, Wq, S, B, M, N, K, bits, g, Y, A);
  if (rc) return rc;
  for (int64_t i = 0; i < M * N; ++i) {
    const double r = r_is_f32 ? static_cast<double>(static_cast<const float*>(R)[i])
                              : bf16_bits_to_double(static_cast<const uint16_t*>(R)[i]);
    Y[i] = r + Y[i];
    if (A) A[i] = std::fabs(r) + A[i];
  }
  return 0;
}

// Gathered product.  W is a stack of E matrices: Wq [E][N][K*bits/32], S, B
// [E][N][K/g].  lhs[i] in 0..T-1 selects the activation row, rhs[i] in 0..E-1
// the matrix.  Y[P,N], A[P,N] as in oracle_qmm.  Returns 2 for an index out
// of range.
int oracle_gather_qmm(const uint16_t* X, const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
                      const int32_t* lhs, const int32_t* rhs, int64_t P, int64_t T, int64_t E, int64_t N,
                      int64_t K, int bits, int64_t g, double* Y, double* A) {
  const int rc = check_shape(T, N, K, bits, g);
  if (rc) return rc;
  if (P < 0 || E < 0) return 2;
  const int64_t words_per_matrix = N * (K * bits / 32);
  const int64_t groups_per_matrix = N * (K / g);
  for (int64_t i = 0; i < P; ++i) {
    const int64_t t = lhs[i], e = rhs[i];
    if (t < 0 || t >= T || e < 0 || e >= E) return 2;
    const uint32_t* We = Wq + e * words_per_matrix;
    const uint16_t* Se = S + e * groups_per_matrix;
    const uint16_t* Be = B + e * groups_per_matrix;
    for (int64_t n = 0; n < N; ++n) {
      double y = 0.0, a = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = bf16_bits_to_double(X[t * K + k]) * weight_at(We, Se, Be, K, bits, g, n, k);
        y += p;
        a += std::fabs(p);
      }
      Y[i * N + n] = y;
      if (A) A[i * N + n] = a;
    }
  }
  return 0;
}

// ggml blocks: type 0 = Q4_0, 1 = Q4_1, 2 = Q8_0 (layouts in the header
// comment).  Dequantized W[N,K] in fp64; returns 2 for a bad shape or type.
int oracle_ggml_dequant(int type, const uint8_t* blocks, int64_t N, int64_t K, double* W) {
  if (type < 0 || type > 2 || N < 0 || K < 0 || K % 32 != 0) return 2;
  const int64_t bytes = type == 0 ? 18 : type == 1 ? 20 : 34;
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (n * nb + b) * bytes;
      const double d = half_bits_to_double(static_cast<uint16_t>(blk[0] | (blk[1] << 8)));
      for (int e = 0; e < 32; ++e) {
        double w;
        if (type == 2) {
          w = d * static_cast<double>(static_cast<int8_t>(blk[2 + e]));
        } else {
          const uint8_t* qs = blk + (type == 0 ? 2 : 4);
          const int c = (e < 16) ? (qs[e] & 15) : (qs[e - 16] >> 4);
          if (type == 0) {
            w = d * static_cast<double>(c - 8);
          } else {
            const double m = half_bits_to_double(static_cast<uint16_t>(blk[2] | (blk[3] << 8)));
            w = d * static_cast<double>(c) + m;
          }
        }
        W[n * K + b * 32 + e] = w;
      }
    }
  }
  return 0;
}

// Y[M,N] = X . W^T for W in ggml blocks, with A = sum |x w| (as oracle_qmm).
int oracle_ggml_qmm(int type, const uint16_t* X, const uint8_t* blocks, int64_t M, int64_t N, int64_t K, double* Y,
                    double* A) {
  if (M < 0) return 2;
  std::vector<double> W(static_cast<size_t>(N * K));
  const int rc = oracle_ggml_dequant(type, blocks, N, K, W.data());
  if (rc) return rc;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double y = 0.0, a = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = bf16_bits_to_double(X[m * K + k]) * W[n * K + k];
        y += p;
        a += std::fabs(p);
      }
      Y[m * N + n] = y;
      if (A) A[m * N + n] = a;
    }
  return 0;
}

// Microscaling element and scale decoders (layouts in the header comment).
double fp4_e2m1_to_double(unsigned c) {
  const int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -mag : mag;
}
double fp8_e4m3_to_double(unsigned c) {
  const int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  double mag;
  if (e == 15 && m == 7) mag = NAN;
  else if (e == 0) mag = std::ldexp(m / 8.0, -6);
  else mag = std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}
double e8m0_to_double(unsigned e) { return e == 255 ? NAN : std::ldexp(1.0, static_cast<int>(e) - 127); }

// format 0 = mxfp4, 1 = mxfp8, 2 = nvfp4.  W[N,K] in fp64; returns 2 for a
// bad shape or format.
int oracle_mx_dequant(int format, const uint32_t* Wq, const uint8_t* S, int64_t N, int64_t K, double* W) {
  if (format < 0 || format > 2 || N < 0 || K < 0 || K % 32 != 0) return 2;
  const int bits = format == 1 ? 8 : 4;
  const int64_t g = format == 2 ? 16 : 32;
  const int64_t words_per_row = K * bits / 32;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      const unsigned c = code_at(Wq, words_per_row, n, k, bits);
      const double v = format == 1 ? fp8_e4m3_to_double(c) : fp4_e2m1_to_double(c);
      const unsigned sb = S[n * (K / g) + k / g];
      W[n * K + k] = (format == 2 ? fp8_e4m3_to_double(sb) : e8m0_to_double(sb)) * v;
    }
  return 0;
}

// Y[M,N] = X . W^T for microscaled W, with A = sum |x w| (as oracle_qmm).
int oracle_mx_qmm(int format, const uint16_t* X, const uint32_t* Wq, const uint8_t* S, int64_t M, int64_t N,
                  int64_t K, double* Y, double* A) {
  if (M < 0) return 2;
  std::vector<double> W(static_cast<size_t>(N * K));
  const int rc = oracle_mx_dequant(format, Wq, S, N, K, W.data());
  if (rc) return rc;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double y = 0.0, a = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = bf16_bits_to_double(X[m * K + k]) * W[n * K + k];
        y += p;
        a += std::fabs(p);
      }
      Y[m * N + n] = y;
      if (A) A[m * N + n] = a;
    }
  return 0;
}

double oracle_fp4_e2m1(unsigned c) { return fp4_e2m1_to_double(c & 15); }
double oracle_fp8_e4m3(unsigned c) { return fp8_e4m3_to_double(c & 255); }
double oracle_e8m0(unsigned e) { return e8m0_to_double(e & 255); }

// The same definition evaluated only at the listed (m, n) output positions,
// for spot checks of full-size problems.
int oracle_qmm_sampled(const uint16_t* X, const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
                       int64_t M, int64_t N, int64_t K, int bits, int64_t g,
                       const int64_t* ms, const int64_t* ns, int64_t count, double* y_out, double* a_out) {
  const int rc = check_shape(M, N, K, bits, g);
  if (rc) return rc;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t m = ms[i], n = ns[i];
    if (m < 0 || m >= M || n < 0 || n >= N) return 2;
    double y = 0.0, a = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double x = bf16_bits_to_double(X[m * K + k]);
      const double w = weight_at(Wq, S, B, K, bits, g, n, k);
      const double p = x * w;
      y += p;
      a += std::fabs(p);
    }
    y_out[i] = y;
    if (a_out) a_out[i] = a;
  }
  return 0;
}

// Dequantized weight matrix W[N,K] in fp64 (used by closed-form pins).
int oracle_dequant(const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
                   int64_t N, int64_t K, int bits, int64_t g, double* W) {
  const int rc = check_shape(0, N, K, bits, g);
  if (rc) return rc;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      W[n * K + k] = weight_at(Wq, S, B, K, bits, g, n, k);
  return 0;
}

}  // extern "C"
