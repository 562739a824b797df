/*
 * qmm.h -- C ABI of libqmm: the small-M affine-quantized matrix multiply
 *
 *     Y[M,N] = X[M,K] . dequant(Wq, scales, biases)[N,K]^T,   1 <= M <= 16
 *
 * that a speculative-decoding verify step issues with a handful of draft rows.
 * The library streams the packed weights from HBM once per call whatever M is,
 * dequantizes each weight group once and reuses it for all M rows.
 *
 * Sources of the definition (page title, section):
 *   - "MLX quantized_matmul small-M verify kernels", fact "Stock qmv streams
 *     the weight matrix once per input row": the problem (cost linear in M).
 *   - same page, fact "Fix family 1": dequantize each group once into
 *     registers and reuse it across the M rows; affine mode.
 *   - same page, fact "Fix family 2": weights as the matrix operand, split K
 *     across the warps of a block, read the bf16 activations directly.
 *   - same page, fact "Group-size mechanism": fp16 scale + fp16 bias per group
 *     (4 bytes per group).
 *   - same page, fact "Microbench": W is stored [N,K] and Y = X . W^T.
 *
 * Data formats (all row-major, all buffers owned by the caller):
 *   X       bf16 [M, K]                         device
 *   Wq      uint32 [N, K*bits/32]               device
 *           code k of row n sits in word k/(32/bits) of that row at bit
 *           offset bits*(k mod (32/bits)); codes are unsigned 0..2^bits-1,
 *           bits = 2, 4 or 8.  (The pages print no bit layout; this is the
 *           layout qmm_pack writes.  8-bit affine: same page, facts
 *           "qmv_wide speedup" (int8 at M=8) and "mlx-dspark skinny_qmm".)
 *   scales  fp16 [N, K/group_size]              device
 *   biases  fp16 [N, K/group_size]              device
 *           w[n,k] = scales[n, k/g] * q[n,k] + biases[n, k/g]
 *   Y       bf16 (round to nearest even) or fp32 [M, N]    device
 *
 * Arithmetic: codes are exact in bf16 and their products with bf16 X are
 * exact in fp32; sums are fp32; each group's scale and bias are applied once
 * to the group's fp32 partial sums.  Results are deterministic for a given
 * (variant, splits, shape): no atomics, fixed reduction order.
 *
 * Execution: every compute call is asynchronous on `stream` (a cudaStream_t
 * passed as void*, 0 = legacy default stream).  Arguments are validated on the
 * host before anything is launched; a validation failure returns an error and
 * launches nothing.  There is no CPU fallback.  The library allocates no device
 * memory and keeps no per-call state.  X, Wq, scales, biases must not overlap Y.
 */
#ifndef QMM_H_
#define QMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QMM_OK = 0,
  QMM_ERR_NULL = 1,        /* a required pointer is null                          */
  QMM_ERR_SHAPE = 2,       /* M outside 0..16, N or K negative, K not a multiple   */
                           /* of group_size, a size that overflows, or a residual  */
                           /* that partly overlaps Y                               */
  QMM_ERR_UNSUPPORTED = 3, /* bits not in {2,4,8}, group_size not in {32,64,128},  */
                           /* unknown variant, bad split count or output dtype     */
  QMM_ERR_ALIGN = 4,       /* X or Wq not 16-byte aligned, scales/biases/Y not     */
                           /* aligned to their element size                        */
  QMM_ERR_CUDA = 5,        /* the CUDA runtime reported an error; see               */
                           /* qmm_last_cuda_error()                                 */
  QMM_ERR_TABLE = 6        /* the dispatch table is unusable: the QMM_TABLE file    */
                           /* cannot be read or holds no entry, or the shape's     */
                           /* entry names an unknown variant or split count        */
} qmm_status;

typedef enum { QMM_OUT_BF16 = 0, QMM_OUT_F32 = 1 } qmm_out_dtype;

/* Y = X . dequant(W)^T with the variant the dispatch table picks for
 * (M, N, K, bits, group_size); bf16 output.
 * M == 0 or N == 0: nothing to compute, returns QMM_OK without launching.
 * K == 0: Y is the empty sum, filled with zeros on `stream`.                    */
qmm_status qmm_small_m(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                       int M, int N, int K, int bits, int group_size, void* Y, void* stream);

/* Same, with the output dtype and an optional forced kernel variant
 * (variant = -1: dispatch table; 0 .. qmm_num_variants()-1: that variant) and
 * the number of CTAs that split K inside one thread-block cluster (splits = -1:
 * the table's or the variant's default; 1..16 otherwise).  A (variant, splits)
 * pair the shape cannot use returns QMM_ERR_UNSUPPORTED and launches nothing:
 * the "tma" variants need K/group_size (G) to be a multiple of splits and
 * 16-byte aligned scales and biases; the row-stacking "tma_w*" ones also need
 * G to be a multiple of 8, the warp-owned "tma_own_*" ones take other G when
 * N*G is a multiple of 8 and G <= 128 (each stage then holds its tile's scales
 * and biases for all G groups), shared memory permitting.                     */
qmm_status qmm_small_m_ex(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                          int M, int N, int K, int bits, int group_size, void* Y,
                          int out_dtype, int variant, int splits, void* stream);

/* Fused residual add: Y = R + X . dequant(W)^T.  R has Y's dtype and layout
 * ([M, N], bf16 or fp32 per out_dtype) and is added to the fp32 result in the
 * kernel's store, before the single rounding to Y's dtype; R may be Y itself
 * (an in-place update of a residual stream) but must not otherwise overlap it.
 * Other arguments, errors and dispatch as qmm_small_m_ex; R == NULL with a
 * non-empty output returns QMM_ERR_NULL.  K == 0 gives Y = R.
 * Source: "metal : few-row MMA mat-mul and batched copies for speculative
 * decoding" (llama.cpp PR #29869), Overview: a fusion-table entry for
 * MUL_MAT + ADD writes the residual sum from the MMA store.                    */
qmm_status qmm_small_m_residual(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                                const void* R, int M, int N, int K, int bits, int group_size, void* Y,
                                int out_dtype, int variant, int splits, void* stream);

/* Gathered form for mixture-of-experts layers at verify widths:
 *     Y[i, :] = X[lhs[i], :] . dequant(W[rhs[i]])^T,   i = 0 .. P-1
 * X bf16 [T, K]; Wq [E][N][K*bits/32], scales and biases fp16 [E][N][K/g]: a
 * stack of E matrices back to back, each in the layout above; lhs, rhs int32
 * [P] device arrays, 0 <= lhs[i] < T, 0 <= rhs[i] < E; Y [P, N].  Each expert
 * in the union of rhs is streamed once per call for all the entries that name
 * it.  P <= 256.  On the mma variants, entries per expert: at most 8 if
 * T <= 8 or P <= 8, else at most 16 (true when the k experts of each token
 * are distinct and T <= 16).
 * Source: "MLX quantized_matmul small-M verify kernels", the open question on
 * "dense and MoE (gather_qmm) verify" and the "expert-union cost per verify
 * row".
 * variant = -1: with T <= 16 and a shape the "tma_own" variants take (see
 * qmm_small_m_ex), the warp-owned kernel (the first cluster size of 1, 2, 4, 8
 * that plans) computes all T rows against each expert of the union and writes
 * the rows the entries name (then any number of entries per expert is fine);
 * otherwise the "mma" variants take each
 * expert's own entries.  A forced "tma" or "tma_own" variant takes the first
 * way (QMM_ERR_UNSUPPORTED if it cannot), a forced "mma" variant the second.
 * splits as in qmm_small_m_ex.  The index
 * lists are read on the device, after the wait for the preceding kernel: an
 * index out of range, or (mma variants) too many entries for one expert,
 * leaves the affected rows of Y unwritten and sets bit 3 of
 * qmm_device_status().  K == 0 fills Y with zeros; P == 0 or N == 0 launches
 * nothing.                                                                     */
qmm_status qmm_gather_small_m(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                              const int32_t* lhs, const int32_t* rhs, int P, int T, int E, int N, int K, int bits,
                              int group_size, void* Y, int out_dtype, int variant, int splits, void* stream);

/* ggml block formats, converted on the device to the layout above.  A row of
 * W is K/32 consecutive blocks of 32 weights; blocks of all rows are
 * contiguous, row after row.  Byte layouts (the public ggml format; the pages
 * name the formats, "metal : few-row MMA mat-mul and batched copies for
 * speculative decoding", Overview):
 *   QMM_GGML_Q4_0, 18 bytes: fp16 d; 16 bytes of 4-bit codes c, byte j holding
 *                  weight j in its low nibble and weight j + 16 in its high
 *                  nibble; w = d (c - 8).
 *   QMM_GGML_Q4_1, 20 bytes: fp16 d, fp16 m, the 16 code bytes; w = d c + m.
 *   QMM_GGML_Q8_0, 34 bytes: fp16 d, 32 signed bytes q; w = d q.                */
typedef enum { QMM_GGML_Q4_0 = 0, QMM_GGML_Q4_1 = 1, QMM_GGML_Q8_0 = 2 } qmm_ggml_type;

/* Exact conversion of a ggml matrix [N, K] (device `blocks`) into Wq
 * [N, K*bits/32], scales and biases fp16 [N, K/32] (device, caller-owned) for
 * qmm_small_m* with group_size 32 and bits = 4 (Q4_0, Q4_1) or 8 (Q8_0):
 * codes unchanged (Q4) or q + 128 (Q8_0), scale d, bias -8 d (Q4_0), m (Q4_1)
 * or -128 d (Q8_0).  Exact for every Q4_1 block, and for Q4_0 / Q8_0 blocks
 * with |d| <= 8188 / 511.75: beyond that (or for a d that is inf or NaN) the
 * bias has no finite fp16 value, the converted group is not the block, and
 * bit 4 of qmm_device_status() is set.  Asynchronous on `stream`.
 * QMM_ERR_UNSUPPORTED for an
 * unknown type, QMM_ERR_SHAPE for K not a multiple of 32, QMM_ERR_NULL /
 * QMM_ERR_ALIGN for the outputs (Wq 4-byte, scales/biases 2-byte aligned).   */
qmm_status qmm_from_ggml(int type, const void* blocks, int64_t N, int64_t K, uint32_t* Wq, void* scales,
                         void* biases, void* stream);

/* Microscaling fp modes: Y = X . W^T with w = 2^(E - 127) * value(code), one
 * E8M0 scale byte E per (row, group of 32 along K), scales uint8 [N, K/32];
 * no bias.  Codes are packed as above: QMM_MXFP4 = FP4 E2M1 (4 bits: sign, 2
 * exponent bits with bias 1, 1 mantissa bit; values 0, 0.5, 1, 1.5, 2, 3, 4,
 * 6 and negatives), QMM_MXFP8 = FP8 E4M3 (8 bits: sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, exponent 0 subnormal).  Encodings: the OCP
 * microscaling format; source of the modes: "MLX quantized_matmul small-M
 * verify kernels", facts "Fix family 1" / "qmv_wide covers affine, nvfp4,
 * mxfp4, mxfp8".  variant -1 (with splits -1): the compiled-in
 * microscaling table's choice for a swept (format, N, K), at the nearest
 * measured M with as many 8-row activation tiles; else the warp-owned family
 * when it can plan the shape (K/g a multiple of the cluster size, scales
 * 16-byte aligned, and K/g a multiple of 16 or else N*K/g a multiple of 16
 * with K/g <= 256), else the first "mma" variant; a forced "mma" or
 * "tma_own" variant is used as given, a "tma" variant returns
 * QMM_ERR_UNSUPPORTED.
 * QMM_NVFP4: FP4 E2M1 codes with one FP8 E4M3 scale byte per group of 16,
 * scales uint8 [N, K/16] (a per-tensor scale, where a model has one, is left
 * to the caller).
 * K must be a multiple of 32.  NaN encodings are NaN, as the OCP format
 * defines them: an E4M3 code or nvfp4 scale byte 0x7F / 0xFF, an E8M0 scale
 * 255; every output whose sum meets one is NaN.  Errors as qmm_small_m_ex.    */
typedef enum { QMM_MXFP4 = 0, QMM_MXFP8 = 1, QMM_NVFP4 = 2 } qmm_mx_format;
qmm_status qmm_small_m_mx(const void* X, const uint32_t* Wq, const uint8_t* scales, int M, int N, int K, int format,
                          void* Y, int out_dtype, int variant, int splits, void* stream);

/* Number of uint32 words of a packed [N, K] matrix: N * K * bits / 32
 * (0 if bits is unsupported or K*bits is not a multiple of 32).                 */
size_t qmm_packed_words(int64_t N, int64_t K, int bits);

/* Host-side packing of codes q[N,K] (one code per byte, each < 2^bits) into the
 * word layout above.  Host pointers.  Returns QMM_ERR_SHAPE for a code out of
 * range or a K that does not fill whole words.                                 */
qmm_status qmm_pack(const uint8_t* q, int64_t N, int64_t K, int bits, uint32_t* Wq);

/* Inverse of qmm_pack (host pointers).                                          */
qmm_status qmm_unpack(const uint32_t* Wq, int64_t N, int64_t K, int bits, uint8_t* q);

/* Conversion between the canonical layout above and the layout the kernels
 * read ("native").  The kernels read the canonical layout directly (the
 * k-permutation their tensor-core fragments need is applied to the
 * activations while they are staged), so the native layout IS the canonical
 * one: both calls are a stream-ordered device-to-device copy of
 * N*K*bits/8 bytes on `stream`, and nothing when the two pointers are equal.
 * Device pointers, caller-owned; the buffers must not partly overlap.
 * QMM_ERR_UNSUPPORTED for bits not in {2,4,8}, QMM_ERR_SHAPE for a K that
 * does not fill whole words, QMM_ERR_NULL for a null pointer with a non-empty
 * matrix, QMM_ERR_CUDA if the copy cannot be queued.                            */
qmm_status qmm_repack(const uint32_t* Wq, int64_t N, int64_t K, int bits, uint32_t* Wq_native, void* stream);
qmm_status qmm_unrepack(const uint32_t* Wq_native, int64_t N, int64_t K, int bits, uint32_t* Wq, void* stream);

/* Introspection of the dispatcher: the variant and split count qmm_small_m
 * would use, or -1 (and *splits untouched) if the shape is unsupported or the
 * table is unusable.  The table is compiled in; the environment variable
 * QMM_TABLE=<path> replaces it, for the whole process, by a file in the
 * format of the compiled one (lines "{M, N, K, bits, group, variant, splits},",
 * text after "//" ignored).  QMM_FORCE_VARIANT=<name or id> and
 * QMM_FORCE_SPLITS=<n> override the choice; QMM_LOG=1 prints it to stderr.      */
int qmm_select_variant(int M, int N, int K, int bits, int group_size, int* splits);

int qmm_num_variants(void);
const char* qmm_variant_name(int variant);     /* NULL for an unknown id          */
const char* qmm_status_string(int status);
int qmm_last_cuda_error(void);                 /* cudaError_t of the last failure */

/* Device status word of the kernels, OR-ed over all kernel units: bit 0 = a
 * consumer gave up waiting for a weight tile, bit 1 = the producer gave up
 * waiting for a free stage, bit 2 = copies still in flight at exit gave up,
 * bit 3 = a gathered call had an invalid index list (see qmm_gather_small_m),
 * bit 4 = qmm_from_ggml met a block outside its exact range.
 * Every wait is bounded (about 2 s), so a fault shows up here instead of as a
 * hang.  Synchronizes with the device; clears the word when `clear` != 0.
 * 0xFFFFFFFF if the word could not be read.                                    */
unsigned int qmm_device_status(int clear);
const char* qmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H_ */
