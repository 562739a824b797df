// Internal interface between the C ABI (qmm_api.cu) and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

// Arguments of one call after host-side validation.
struct CallArgs {
  const uint16_t* X;   // bf16 [M, K]
  const uint32_t* Wq;  // packed codes [N, K*bits/32]
  const uint16_t* S;   // fp16 [N, K/gs]
  const uint16_t* B;   // fp16 [N, K/gs]
  void* Y;             // bf16 or fp32 [M, N]
  const void* R;       // residual, Y's dtype [M, N], added in the store; may be Y; null: none
  int M, N, K, bits, gs, out_f32;
  // Gathered form (null rhs: a plain call): entry i of P multiplies activation
  // row lhs[i] of X [T, K] by matrix rhs[i] of the stack Wq/S/B [E][N][...]
  // into row i of Y [P, N]; M is then the largest row count one expert can
  // take (8 or 16).
  const int32_t* lhs = nullptr;
  const int32_t* rhs = nullptr;
  int P = 0, T = 0, E = 0;
  // Microscaled weights (S8 non-null): one scale byte per group (E8M0 per
  // 32, or E4M3 per 16 for nvfp4), no biases.
  const uint8_t* S8 = nullptr;
};

// Code formats of the mma family's kernels.
constexpr int kCodesAffine = 0;   // b-bit affine codes read natively (2 or 4 bits)
constexpr int kCodesAffine8 = 1;  // 8-bit affine codes as virtual 4-bit codes
constexpr int kCodesMx4 = 2;      // mxfp4: FP4 E2M1 codes, E8M0 scale per 32
constexpr int kCodesMx8 = 3;      // mxfp8: FP8 E4M3 codes, E8M0 scale per 32
constexpr int kCodesNv4 = 4;      // nvfp4: FP4 E2M1 codes, E4M3 scale per 16

// Most entries of a gathered call: the kernels scan the index lists with one
// entry per thread.
constexpr int kMaxGatherEntries = 256;

// 8-bit codes run on the 4-bit kernels as "virtual" 4-bit codes (each byte
// read as its low and high nibble): the same words, groups and scales, with
// twice as many codes per row and per group.
inline CallArgs as_virtual_nibbles(const CallArgs& a) {
  CallArgs v = a;
  v.K = 2 * a.K;
  v.gs = 2 * a.gs;
  v.bits = 4;
  return v;
}

enum Family { kFamilyMma = 0, kFamilySimt = 1, kFamilyTma = 2, kFamilyOwn = 3 };

// One kernel variant: a family and its CTA tiling.
struct VariantDesc {
  const char* name;
  int family;
  int R;   // mma: m16 row tiles per warp; tma: ring stages; own: ring stages per warp
  int WN;  // mma: warps along N; tma, own: consumer warps
  int WK;  // mma: warps along K (intra-CTA split-K); tma, own: CTAs per SM the shared memory is sized for
  int wave;  // own: at most this many CTAs per SM launched (0: as many as fit); with wave < WK
             // the next call's CTAs fit beside this call's and stream their weights early
};

const VariantDesc* variant_desc(int v);
int variant_count();

// Rows of W one CTA of variant `v` covers.
int variant_rows_per_cta(const VariantDesc& d);

// Launch variant `d` with `splits` CTAs per cluster along K.  Returns the CUDA
// error of the launch (cudaSuccess when it was queued).
cudaError_t launch_mma(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream);
cudaError_t launch_tma(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream);
// With plan_only, nothing is launched: cudaSuccess if the shape can run,
// cudaErrorNotSupported if it cannot.
cudaError_t launch_own(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream, bool plan_only);

// Whether the TMA family can run (K, bits, gs) split across `csize` CTAs.
bool tma_supported(const CallArgs& a, int csize, const VariantDesc& d);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace qmm
