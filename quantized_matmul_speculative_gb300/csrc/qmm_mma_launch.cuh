// Host-side launcher of the tensor-core kernel family (see qmm_mma.cuh).
#pragma once

#include <mutex>

#include "qmm_internal.h"
#include "qmm_mma.cuh"
#include "qmm_tiles.h"

namespace qmm {

// Shared memory one CTA may use; keeps two 256-thread CTAs resident per SM.
constexpr int kMmaSmemBudget = 100 * 1024;

template <int BITS, int GS, int NB, int R, int WN, int WK, int CODES>
cudaError_t launch_mma_impl(const CallArgs& a, int splits, cudaStream_t stream) {
  using C = MmaCfg<BITS, GS, NB, R, WN, WK>;
  MmaParams p;
  p.X = a.X;
  p.Wq = a.Wq;
  p.S = a.S;
  p.B = a.B;
  p.Y = a.Y;
  p.R = a.R;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.out_f32 = a.out_f32;
  p.G = a.K / GS;
  p.gpc = (p.G + splits - 1) / splits;
  p.S8 = a.S8;
  p.lhs = a.lhs;
  p.rhs = a.rhs;
  p.P = a.P;
  p.T = a.T;
  p.E = a.E;
  p.tiles = (a.N + C::NT - 1) / C::NT;
  p.w_stride = static_cast<int64_t>(a.N) * (a.K / C::VPW);
  p.m_stride = static_cast<int64_t>(a.N) * p.G;
  // gathered form: one group of row tiles per possible expert of the union
  const int slots = (a.rhs != nullptr) ? (a.E < a.P ? a.E : a.P) : 1;
  if (a.rhs != nullptr && (a.P > C::THREADS || slots < 1)) return cudaErrorInvalidValue;
  // Largest chunk that fits the budget, then even chunks across the K-range.
  int cmax = p.gpc;
  while (cmax > 1 && MmaSmem<C>(cmax).total > kMmaSmemBudget) --cmax;
  const int nchunks = (p.gpc + cmax - 1) / cmax;
  p.chunk = (p.gpc + nchunks - 1) / nchunks;
  if (p.chunk < 1) p.chunk = 1;
  const int smem = MmaSmem<C>(p.chunk).total;

  auto kern = qmm_mma_kernel<BITS, GS, NB, R, WN, WK, CODES>;
  static std::mutex mu;
  static int smem_set = 0;
  static bool nonportable_set = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (smem > smem_set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      smem_set = smem;
    }
    if (splits > 8 && !nonportable_set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      nonportable_set = true;
    }
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.tiles * slots, splits, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (splits > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = splits;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BITS, int GS, int NB, int CODES>
cudaError_t launch_mma_tile(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream) {
#define QMM_TRY_TILE(r, wn, wk)                                                     \
  if (d.R == (r) && d.WN == (wn) && d.WK == (wk))                                   \
    return launch_mma_impl<BITS, GS, NB, r, wn, wk, CODES>(a, splits, stream);
  QMM_MMA_TILES(QMM_TRY_TILE)
#undef QMM_TRY_TILE
  return cudaErrorInvalidValue;
}

// Entry for one (bits, group size): picks the activation-tile count from M.
template <int BITS, int GS>
cudaError_t launch_mma_bg(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream) {
  if constexpr (BITS == 8) {
    const CallArgs v = as_virtual_nibbles(a);
    if (v.M <= 8) return launch_mma_tile<4, 2 * GS, 1, kCodesAffine8>(v, d, splits, stream);
    return launch_mma_tile<4, 2 * GS, 2, kCodesAffine8>(v, d, splits, stream);
  } else {
    if (a.M <= 8) return launch_mma_tile<BITS, GS, 1, kCodesAffine>(a, d, splits, stream);
    return launch_mma_tile<BITS, GS, 2, kCodesAffine>(a, d, splits, stream);
  }
}

// Microscaled weights: FMT 0 = mxfp4 (4-bit codes, groups of 32), 1 = mxfp8
// (8-bit codes, groups of 32), 2 = nvfp4 (4-bit codes, groups of 16).
template <int FMT>
cudaError_t launch_mma_mx(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream) {
  constexpr int BITS = FMT == 1 ? 8 : 4;
  constexpr int GS = FMT == 2 ? 16 : 32;
  constexpr int CODES = FMT == 0 ? kCodesMx4 : FMT == 1 ? kCodesMx8 : kCodesNv4;
  if (a.M <= 8) return launch_mma_tile<BITS, GS, 1, CODES>(a, d, splits, stream);
  return launch_mma_tile<BITS, GS, 2, CODES>(a, d, splits, stream);
}

}  // namespace qmm
