// Host-side planner and launcher of the warp-owned TMA family (qmm_own.cuh).
#pragma once

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "qmm_geometry.h"
#include "qmm_internal.h"
#include "qmm_own.cuh"
#include "qmm_tiles.h"
#include "qmm_tma_launch.cuh"

namespace qmm {

// Plan one call: K-piece, parts per tile, box widths, clusters, receive
// slots and shared memory.  Returns cudaErrorNotSupported (and launches
// nothing) when (W, D, csize, CTAs per SM) cannot run the shape.
template <int BITS, int GS, int NB, int W, int D, int CODES, bool GATHER>
cudaError_t own_plan(const CallArgs& a, int csize, int ctas_per_sm, int wave, OwnParams* p, int* smem, int* budget) {
  using GM = GroupMath<BITS, GS, NB, CODES>;
  constexpr int GW = GM::GW;
  constexpr bool MX = GM::MX;
  constexpr int MP = 8 * NB;
  const int G = a.K / GS;
  if (G % csize != 0) return cudaErrorNotSupported;
  bool meta_tile = false;
  if (MX) {
    // one scale byte per group: rows that are not 16-byte strided (G % 16 != 0) are copied a
    // whole tile at a time through a [rows*G/16, 16] view (rows*G % 16 == 0, one box: G <= 256)
    if (reinterpret_cast<uintptr_t>(a.S8) & 15) return cudaErrorNotSupported;
    if (G % 16 != 0) {
      if (G > 256 || (static_cast<int64_t>(a.N) * G) % 16 != 0) return cudaErrorNotSupported;
      meta_tile = true;
    }
  } else {
    if ((reinterpret_cast<uintptr_t>(a.S) | reinterpret_cast<uintptr_t>(a.B)) & 15) return cudaErrorNotSupported;
    if (G % 8 != 0) {
      // Scale/bias rows that are not 16-byte strided: each stage takes its whole tile's
      // metadata as one box of 2G rows of a [rows*G/8, 8] view, which must hold every
      // element (rows*G % 8 == 0; a gathered stack's matrices start on view rows too) and
      // fit one box (2G <= 256).
      const int64_t rows = GATHER ? static_cast<int64_t>(a.E) * a.N : a.N;
      if (G > 128 || (rows * G) % 8 != 0 || (static_cast<int64_t>(a.N) * G) % 8 != 0) return cudaErrorNotSupported;
      meta_tile = true;
    }
  }
  p->meta_tile = meta_tile ? 1 : 0;
  p->X = a.X;
  p->Y = a.Y;
  p->R = a.R;
  p->M = a.M;
  p->N = a.N;
  p->K = a.K;
  p->out_f32 = a.out_f32;
  p->gp = G / csize;
  p->gp_magic = ((1ull << 32) + static_cast<unsigned long long>(p->gp) - 1) / static_cast<unsigned long long>(p->gp);
  p->tiles = (a.N + 15) / 16;
  p->tpe = p->tiles;
  p->lhs = a.lhs;
  p->rhs = a.rhs;
  p->P = a.P;
  p->E = a.E;
  p->gather_off = 0;
  if constexpr (GATHER) {
    // every entry scanned by one thread; tiles of the largest possible union
    if (a.P > 32 * W || a.P > kMaxGatherEntries || a.E < 1) return cudaErrorNotSupported;
    p->tiles = (a.E < a.P ? a.E : a.P) * p->tpe;
  }
  const int gather_bytes = GATHER ? kGatherSmemInts * 4 : 0;

  auto kern = qmm_own_kernel<BITS, GS, NB, W, D, CODES, GATHER>;
  int sm_bytes = 0, optin = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  *budget = tma_smem_budget(sm_bytes, optin, ctas_per_sm);
  {
    static std::mutex mu;
    static int smem_set = 0;
    static bool nonportable = false;
    std::lock_guard<std::mutex> lock(mu);
    if (*budget > smem_set) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, *budget);
      if (e != cudaSuccess) return e;
      smem_set = *budget;
    }
    if (csize > 8 && !nonportable) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      nonportable = true;
    }
  }
  int ncl = max_active_clusters(reinterpret_cast<const void*>(kern), 32 * W, *budget, csize);
  if (ncl < 1) return cudaErrorNotSupported;
  if (wave > 0 && wave < ctas_per_sm) {
    // at most `wave` CTAs per SM: the rest of the SM is left to the next call's CTAs
    const int cap = wave * device_sm_count() / csize;
    if (cap >= 1 && ncl > cap) ncl = cap;
  }
  if (ncl > p->tiles) ncl = p->tiles;
  p->ncl = ncl;
  const int nt_max = (p->tiles + ncl - 1) / ncl;
  const int nt_min = p->tiles / ncl;

  // Parts per tile: the fewest (largest units) that give every warp at least
  // two units and fit; failing that, the most that fit.
  bool found = false;
  for (int kp = 1; kp <= p->gp; ++kp) {
    if (p->gp % kp != 0) continue;
    const int gq = p->gp / kp;
    // Weight boxes: 32-word (128-byte) rows copied with the 128-byte swizzle
    // when a unit is whole such boxes of 4 or 8 groups (4 or 8 words per group
    // row: 4-bit g32 / g64, 2-bit g64 / g128; measured slower with 16-word
    // groups, two per box); the fragment loads are then free of
    // shared-memory bank conflicts); else boxes of whole groups, 16-byte
    // multiples of <= 256 words, the widest (fewer copies per unit measured
    // better than narrow unswizzled boxes without conflicts).
    const bool swz = (GW == 4 || GW == 8) && (gq * GW) % 32 == 0;
    int bw = swz ? 32 : 0;
    for (int d = 1; !swz && d <= gq; ++d) {
      if (gq % d != 0) continue;
      const int w = d * GW;
      if (w <= 256 && w % 4 == 0) bw = w;
    }
    if (bw == 0) continue;
    // scale box width: any start within 8 groups (fp16) or 16 groups (bytes) of the box start
    const int mbw = meta_tile ? G : MX ? (15 + gq + 15) / 16 * 16 : (7 + gq + 7) / 8 * 8;
    if (mbw > 256) continue;
    // the bias box starts 128-byte aligned in the stage, like every TMA destination
    const int bofs = meta_tile ? (16 * G + 63) / 64 * 64 : 16 * mbw;
    const int meta_row = MX ? mbw : (bofs + 16 * mbw) / 8;
    int maxw = 1;
    for (int nt : {nt_min, nt_max}) {
      if (nt < 1) continue;
      for (int i = 0; i < nt; ++i) {
        int sl;
        const int n = own_contributors(i, kp, nt * kp, W, -1, &sl);
        maxw = n > maxw ? n : maxw;
      }
    }
    const int owned_max = (nt_max + csize - 1) / csize;
    const OwnLayout L(W, D, p->gp, GS, MP, NB, gq * GW / bw, bw, meta_row, owned_max, csize, maxw, a.M, swz ? 1 : 0);
    int total = L.total;
    if constexpr (GATHER) {
      // The union decides the tile count nt <= nt_max in the kernel, which
      // then strides the receive slots by maxw(nt): reserve the largest
      // owned(nt) * maxw(nt) (owned by CTA rank 0, the most).
      int64_t slots = 0;
      for (int nt = 1; nt <= nt_max; ++nt) {
        int mw = 1;
        for (int i = 0; i < nt; ++i) {
          int sl;
          const int n = own_contributors(i, kp, nt * kp, W, -1, &sl);
          mw = n > mw ? n : mw;
        }
        const int64_t need = static_cast<int64_t>((nt + csize - 1) / csize) * mw;
        slots = need > slots ? need : slots;
      }
      total = L.recv_off + static_cast<int>(slots) * csize * L.slot_bytes;
      const int x_end = L.x_off + MP * L.rsx * 2;
      if (total < x_end) total = x_end;
      total = ((total + 15) & ~15) + gather_bytes + (swz ? 1024 : 0);
      maxw = 0;  // the kernel finds its own
    }
    if (total > *budget) continue;
    p->kp = kp;
    p->gq = gq;
    p->swz = swz ? 1 : 0;
    p->bw = bw;
    p->nbox = gq * GW / bw;
    p->mbw = mbw;
    p->bofs = bofs;
    p->maxw = maxw;
    p->owned_max = owned_max;
    p->gather_off = GATHER ? total - gather_bytes - (swz ? 1024 : 0) : 0;
    *smem = total;
    found = true;
    if (nt_min * kp >= 2 * W) break;
  }
  return found ? cudaSuccess : cudaErrorNotSupported;
}

template <int BITS, int GS, int NB, int W, int D, int CODES, bool GATHER>
cudaError_t launch_own_impl(const CallArgs& a, int csize, int ctas_per_sm, int wave, cudaStream_t stream,
                            bool plan_only) {
  OwnParams p;
  int smem = 0, budget = 0;
  const cudaError_t pe = own_plan<BITS, GS, NB, W, D, CODES, GATHER>(a, csize, ctas_per_sm, wave, &p, &smem, &budget);
  constexpr bool MX = GroupMath<BITS, GS, NB, CODES>::MX;
  const int64_t map_rows = GATHER ? static_cast<int64_t>(a.E) * a.N : a.N;  // gathered: the whole stack
  if (pe != cudaSuccess || plan_only) return pe;

  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorUnknown;
  CUtensorMap tmap, tmap_s, tmap_b;
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(a.K) * BITS / 32, static_cast<cuuint64_t>(map_rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(a.K) * BITS / 8};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.bw), 16u};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.Wq), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, p.swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int G = a.K / GS;
  if (MX) {
    // one byte per (row, group); the bias map is not read (a copy stands in for it).  [rows, G]
    // with a box of mbw groups x 16 rows, or (meta_tile) the [rows*G/16, 16] view, box 16 x G
    const cuuint64_t gdim[2] = {p.meta_tile ? 16u : static_cast<cuuint64_t>(G),
                                p.meta_tile ? static_cast<cuuint64_t>(map_rows) * G / 16
                                            : static_cast<cuuint64_t>(map_rows)};
    const cuuint64_t gstride[1] = {p.meta_tile ? 16u : static_cast<cuuint64_t>(G)};
    const cuuint32_t box[2] = {p.meta_tile ? 16u : static_cast<cuuint32_t>(p.mbw),
                               p.meta_tile ? static_cast<cuuint32_t>(G) : 16u};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.S8), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    tmap_b = tmap_s;
  }
  for (int arr = 0; arr < (MX ? 0 : 2); ++arr) {
    // [rows, G] with a box of mbw groups x 16 rows; or (meta_tile) the [rows*G/8, 8] view, box 8 x 2G
    const cuuint64_t gdim[2] = {p.meta_tile ? 8u : static_cast<cuuint64_t>(G),
                                p.meta_tile ? static_cast<cuuint64_t>(map_rows) * G / 8
                                            : static_cast<cuuint64_t>(map_rows)};
    const cuuint64_t gstride[1] = {p.meta_tile ? 16u : static_cast<cuuint64_t>(G) * 2};
    const cuuint32_t box[2] = {p.meta_tile ? 8u : static_cast<cuuint32_t>(p.mbw),
                               p.meta_tile ? static_cast<cuuint32_t>(2 * G) : 16u};
    const cuuint32_t estride[2] = {1u, 1u};
    void* base = const_cast<uint16_t*>(arr ? a.B : a.S);
    if (encode(arr ? &tmap_b : &tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const char* lg = std::getenv("QMM_LOG");
    if (lg != nullptr && lg[0] != '\0' && lg[0] != '0')
      std::fprintf(stderr,
                   "qmm own: grid %dx%d (clusters of %d) threads %d smem %d budget %d depth %d gp %d parts %d "
                   "gq %d box %dx%d%s maxw %d owned %d\n",
                   csize, p.ncl, csize, 32 * W, smem, budget, D, p.gp, p.kp, p.gq, p.nbox, p.bw, p.swz ? " swizzled" : "", p.maxw,
                   p.owned_max);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, p.ncl, 1);
  cfg.blockDim = dim3(32 * W, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, qmm_own_kernel<BITS, GS, NB, W, D, CODES, GATHER>, tmap, tmap_s, tmap_b, p);
}

// Gathered calls exist for the affine code formats only.
template <int BITS, int GS, int NB, int W, int D, int CODES>
cudaError_t launch_own_impl_g(const CallArgs& a, int csize, int ctas_per_sm, int wave, cudaStream_t stream,
                              bool plan_only) {
  if (a.rhs == nullptr) return launch_own_impl<BITS, GS, NB, W, D, CODES, false>(a, csize, ctas_per_sm, wave, stream,
                                                                                   plan_only);
  if constexpr (CODES == kCodesAffine || CODES == kCodesAffine8)
    return launch_own_impl<BITS, GS, NB, W, D, CODES, true>(a, csize, ctas_per_sm, wave, stream, plan_only);
  else
    return cudaErrorNotSupported;
}

template <int BITS, int GS, int NB, int CODES>
cudaError_t launch_own_tile(const CallArgs& a, const VariantDesc& d, int csize, cudaStream_t stream, bool plan_only) {
#define QMM_TRY_OWN(w, dd)                 \
  if (d.WN == (w) && d.R == (dd))          \
    return launch_own_impl_g<BITS, GS, NB, w, dd, CODES>(a, csize, d.WK, d.wave, stream, plan_only);
  QMM_OWN_TILES(QMM_TRY_OWN)
#undef QMM_TRY_OWN
  return cudaErrorNotSupported;
}

template <int BITS, int GS>
cudaError_t launch_own_bg(const CallArgs& a, const VariantDesc& d, int csize, cudaStream_t stream, bool plan_only) {
  if constexpr (BITS == 8) {
    const CallArgs v = as_virtual_nibbles(a);
    if (v.M <= 8) return launch_own_tile<4, 2 * GS, 1, kCodesAffine8>(v, d, csize, stream, plan_only);
    return launch_own_tile<4, 2 * GS, 2, kCodesAffine8>(v, d, csize, stream, plan_only);
  } else {
    if (a.M <= 8) return launch_own_tile<BITS, GS, 1, kCodesAffine>(a, d, csize, stream, plan_only);
    return launch_own_tile<BITS, GS, 2, kCodesAffine>(a, d, csize, stream, plan_only);
  }
}

// Microscaled weights on the warp-owned family: FMT 0 = mxfp4, 1 = mxfp8, 2 = nvfp4.
template <int FMT>
cudaError_t launch_own_mx(const CallArgs& a, const VariantDesc& d, int csize, cudaStream_t stream, bool plan_only) {
  constexpr int BITS = FMT == 1 ? 8 : 4;
  constexpr int GS = FMT == 2 ? 16 : 32;
  constexpr int CODES = FMT == 0 ? kCodesMx4 : FMT == 1 ? kCodesMx8 : kCodesNv4;
  if (a.M <= 8) return launch_own_tile<BITS, GS, 1, CODES>(a, d, csize, stream, plan_only);
  return launch_own_tile<BITS, GS, 2, CODES>(a, d, csize, stream, plan_only);
}

}  // namespace qmm
