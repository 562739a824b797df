// Host-side launcher of the warp-specialized TMA family (see qmm_tma.cuh).
#pragma once

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "qmm_geometry.h"
#include "qmm_internal.h"
#include "qmm_tiles.h"
#include "qmm_tma.cuh"

namespace qmm {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Maximum co-resident clusters of `csize` CTAs for a kernel and shared-memory
// size, cached per (device, kernel, csize, smem).
inline int max_active_clusters(const void* kern, int threads, int smem, int csize) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, kern, csize, smem);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

template <int BITS, int GS, int NB, int W, int S, bool E8, bool GATHER>
cudaError_t launch_tma_impl(const CallArgs& a, int csize, int ctas_per_sm, cudaStream_t stream) {
  using Cfg = TmaCfg<BITS, GS, NB, W, S>;
  TmaParams p;
  p.X = a.X;
  p.S = a.S;
  p.B = a.B;
  p.Y = a.Y;
  p.R = a.R;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.G = a.K / GS;
  p.out_f32 = a.out_f32;
  // Test-only fault injection (host-triggered): a short limit for the waits on
  // tile data and one tile whose declared bytes never all arrive; those waits
  // give up and set bits of the device status word, the call still completes.
  {
    const char* inject = std::getenv("QMM_TEST_INJECT");
    const bool short_wait = inject != nullptr && std::strcmp(inject, "short_wait") == 0 && a.rhs == nullptr;
    p.wait_ns = short_wait ? 100000ull : kWaitLimitNs;
    p.inject = short_wait ? 1 : 0;
  }
  if (!tma_geometry(a.K, BITS, GS, csize, &p.gp, &p.pw, &p.box_words, &p.nbox, &p.mbw)) return cudaErrorInvalidValue;
  p.gp_magic = ((1ull << 32) + static_cast<unsigned long long>(p.gp) - 1) / static_cast<unsigned long long>(p.gp);
  if ((reinterpret_cast<uintptr_t>(a.S) | reinterpret_cast<uintptr_t>(a.B)) & 15) return cudaErrorInvalidValue;
  p.tiles = (a.N + 15) / 16;
  // Gathered form: tiles of the largest possible union; the stack's rows in the tensor maps
  p.lhs = a.lhs;
  p.rhs = a.rhs;
  p.P = a.P;
  p.E = a.E;
  p.tpe = p.tiles;
  p.gather_off = 0;
  constexpr bool gathered = GATHER;
  int64_t map_rows = a.N;
  if (gathered) {
    if (a.P > Cfg::THREADS || a.P > kMaxGatherEntries || a.E < 1) return cudaErrorInvalidValue;
    p.tiles = (a.E < a.P ? a.E : a.P) * p.tpe;
    map_rows = static_cast<int64_t>(a.E) * a.N;
  }
  const int gather_bytes = gathered ? kGatherSmemInts * 4 : 0;

  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  auto kern = qmm_tma_kernel<BITS, GS, NB, W, S, E8, GATHER>;
  // Shared memory: what remains of the SM's budget for ctas_per_sm CTAs goes to
  // the partial tiles of one reduction round.
  int sm_bytes = 0, optin = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int budget_all = tma_smem_budget(sm_bytes, optin, ctas_per_sm);
  const int budget = budget_all - gather_bytes;  // what the stages and partials may use
  static std::mutex mu;
  static int smem_set = 0;
  static bool nonportable = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (budget_all > smem_set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, budget_all);
      if (e != cudaSuccess) return e;
      smem_set = budget_all;
    }
    if (csize > 8 && !nonportable) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      nonportable = true;
    }
  }
  // Clusters: as many as fit at the budget's shared-memory size, no more than tiles.
  int ncl = max_active_clusters(reinterpret_cast<const void*>(kern), Cfg::THREADS, budget_all, csize);
  if (ncl < 1) return cudaErrorInvalidConfiguration;
  if (ncl > p.tiles) ncl = p.tiles;
  p.ncl = ncl;
  const int nt_max = (p.tiles + ncl - 1) / ncl;  // tiles per cluster (cluster_tile_begin)
  // The fewest tiles a cluster can get.  A gathered call's union, known only on
  // the device, can be anything from one expert to the largest: its clusters
  // can get as little as one tile, and a window of fewer tiles is met by more
  // warps (tma_slots is largest at one tile).
  const int nt_min = gathered ? 1 : p.tiles / ncl;

  TmaPlan plan;
  if (!tma_plan(p.pw, p.gp, GS, Cfg::MP, p.mbw, W, S, csize, nt_max, nt_min, budget, &plan)) return cudaErrorInvalidValue;
  p.single = plan.single;
  p.stages = plan.stages;
  p.rt = plan.rt;
  p.slots = plan.slots;
  p.ws = plan.ws;
  p.push = plan.push;
  p.recv_tiles = plan.recv_tiles;
  int smem = TmaLayout(p.pw, p.gp, GS, Cfg::MP, p.stages, p.rt, p.slots, p.mbw, p.recv_tiles, csize).total;
  if (gathered) {
    p.gather_off = (smem + 15) & ~15;
    smem = p.gather_off + gather_bytes;
  }

  CUtensorMap tmap, tmap_s, tmap_b;
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(a.K) * BITS / 32, static_cast<cuuint64_t>(map_rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(a.K) * BITS / 8};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.box_words), 16u};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.Wq), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int arr = 0; arr < 2; ++arr) {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(p.G), static_cast<cuuint64_t>(map_rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(p.G) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.mbw), 16u};
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
                   "qmm tma: grid %dx%d (clusters of %d) threads %d smem %d budget %d stages %d window %d round %d slots %d "
                   "single %d push %d gp %d pw %d boxes %d\n",
                   csize, ncl, csize, Cfg::THREADS, smem, budget, p.stages, p.ws, p.rt, p.slots, p.single, p.push,
                   p.gp, p.pw, p.nbox);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, ncl, 1);
  cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
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
  return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_s, tmap_b, p);
}

template <int BITS, int GS, int NB, bool E8>
cudaError_t launch_tma_tile(const CallArgs& a, const VariantDesc& d, int csize, cudaStream_t stream) {
#define QMM_TRY_TMA(w, s)                                                   \
  if (d.WN == (w) && d.R == (s))                                            \
    return (a.rhs != nullptr) ? launch_tma_impl<BITS, GS, NB, w, s, E8, true>(a, csize, d.WK, stream)  \
                              : launch_tma_impl<BITS, GS, NB, w, s, E8, false>(a, csize, d.WK, stream);
  QMM_TMA_TILES(QMM_TRY_TMA)
#undef QMM_TRY_TMA
  return cudaErrorInvalidValue;
}

template <int BITS, int GS>
cudaError_t launch_tma_bg(const CallArgs& a, const VariantDesc& d, int csize, cudaStream_t stream) {
  if constexpr (BITS == 8) {
    const CallArgs v = as_virtual_nibbles(a);
    if (v.M <= 8) return launch_tma_tile<4, 2 * GS, 1, true>(v, d, csize, stream);
    return launch_tma_tile<4, 2 * GS, 2, true>(v, d, csize, stream);
  } else {
    if (a.M <= 8) return launch_tma_tile<BITS, GS, 1, false>(a, d, csize, stream);
    return launch_tma_tile<BITS, GS, 2, false>(a, d, csize, stream);
  }
}

}  // namespace qmm
