// One translation unit per (bits, group size), chosen by -DQMM_BITS / -DQMM_GS,
// so the kernel instantiations compile in parallel.
#include "qmm_mma_launch.cuh"
#include "qmm_own_launch.cuh"
#include "qmm_tma_launch.cuh"

#ifndef QMM_BITS
#error "QMM_BITS must be defined"
#endif
#ifndef QMM_GS
#error "QMM_GS must be defined"
#endif

namespace qmm {

// Host reader of this translation unit's device status word.
template <int BITS, int GS>
unsigned int read_device_status(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qmm_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear && v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_qmm_status, &zero, sizeof(zero));
  }
  return v;
}

template unsigned int read_device_status<QMM_BITS, QMM_GS>(int);
template cudaError_t launch_mma_bg<QMM_BITS, QMM_GS>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template cudaError_t launch_tma_bg<QMM_BITS, QMM_GS>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template cudaError_t launch_own_bg<QMM_BITS, QMM_GS>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
#if QMM_BITS == 4 && QMM_GS == 32
template cudaError_t launch_mma_mx<0>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template cudaError_t launch_own_mx<0>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
#endif
#if QMM_BITS == 4 && QMM_GS == 64
template cudaError_t launch_mma_mx<2>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template cudaError_t launch_own_mx<2>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
#endif
#if QMM_BITS == 8 && QMM_GS == 32
template cudaError_t launch_mma_mx<1>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template cudaError_t launch_own_mx<1>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
#endif
}
