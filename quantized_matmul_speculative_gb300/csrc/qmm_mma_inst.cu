// One translation unit per (bits, group size), chosen by -DQMM_BITS / -DQMM_GS,
// so the kernel instantiations compile in parallel.
#include "qmm_mma_launch.cuh"

#ifndef QMM_BITS
#error "QMM_BITS must be defined"
#endif
#ifndef QMM_GS
#error "QMM_GS must be defined"
#endif

namespace qmm {
template cudaError_t launch_mma_bg<QMM_BITS, QMM_GS>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
}
