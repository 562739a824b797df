// Device side of the gathered (mixture-of-experts) form of the product:
//     Y[i, :] = X[lhs[i], :] . dequant(W[rhs[i]])^T,   i < P,
// over a stack of E quantized matrices.  The union of the experts the entries
// name is computed in every CTA from the index lists; CTA slot s takes the
// s-th expert of the union (in order of first appearance) and all entries
// that name it, so each expert of the union is streamed once per call for
// all of its activation rows ("MLX quantized_matmul small-M verify kernels":
// the open question on "dense and MoE (gather_qmm) verify" and the
// "expert-union cost per verify row").
#pragma once

#include <cstdint>

#include "qmm_device.cuh"

namespace qmm {

// All THREADS threads of the CTA call this (it has barriers); P <= THREADS.
// On success: *expert = the slot's expert, *rows = its entry count (<= max_rows),
// row[m] = the activation row and out[m] = the output row of its m-th entry in
// increasing entry order.  Returns false (the same value in every thread) if
// the slot is past the end of the union, or if the lists are invalid: an index
// out of range (that entry is skipped) or more than max_rows entries for the
// slot's expert; both set kStatusBadGather.
template <int THREADS>
__device__ bool gather_setup(const int32_t* lhs, const int32_t* rhs, int P, int T, int E, int slot, int max_rows,
                             int* row, int* out, int* expert, int* rows) {
  static_assert(THREADS % 32 == 0 && THREADS <= 1024, "whole warps");
  __shared__ int s_e[THREADS];
  __shared__ unsigned int s_bal[THREADS / 32];
  __shared__ int s_expert;
  const int tid = static_cast<int>(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned int lt = (1u << lane) - 1u;
  int e_i = -1, t_i = 0;
  if (tid < P) {
    e_i = rhs[tid];
    t_i = lhs[tid];
    if (e_i < 0 || e_i >= E || t_i < 0 || t_i >= T) {
      atomicOr(&g_qmm_status, kStatusBadGather);
      e_i = -1;
    }
  }
  s_e[tid] = e_i;
  if (tid == 0) s_expert = -1;
  __syncthreads();
  // first appearance of this entry's expert (all threads read s_e[j] together: broadcasts)
  bool first = e_i >= 0;
  for (int j = 0; j < P; ++j) first = first && !(j < tid && s_e[j] == e_i);
  const unsigned int bal = __ballot_sync(0xffffffffu, first);
  if (lane == 0) s_bal[warp] = bal;
  __syncthreads();
  int before = __popc(bal & lt);
  for (int w = 0; w < warp; ++w) before += __popc(s_bal[w]);
  if (first && before == slot) s_expert = e_i;
  __syncthreads();
  const int e = s_expert;
  if (e < 0) return false;
  const bool mine = e_i == e;
  const unsigned int bal2 = __ballot_sync(0xffffffffu, mine);
  if (lane == 0) s_bal[warp] = bal2;
  __syncthreads();
  int m = __popc(bal2 & lt), cnt = 0;
  for (int w = 0; w < THREADS / 32; ++w) {
    const int c = __popc(s_bal[w]);
    cnt += c;
    if (w < warp) m += c;
  }
  if (mine && m < max_rows) {
    row[m] = t_i;
    out[m] = tid;
  }
  __syncthreads();
  if (cnt > max_rows) {
    if (tid == 0) atomicOr(&g_qmm_status, kStatusBadGather);
    return false;
  }
  *expert = e;
  *rows = cnt;
  return true;
}

}  // namespace qmm
