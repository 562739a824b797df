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
#include "qmm_internal.h"

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

namespace qmm {

// Index lists of a gathered call sorted for a kernel that computes every
// token row against each expert of the union (the TMA family): the union in
// order of first appearance, and the valid entries ordered by (slot, entry).
constexpr int kGatherSmemInts = 6 * kMaxGatherEntries + 32 + 2;  // shared scratch of gather_lists

struct GatherLists {
  int u;        // experts in the union
  int* expert;  // [u]: expert of slot s
  int* start;   // [u + 1]: entries of slot s are entry[start[s] .. start[s+1])
  int* entry;   // entry index i (its output row), in (slot, i) order
  int* token;   // lhs of that entry (its activation row)
};

// All THREADS threads of the CTA call this (barriers); P <= min(THREADS,
// kMaxGatherEntries).  `sm` is kGatherSmemInts ints of shared memory; the
// lists live in it.  An index out of range sets kStatusBadGather and its entry
// is dropped.  Cost: two passes over the P entries per thread (shared-memory
// broadcasts) and a few barriers.
template <int THREADS>
__device__ GatherLists gather_lists(const int32_t* lhs, const int32_t* rhs, int P, int T, int E, int* sm) {
  static_assert(THREADS % 32 == 0 && THREADS <= 1024, "whole warps");
  constexpr int NE = kMaxGatherEntries;
  GatherLists gl;
  gl.expert = sm;
  gl.start = sm + NE;
  gl.entry = sm + 2 * NE + 1;
  gl.token = sm + 3 * NE + 1;
  int* s_e = sm + 4 * NE + 1;
  int* s_slot = sm + 5 * NE + 1;
  unsigned int* s_bal = reinterpret_cast<unsigned int*>(sm + 6 * NE + 1);
  int* s_u = sm + 6 * NE + 33;
  const int tid = static_cast<int>(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;
  int e_i = -1, t_i = 0;
  if (tid < P) {
    e_i = rhs[tid];
    t_i = lhs[tid];
    if (e_i < 0 || e_i >= E || t_i < 0 || t_i >= T) {
      atomicOr(&g_qmm_status, kStatusBadGather);
      e_i = -1;
    }
    s_e[tid] = e_i;
  }
  __syncthreads();
  // first entry naming this entry's expert
  int f = -1;
  if (e_i >= 0)
    for (int j = P - 1; j >= 0; --j) f = (s_e[j] == e_i) ? j : f;
  const bool first = e_i >= 0 && f == tid;
  const unsigned int bal = __ballot_sync(0xffffffffu, first);
  if (lane == 0) s_bal[warp] = bal;
  __syncthreads();
  int slot = __popc(bal & ((1u << lane) - 1u)), u = 0;
  for (int w = 0; w < THREADS / 32; ++w) {
    const int c = __popc(s_bal[w]);
    u += c;
    if (w < warp) slot += c;
  }
  if (first) {
    s_slot[tid] = slot;
    gl.expert[slot] = e_i;
  }
  __syncthreads();
  const int my_slot = (e_i >= 0) ? s_slot[f] : -1;
  __syncthreads();
  if (tid < P) s_slot[tid] = my_slot;  // now: the slot of every entry (-1: dropped)
  __syncthreads();
  // position in (slot, entry) order
  if (my_slot >= 0) {
    int pos = 0;
    for (int j = 0; j < P; ++j) {
      const int sj = s_slot[j];
      pos += (sj >= 0 && (sj < my_slot || (sj == my_slot && j < tid))) ? 1 : 0;
    }
    gl.entry[pos] = tid;
    gl.token[pos] = t_i;
    if (first) gl.start[my_slot] = pos;
  }
  const unsigned int vb = __ballot_sync(0xffffffffu, my_slot >= 0);
  if (lane == 0) s_bal[warp] = vb;  // every read of the first ballots is behind the barriers above
  __syncthreads();
  if (tid == 0) {
    int valid = 0;
    for (int w = 0; w < THREADS / 32; ++w) valid += __popc(s_bal[w]);
    gl.start[u] = valid;
    *s_u = u;
  }
  __syncthreads();
  gl.u = *s_u;
  return gl;
}

}  // namespace qmm
