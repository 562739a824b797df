// Device helpers for the libqmm kernels (sm_103a): inline PTX wrappers for
// streaming loads, the bf16 tensor-core MMA, thread-block-cluster barriers and
// distributed shared memory, and the code -> bf16 unpack.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace qmm {

// ---------------------------------------------------------------------------
// Streaming loads of the packed weights: read once per call, so they bypass L1
// (no_allocate).
// ---------------------------------------------------------------------------
template <int WORDS>
__device__ __forceinline__ void ld_stream(uint32_t (&dst)[WORDS], const uint32_t* p);

template <>
__device__ __forceinline__ void ld_stream<1>(uint32_t (&d)[1], const uint32_t* p) {
  asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(d[0]) : "l"(p));
}
template <>
__device__ __forceinline__ void ld_stream<2>(uint32_t (&d)[2], const uint32_t* p) {
  asm("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];"
               : "=r"(d[0]), "=r"(d[1]) : "l"(p));
}
template <>
__device__ __forceinline__ void ld_stream<4>(uint32_t (&d)[4], const uint32_t* p) {
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]) : "l"(p));
}

// Read-only 16-byte load of activations (cached: every CTA of a row tile reads them).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Code unpack.  A b-bit code c is OR-ed into the low mantissa bits of the bf16
// pattern 0x4300 (= 128.0, whose unit in the last place is 1), which gives the
// bf16 value 128 + c exactly.  One 32-bit word yields two such bf16 values per
// LOP3: bits [b*i, b*i+b) land in the low half and bits [16+b*i, 16+b*i+b) in
// the high half, i.e. codes i and i + 16/b of the word.  The +128 offset is
// removed later, once per group, through the group's activation sum.
// ---------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, int i) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  constexpr uint32_t kMask2 = kMask | (kMask << 16);
  return ((w >> (BITS * i)) & kMask2) | 0x43004300u;
}

// ---------------------------------------------------------------------------
// Warp-level bf16 MMA, m16n8k16, fp32 accumulate: d += a * b.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Thread-block clusters: barrier and distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Load a float from the shared memory of CTA `rank` of this cluster, at the
// same offset as `local` has in this CTA's shared memory.
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Pair the low halves / high halves of two 32-bit words: (a.lo, b.lo), (a.hi, b.hi).
__device__ __forceinline__ uint32_t prmt_lo(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t prmt_hi(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

}  // namespace qmm
