// Device helpers for the libqmm kernels (sm_103a): inline PTX wrappers for
// streaming loads, the bf16 tensor-core MMA, thread-block-cluster barriers and
// distributed shared memory, and the code -> bf16 unpack.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

// Trace points: a build that defines QMM_TRACE_POINT(id) (for instance to
// record %globaltimer per CTA) sees the phases of the kernels; the library
// build compiles them to nothing.
#ifndef QMM_TRACE_POINT
#define QMM_TRACE_POINT(id) ((void)0)
#endif

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
template <>
__device__ __forceinline__ void ld_stream<8>(uint32_t (&d)[8], const uint32_t* p) {
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]) : "l"(p));
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]) : "l"(p + 4));
}

// Read-only 16-byte load of activations (cached: every CTA of a row tile reads them).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Read-only 8-byte load of activations.
__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 v;
  asm("ld.global.nc.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Both bf16 halves of v times 16, exactly (a power-of-two scaling; finite for
// |x| < 2^124): one bf16x2 FMA, v * 16 + (-0).
__device__ __forceinline__ uint32_t bf16x2_times16(uint32_t v) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0x41804180u), "r"(0x80008000u));
  return r;
}

// ---------------------------------------------------------------------------
// Microscaling codes.  An FP4 E2M1 code s|e|m placed at bf16 bits 15 | 7-8 |
// 6 (sign, low exponent bits, top mantissa bit) is exactly 2^-126 times its
// value (exponent 0 lands on the bf16 subnormal m * 2^-127), and an FP8 E4M3
// code s|eeee|mmm placed at bits 15 | 7-10 | 4-6 is exactly 2^-120 times its
// value; one bf16x2 FMA by 2^126 or 2^120 then gives the value exactly.  A
// word's pair i holds codes i and i + 16/b, as in unpack_pair (for FP8 the
// fields move straight from their place in the word: one shift for the sign,
// one for the rest).  An E4M3 NaN code (S.1111.111) becomes a bf16 NaN: its
// exponent bits are completed to all ones before the FMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bf16x2_scale(uint32_t v, uint32_t f2) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(f2), "r"(0x80008000u));
  return r;
}
__device__ __forceinline__ uint32_t unpack_fp4_pair(uint32_t w, int i) {
  const uint32_t u = w >> (4 * i);
  const uint32_t v = ((u & 0x00070007u) << 6) | ((u & 0x00080008u) << 12);
  return bf16x2_scale(v, 0x7E807E80u);  // 2^126
}
__device__ __forceinline__ uint32_t unpack_fp8_pair(uint32_t w, int i) {
  // codes i and i + 2: sign bits 8i + 7 and 8i + 23 to bits 15 and 31,
  // exponent and mantissa bits 8i .. 8i + 6 (and + 16) to bits 4..10 (20..26)
  const uint32_t sgn = i ? w : (w << 8);
  const uint32_t mag = (i ? (w >> 4) : (w << 4)) & 0x07F007F0u;
  // A NaN code has all seven of them set: adding 1 at bit 4 carries into bit
  // 11 of that half only (no other magnitude reaches it), and bits 11..14
  // set then make the half a bf16 NaN.
  const uint32_t nanb = (mag + 0x00100010u) & 0x08000800u;
  return bf16x2_scale((sgn & 0x80008000u) | mag | (nanb * 15u), 0x7B807B80u);  // 2^120
}
// E4M3 byte -> fp32, exactly (same placement as unpack_fp8_pair); S.1111.111 is NaN.
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
  if ((c & 0x7Fu) == 0x7Fu) return __uint_as_float(0x7FC00000u);
  const uint32_t v = ((c & 0x7Fu) << 4) | ((c & 0x80u) << 8);
  return __uint_as_float(v << 16) * 1.329227995784915872903807060280344576e36f;  // 2^120
}
// E8M0 scale byte -> fp32: 2^(E - 127); 0 is the fp32 subnormal 2^-127, 255 NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
  return __uint_as_float(e == 0 ? 0x00400000u : e == 255 ? 0x7FC00000u : (e << 23));
}

// ---------------------------------------------------------------------------
// Code unpack.  A b-bit code c is OR-ed into the low mantissa bits of the bf16
// pattern 0x4300 (= 128.0, whose unit in the last place is 1), which gives the
// bf16 value 128 + c exactly.  One 32-bit word yields two such bf16 values per
// LOP3: bits [b*i, b*i+b) land in the low half and bits [16+b*i, 16+b*i+b) in
// the high half, i.e. codes i and i + 16/b of the word.  The +128 offset is
// removed later, once per group, through the group's activation sum.
//
// The mask-and-or has two 32-bit constants, and the hardware's three-input
// logic instruction takes one immediate: with both as literals the compiler
// spends two instructions per pair.  The OR constant therefore comes in a
// register (`magic`, from unpack_magic(), made once per thread), which keeps
// the pair at one logic instruction (plus the shift for i > 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t unpack_magic() {
  // %laneid >> 5 is always 0; the compiler cannot know it, so the constant
  // stays in a register instead of being folded back into an immediate.
  uint32_t z;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(z));
  return 0x43004300u | (z >> 5);
}
template <int BITS>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, int i, uint32_t magic) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  constexpr uint32_t kMask2 = kMask | (kMask << 16);
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w >> (BITS * i)), "n"(kMask2), "r"(magic));  // (a & b) | c
  return r;
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

// The same with a zero accumulator input: d = a * b (the first MMA of a group
// needs no zeroed registers).
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
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

// s + lo(v) + hi(v) in fp32, evaluated as hi + (lo + s): the two bf16 halves
// of v are widened exactly and each add rounds to fp32 (one mixed-precision
// add per half, sm_100+).
__device__ __forceinline__ float add_bf16x2_f32(uint32_t v, float s) {
  float d;
  asm("{\n .reg .b16 lo, hi;\n .reg .f32 t;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.bf16 t, lo, %2;\n"
      " add.rn.f32.bf16 %0, hi, t;\n}\n"
      : "=f"(d) : "r"(v), "f"(s));
  return d;
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

// ---------------------------------------------------------------------------
// mbarriers, TMA and cp.async (sm_90+ async proxy), programmatic dependent launch.
// ---------------------------------------------------------------------------
// Device status word: bit flags set by kernels that gave up a bounded wait.
// Each translation unit holds its own word (no relocatable device code); the
// host reads and clears all of them through qmm_device_status().
static __device__ unsigned int g_qmm_status = 0;
constexpr unsigned int kStatusTimeoutFull = 1u;   // a consumer gave up waiting for a tile
constexpr unsigned int kStatusTimeoutEmpty = 2u;  // the producer gave up waiting for a free stage
constexpr unsigned int kStatusTimeoutDrain = 4u;  // copies still in flight at exit gave up
constexpr unsigned int kStatusBadGather = 8u;     // a gathered call had an index out of range, or more
                                                  // entries for one expert than its activation tile holds
// Time after which a wait is abandoned (ns).  Far above any legitimate wait.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Test the phase with the given parity; a thread whose phase is not complete
// is suspended by the hardware until it completes or `hint_ns` elapses, so a
// waiting warp does not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// `limit_ns` (kWaitLimitNs unless a test asks for less), sets `flag` in the
// status word and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int flag,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity, 20000u)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity, 20000u)) return true;
    __nanosleep(64);
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(&g_qmm_status, flag);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes)
               : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// 4-byte asynchronous copy global -> shared (L2 only).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once all of this thread's prior cp.async copies have landed
// (the pending count is raised by one now and lowered on completion).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" :: "l"(p)); }

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Vector load of 1, 2 or 4 consecutive 32-bit words from shared memory (the
// address is aligned to the vector size by construction).
template <int N>
__device__ __forceinline__ void ld_shared_words(uint32_t (&d)[N], const uint32_t* p) {
  static_assert(N == 1 || N == 2 || N == 4 || N == 8, "1, 2, 4 or 8 words");
  if constexpr (N == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint4 w = *reinterpret_cast<const uint4*>(p + 4);
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    d[4] = w.x; d[5] = w.y; d[6] = w.z; d[7] = w.w;
  } else if constexpr (N == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    d[0] = v.x; d[1] = v.y;
  } else {
    d[0] = p[0];
  }
}

// Packed fp32 FMA on two lanes of a register pair (sm_100+):
// (a0, a1) = (b0 * c0 + a0, b1 * c1 + a1), each rounded once.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float b0, float b1, float c0, float c1) {
  asm("{\n .reg .b64 a, b, c;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n mov.b64 c, {%4, %5};\n"
      " fma.rn.f32x2 a, b, c, a;\n mov.b64 {%0, %1}, a;\n}\n"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// The epilogue store of one output element: Y[off] = v, or with a residual R
// (Y's dtype and layout) Y[off] = R[off] + v, added in fp32 and rounded once
// to Y's dtype.  The same thread reads R[off] before it writes Y[off], so R may
// be Y itself (an in-place residual update).
__device__ __forceinline__ void store_y(void* Y, const void* R, int64_t off, float v, int out_f32) {
  if (out_f32) {
    if (R != nullptr) v += static_cast<const float*>(R)[off];
    static_cast<float*>(Y)[off] = v;
  } else {
    if (R != nullptr) v += __bfloat162float(static_cast<const __nv_bfloat16*>(R)[off]);
    static_cast<__nv_bfloat16*>(Y)[off] = __float2bfloat16_rn(v);
  }
}

// Split cluster barrier: arrive now, wait (acquire) later.  The arrive is
// relaxed: it only publishes mbarrier initializations, which
// fence.mbarrier_init.release.cluster has already ordered before it.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

// 16-byte store into the shared memory of a CTA of this cluster; completion is
// counted in bytes on that CTA's mbarrier `remote_bar`.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float4 v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
      :: "r"(remote_addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar) : "memory");
}

}  // namespace qmm
