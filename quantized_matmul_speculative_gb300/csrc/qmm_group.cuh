// Per-group arithmetic shared by the TMA kernel families: staging of the
// activations in unpack order, the tensor-core MMAs of one 16-row block of one
// quantization group, and the fold of the group's scale and bias.
//
// The dequantized weight w = s * q + b of a group is never formed.  A code q
// becomes the exact bf16 value 128 + q (see unpack_pair), the MMA computes
// P = sum_k x_k (128 + q_k) exactly in fp32 per output, and the fold adds
// s * P + (b - 128 s) * sum_k x_k.  That is the group's contribution
// s * sum x q + b * sum x of the affine dequantization ("MLX quantized_matmul
// small-M verify kernels", facts "Fix family 1" and "Group-size mechanism").
//
// 8-bit codes (E8) run on the same 4-bit machinery.  A word of four 8-bit
// codes is read as eight 4-bit "virtual" codes: byte c of the word gives the
// virtual codes lo(q) and hi(q), at virtual positions 2c and 2c + 1.  The
// activations are staged for the virtual positions as x and 16 x (16 x is
// exact in bf16), so the MMA sums x (128 + lo) + 16 x (128 + hi) =
// x (q + 2176) exactly per product, and the fold removes 2176 s sum x instead
// of 128 s sum x.  With E8 the template's (BITS, GS) are the virtual ones (4,
// 2g) and the K handed to stage_x is the virtual 2K; the word layout, the
// group count and the scale/bias layout are those of the 8-bit matrix.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

// CODES: kCodesAffine (b-bit affine), kCodesAffine8 (8-bit affine as virtual
// nibbles), or a microscaling format (kCodesMx4, kCodesMx8, kCodesNv4: the
// codes' values enter the MMA exactly, see unpack_fp4_pair / unpack_fp8_pair,
// and the fold multiplies by the group's decoded scale byte; no bias).
template <int BITS, int GS, int NB, int CODES = kCodesAffine>
struct GroupMath {
  static constexpr bool E8 = CODES == kCodesAffine8;
  static constexpr bool MX = CODES == kCodesMx4 || CODES == kCodesMx8 || CODES == kCodesNv4;
  static_assert(!E8 || BITS == 4, "8-bit codes run as virtual 4-bit codes");
  static_assert(!MX || BITS == (CODES == kCodesMx8 ? 8 : 4), "microscaling code width");
  static constexpr float OFFSET = E8 ? 2176.f : 128.f;  // sum of the unpack offsets per code
  static constexpr int VPW = 32 / BITS;               // codes per 32-bit word
  static constexpr int HALF = VPW / 2;                // code pairs per word
  static constexpr int GW = GS / VPW;                 // words per row and group
  static constexpr int STEPS = GS / 16;               // m16n8k16 steps per group
  static constexpr int SPW = VPW / 4;                 // steps per word
  static constexpr int LW = (GW >= 4) ? GW / 4 : 1;   // words of a row one thread loads per group
  static constexpr int TPW = (GW >= 4) ? 1 : 4 / GW;  // threads that share one word
  static constexpr int MP = 8 * NB;                   // activation rows held (8 or 16)

  // Stage X[m, g0*GS .. (g0 + gp)*GS) for m < M into Xs (row stride rsx
  // halves) in unpack order: within each word's chunk of 32/b codes, 32-bit
  // element i holds (x[i], x[i + 16/b]).  xsum[j * MP + m] = sum of x[m, k]
  // over group g0 + j.  A task is one chunk of one row (16 or 32 bytes); the
  // tasks of a (row, group) unit sit in adjacent lanes, which add up their sums
  // by shuffles.  Loads are issued a batch at a time before any is used.  Rows
  // m >= M are not staged: an MMA output column depends only on its own
  // activation row, and the columns of rows >= M are never stored.  Every
  // thread of [0, nthreads) must call this (warp shuffles).
  __device__ static void stage_x(const uint16_t* X, int K, int M, int g0, int gp, unsigned long long gp_magic,
                                 uint16_t* Xs, int rsx, float* xsum, int tid, int nthreads) {
    if constexpr (E8) {
      stage_x_e8(X, K / 2, M, g0, gp, gp_magic, Xs, rsx, xsum, tid, nthreads);
      return;
    } else if constexpr (BITS == 8) {
      stage_x_8(X, K, M, g0, gp, gp_magic, Xs, rsx, xsum, tid, nthreads);
      return;
    }
    constexpr int CH = GS / VPW;  // tasks per unit (2..16, divides 32)
    constexpr int TQ = VPW >= 8 ? VPW / 8 : 1;  // 16-byte loads per task (8-bit codes returned above)
    constexpr int BATCH = 4;
    static_assert(32 % CH == 0, "a unit's tasks must share a warp");
    const int ntask = M * gp * CH;
    for (int base = 0; base < ntask; base += BATCH * nthreads) {
      uint4 v[BATCH][TQ];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        const uint16_t* src =
            X + static_cast<int64_t>(m) * K + static_cast<int64_t>(g0 + j) * GS + (u - unit * CH) * VPW;
#pragma unroll
        for (int q8 = 0; q8 < TQ; ++q8) v[b][q8] = (u < ntask) ? ld_nc_v4(src + 8 * q8) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int c = u - unit * CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        const uint32_t* e = reinterpret_cast<const uint32_t*>(v[b]);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < VPW / 2; ++i) sum = add_bf16x2_f32(e[i], sum);
        if (u < ntask) {
          uint32_t out[HALF];
#pragma unroll
          for (int i = 0; i < HALF; ++i) {
            const uint32_t a = e[i / 2];
            const uint32_t bb = e[(i + HALF) / 2];
            out[i] = (i % 2 == 0) ? prmt_lo(a, bb) : prmt_hi(a, bb);
          }
          uint2* d2 = reinterpret_cast<uint2*>(Xs + m * rsx + j * GS + c * VPW);
#pragma unroll
          for (int i = 0; i < HALF / 2; ++i) d2[i] = make_uint2(out[2 * i], out[2 * i + 1]);
        }
#pragma unroll
        for (int o = CH / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (u < ntask && c == 0) xsum[j * MP + m] = sum;
      }
    }
  }

  // stage_x for 8-bit codes: a task is one packed word, i.e. 4 activations
  // x0..x3 of one row (8 bytes, real row length Kr), staged as the 8 virtual
  // values (x0, 16x0, x1, 16x1, x2, 16x2, x3, 16x3) in unpack order:
  // (x0, x2), (16x0, 16x2), (x1, x3), (16x1, 16x3).  xsum holds sums of the
  // real activations.
  __device__ static void stage_x_e8(const uint16_t* X, int Kr, int M, int g0, int gp, unsigned long long gp_magic,
                                    uint16_t* Xs, int rsx, float* xsum, int tid, int nthreads) {
    constexpr int CH = GS / VPW;  // words per row and group (8..32, divides 32)
    constexpr int GSR = GS / 2;   // real codes per group
    constexpr int BATCH = 4;
    static_assert(32 % CH == 0, "a unit's tasks must share a warp");
    const int ntask = M * gp * CH;
    for (int base = 0; base < ntask; base += BATCH * nthreads) {
      uint2 v[BATCH];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        const uint16_t* src =
            X + static_cast<int64_t>(m) * Kr + static_cast<int64_t>(g0 + j) * GSR + (u - unit * CH) * 4;
        v[b] = (u < ntask) ? ld_nc_v2(src) : make_uint2(0, 0);
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int c = u - unit * CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        float sum = add_bf16x2_f32(v[b].y, add_bf16x2_f32(v[b].x, 0.f));
        if (u < ntask) {
          const uint32_t h0 = bf16x2_times16(v[b].x), h1 = bf16x2_times16(v[b].y);
          uint2* d2 = reinterpret_cast<uint2*>(Xs + m * rsx + j * GS + c * VPW);
          d2[0] = make_uint2(prmt_lo(v[b].x, v[b].y), prmt_lo(h0, h1));
          d2[1] = make_uint2(prmt_hi(v[b].x, v[b].y), prmt_hi(h0, h1));
        }
#pragma unroll
        for (int o = CH / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (u < ntask && c == 0) xsum[j * MP + m] = sum;
      }
    }
  }

  // stage_x for native 8-bit codes (FP8 E4M3): a task is one packed word of 4
  // codes, i.e. 4 activations of one row (8 bytes), staged as (x0, x2), (x1, x3).
  __device__ static void stage_x_8(const uint16_t* X, int K, int M, int g0, int gp, unsigned long long gp_magic,
                                   uint16_t* Xs, int rsx, float* xsum, int tid, int nthreads) {
    constexpr int CH = GS / VPW;  // words per row and group
    constexpr int BATCH = 4;
    static_assert(32 % CH == 0, "a unit's tasks must share a warp");
    const int ntask = M * gp * CH;
    for (int base = 0; base < ntask; base += BATCH * nthreads) {
      uint2 v[BATCH];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        const uint16_t* src = X + static_cast<int64_t>(m) * K + static_cast<int64_t>(g0 + j) * GS + (u - unit * CH) * 4;
        v[b] = (u < ntask) ? ld_nc_v2(src) : make_uint2(0, 0);
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int u = base + b * nthreads + tid;
        const int unit = u / CH;
        const int c = u - unit * CH;
        const int m = static_cast<int>((static_cast<unsigned long long>(unit) * gp_magic) >> 32);
        const int j = unit - m * gp;
        float sum = add_bf16x2_f32(v[b].y, add_bf16x2_f32(v[b].x, 0.f));
        if (u < ntask)
          *reinterpret_cast<uint2*>(Xs + m * rsx + j * GS + c * VPW) =
              make_uint2(prmt_lo(v[b].x, v[b].y), prmt_hi(v[b].x, v[b].y));
#pragma unroll
        for (int o = CH / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (u < ntask && c == 0) xsum[j * MP + m] = sum;
      }
    }
  }

  // The A operand pair i of a packed word for this code format.
  __device__ static uint32_t unpack(uint32_t w, int i, uint32_t magic) {
    if constexpr (CODES == kCodesMx4 || CODES == kCodesNv4) return unpack_fp4_pair(w, i);
    else if constexpr (CODES == kCodesMx8) return unpack_fp8_pair(w, i);
    else return unpack_pair<BITS>(w, i, magic);
  }

  // Fragment geometry of a lane: rows g and g + 8 of the 16-row block,
  // activation columns 2t, 2t + 1 (+ 8 per activation tile), the word offset
  // of its weight words within a row and group, and (for words shared by TPW
  // threads) the first MMA step it feeds.
  struct Lane {
    int g, t, wofs, tsub;
    uint32_t magic;  // unpack_magic(), the OR constant of the affine unpack
  };
  __device__ static Lane lane_geometry(int lane) {
    Lane l;
    l.magic = unpack_magic();
    l.g = lane >> 2;
    l.t = lane & 3;
    l.wofs = (TPW == 1) ? l.t * LW : l.t / TPW;
    l.tsub = (TPW == 1) ? 0 : (l.t % TPW) * (SPW / TPW);
    return l;
  }
  // This lane's first activation element of group 0 in Xs.
  __device__ static const uint16_t* x_row(const uint16_t* Xs, int rsx, const Lane& l) {
    return Xs + l.g * rsx + l.wofs * VPW + ((TPW == 1) ? 0 : 4 * l.tsub);
  }

  // The lane's packed words of one group: row g at wp, row g + 8 at
  // wp + 8 * row_stride.
  __device__ static void load_words(const uint32_t* wp, int row_stride, uint32_t (&wl)[LW], uint32_t (&wh)[LW]) {
    ld_shared_words<LW>(wl, wp);
    ld_shared_words<LW>(wh, wp + 8 * row_stride);
  }

  // P of one group for the block (fresh accumulator): A = the unpacked codes
  // of rows g, g + 8 (from wl, wh), B = the activations at xg (the group's
  // start in this lane's row of Xs, rows 8 apart by 8 * rsx).
  __device__ static void mma(const uint32_t (&wl)[LW], const uint32_t (&wh)[LW], const uint16_t* xg, int rsx,
                             int tsub, float (&tmp)[NB][4], uint32_t magic) {
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int lwi = (TPW == 1) ? st / SPW : 0;
      const int sub = (TPW == 1) ? st % SPW : tsub + st;
      uint32_t a[4];
      a[0] = unpack(wl[lwi], 2 * sub, magic);
      a[1] = unpack(wh[lwi], 2 * sub, magic);
      a[2] = unpack(wl[lwi], 2 * sub + 1, magic);
      a[3] = unpack(wh[lwi], 2 * sub + 1, magic);
      const int ko = (TPW == 1) ? (lwi * VPW + 4 * sub) : 4 * st;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint2 xb = *reinterpret_cast<const uint2*>(xg + nb * 8 * rsx + ko);
        if (st == 0) mma_bf16_16816_z(tmp[nb], a, xb.x, xb.y);  // the group's first step starts the sum
        else mma_bf16_16816(tmp[nb], a, xb.x, xb.y);
      }
    }
  }

  // acc += s * P + (b - OFFSET s) * sum x for one group.  meta_j -> fp16 scale of
  // (row g, this group); row g + 8 at + 8 * mbw, the biases at + bofs and
  // + bofs + 8 * mbw.  xs_j -> the group's activation sums (MP floats).
  __device__ static void fold(const uint16_t* meta_j, int mbw, int bofs, const float* xs_j, int t,
                              const float (&tmp)[NB][4], float (&acc)[NB][4]) {
    const float s_lo = __half2float(__ushort_as_half(meta_j[0]));
    const float s_hi = __half2float(__ushort_as_half(meta_j[8 * mbw]));
    const float b_lo = fmaf(-OFFSET, s_lo, __half2float(__ushort_as_half(meta_j[bofs])));
    const float b_hi = fmaf(-OFFSET, s_hi, __half2float(__ushort_as_half(meta_j[bofs + 8 * mbw])));
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float2 xs = *reinterpret_cast<const float2*>(xs_j + 8 * nb + 2 * t);
      ffma2(acc[nb][0], acc[nb][1], b_lo, b_lo, xs.x, xs.y);
      ffma2(acc[nb][0], acc[nb][1], s_lo, s_lo, tmp[nb][0], tmp[nb][1]);
      ffma2(acc[nb][2], acc[nb][3], b_hi, b_hi, xs.x, xs.y);
      ffma2(acc[nb][2], acc[nb][3], s_hi, s_hi, tmp[nb][2], tmp[nb][3]);
    }
  }

  // Microscaling fold: acc += s * P with s the group's decoded scale byte
  // (E8M0, or E4M3 for nvfp4).  meta_j -> the byte of (row g, this group); row
  // g + 8 at + 8 * mbw (mbw: bytes per staged scale row).
  __device__ static void fold_mx(const uint8_t* meta_j, int mbw, const float (&tmp)[NB][4], float (&acc)[NB][4]) {
    const uint32_t blo = meta_j[0], bhi = meta_j[8 * mbw];
    const float s_lo = (CODES == kCodesNv4) ? e4m3_to_float(blo) : e8m0_to_float(blo);
    const float s_hi = (CODES == kCodesNv4) ? e4m3_to_float(bhi) : e8m0_to_float(bhi);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      ffma2(acc[nb][0], acc[nb][1], s_lo, s_lo, tmp[nb][0], tmp[nb][1]);
      ffma2(acc[nb][2], acc[nb][3], s_hi, s_hi, tmp[nb][2], tmp[nb][3]);
    }
  }
};

}  // namespace qmm
