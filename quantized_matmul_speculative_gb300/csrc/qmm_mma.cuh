// Tensor-core ("mma") kernel family of libqmm.
//
// Y[M,N] = X[M,K] . dequant(Wq)[N,K]^T for M <= 16, computed as the swapped
// product Y^T = dequant(W) . X^T on warp-level bf16 MMAs (m16n8k16): the
// weights are the 16-row A operand and the <= 8 (or 16, two n8 tiles)
// activation rows are the narrow B operand.  This is the weights-as-matrix-
// operand design ("MLX quantized_matmul small-M verify kernels", fact "Fix
// family 2", mlx-dspark skinny_qmm) with per-group dequantization (same fact:
// dequantize per quantization group, not per MMA tile) and split-K across the
// warps of a block (same fact; llama.cpp PR #29869 "few-row MMA": the
// simdgroups of a threadgroup split K).
//
// Per group of g codes along K and per 16-row tile:
//   * every code is unpacked once to the exact bf16 value 128 + q (one LOP3
//     per pair, see unpack_pair) and feeds all M activation rows at once;
//   * the MMAs of the group accumulate P'[n,m] = sum_k (128 + q[n,k]) x[m,k]
//     in a fresh fp32 tile;
//   * the group's scale s and bias b are applied once to that tile:
//         acc[n,m] += s * P'[n,m] + (b - 128 s) * xsum[m]
//     with xsum[m] = sum over the group of x[m,k]; this equals
//     s * sum q x + b * sum x, the affine dequantization summed over the group
//     ("MLX quantized_matmul small-M verify kernels", fact "qmv_wide tuning":
//     the per-group scale multiply moved out of the loop).
//
// Operand layout.  Thread (g = lane/4, t = lane%4) of a warp feeds rows g and
// g+8 of the A tile at MMA columns {2t, 2t+1, 2t+8, 2t+9}, and the B fragment
// for activation row g at the same four columns.  The columns of one MMA may
// stand for any four k as long as A and B agree, so the kernel reads the
// packed words in their stored order (no weight repack) and instead stores X
// in shared memory with each word's k permuted into unpack order: within the
// chunk of 32/b codes of one word, 32-bit element i holds (x[i], x[i + 16/b]).
// Each MMA step then takes two unpacked pairs of one word and one 64-bit
// shared load of X.  The four threads of a quad read four different words of
// the same group, so every MMA stays inside one quantization group.
//
// Work split.  A CTA owns NT = 16*R*WN rows of W and one of `splits` K-ranges;
// the `splits` CTAs of a row tile form a thread-block cluster along K.  Warps
// (wn, wk) take R 16-row tiles and every WK-th group of the CTA's K-range.
// Partial sums are reduced in fixed order: across the WK warps in shared
// memory, then across the cluster through distributed shared memory, each
// CTA reducing and writing a slice of the tile.  No atomics, no scratch
// buffers in global memory.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qmm_device.cuh"
#include "qmm_gather.cuh"
#include "qmm_internal.h"

namespace qmm {

struct MmaParams {
  const uint16_t* __restrict__ X;
  const uint32_t* __restrict__ Wq;
  const uint16_t* __restrict__ S;
  const uint16_t* __restrict__ B;
  void* __restrict__ Y;
  const void* R;  // residual added to Y (Y's dtype, [M, N]), may be Y itself; null: none
  int M, N, K;
  int G;        // groups per row (K / GS)
  int gpc;      // groups per CTA K-range
  int chunk;    // groups staged in shared memory at a time
  int out_f32;
  // Gathered form (rhs null: a plain call): entry i pairs X row lhs[i] with
  // matrix rhs[i] of the stack; CTA x = slot * tiles + row tile (qmm_gather.cuh).
  const int32_t* lhs;
  const int32_t* rhs;
  int P, T, E;
  const uint8_t* S8;   // microscaled weights: E8M0 scales [N, K/32] (then S, B are unused)
  int tiles;           // CTA row tiles per matrix
  int64_t w_stride;    // packed words per matrix of the stack
  int64_t m_stride;    // scales (and biases) per matrix of the stack
};

template <int BITS, int GS, int NB, int R, int WN, int WK>
struct MmaCfg {
  static constexpr int VPW = 32 / BITS;                // codes per word
  static constexpr int HALF = VPW / 2;                 // code distance of an unpacked pair
  static constexpr int GW = GS / VPW;                  // words per group and row
  static constexpr int STEPS = GS / 16;                // k16 MMA steps per group
  static constexpr int SPW = VPW / 4;                  // MMA steps one word feeds
  static constexpr int LW = (GW >= 4) ? GW / 4 : 1;    // words a thread loads per row and group
  static constexpr int TPW = (GW >= 4) ? 1 : 4 / GW;   // threads sharing one word
  static constexpr int MP = 8 * NB;                    // activation rows held (padded)
  static constexpr int NT = 16 * R * WN;               // weight rows per CTA
  static constexpr int THREADS = 32 * WN * WK;
  static constexpr int WARPS_K = WK;
  static_assert(GW * VPW == GS, "group must hold whole words");
  static_assert(TPW * STEPS == SPW || TPW == 1, "word sharing must split the steps evenly");
};

// Shared-memory carve-up, in bytes, for a given chunk (groups staged at once).
template <class C>
struct MmaSmem {
  int rsx;       // X row stride in bf16 elements (padded by 4 to spread banks)
  int x_bytes, xs_bytes, meta_bytes, red_bytes, part_bytes;
  int xs_off, meta_off, part_off, total;
  __host__ __device__ explicit MmaSmem(int chunk) {
    rsx = chunk * C::GW * C::VPW + 4;
    x_bytes = C::MP * rsx * 2;
    xs_bytes = C::MP * chunk * 4;
    meta_bytes = C::NT * chunk * 8;
    red_bytes = C::WARPS_K * C::MP * C::NT * 4;
    part_bytes = C::MP * C::NT * 4;
    xs_off = (x_bytes + 15) & ~15;
    meta_off = (xs_off + xs_bytes + 15) & ~15;
    int staged = meta_off + meta_bytes;
    int uni = staged > red_bytes ? staged : red_bytes;
    part_off = (uni + 15) & ~15;
    total = part_off + part_bytes;
  }
};

template <int BITS, int GS, int NB, int R, int WN, int WK, int CODES>
__global__ void __launch_bounds__(32 * WN * WK, (32 * WN * WK >= 256) ? 2 : 4)
qmm_mma_kernel(const MmaParams p) {
  using C = MmaCfg<BITS, GS, NB, R, WN, WK>;
  constexpr bool E8 = CODES == kCodesAffine8;
  constexpr bool MX = CODES == kCodesMx4 || CODES == kCodesMx8 || CODES == kCodesNv4;
  static_assert(!MX || GS == (CODES == kCodesNv4 ? 16 : 32), "microscaling groups are 32 codes (nvfp4: 16)");
  static_assert(CODES != kCodesMx4 || BITS == 4, "mxfp4 codes are 4 bits");
  static_assert(CODES != kCodesNv4 || BITS == 4, "nvfp4 codes are 4 bits");
  static_assert(CODES != kCodesMx8 || BITS == 8, "mxfp8 codes are 8 bits");
  extern __shared__ __align__(16) unsigned char smem[];
  const MmaSmem<C> L(p.chunk);
  uint16_t* Xs = reinterpret_cast<uint16_t*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + L.xs_off);
  float2* meta = reinterpret_cast<float2*>(smem + L.meta_off);
  float* red = reinterpret_cast<float*>(smem);
  float* part = reinterpret_cast<float*>(smem + L.part_off);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int wn = warp % WN;
  const int wk = warp / WN;
  const int g = lane >> 2;
  const uint32_t magic = unpack_magic();  // the affine unpack's OR constant, in a register
  const int t = lane & 3;

  // Gathered form: this CTA's expert, its entries' activation rows and output
  // rows; a CTA whose slot is past the union exits (so does its whole
  // cluster, which shares blockIdx.x).
  __shared__ int g_row[C::MP], g_out[C::MP];
  int M = p.M;
  int tile = blockIdx.x;
  const uint32_t* Wq = p.Wq;
  const uint16_t* Sg = p.S;
  const uint16_t* Bg = p.B;
  const bool gathered = p.rhs != nullptr;
  // Programmatic dependent launch: the next kernel may start now.  Until the
  // previous one has finished, only the weights (which it cannot have
  // written) are touched: a plain call pulls its CTA's weight rows and
  // scales/biases into L2.  X, the index lists and Y come after the wait.
  griddep_launch_dependents();
  if (!gathered) {
    const int g_lo = blockIdx.y * p.gpc;
    const int g_hi = (g_lo + p.gpc < p.G) ? g_lo + p.gpc : p.G;
    const int64_t rw = static_cast<int64_t>(p.K) / C::VPW;
    const int bytes = (g_hi - g_lo) * C::GW * 4;    // of one row's K-range
    const int lines = (bytes + 127) / 128 + 1;       // 128-byte lines it can touch
    for (int u = tid; u < C::NT * lines; u += C::THREADS) {
      const int r = u / lines;
      const int n = tile * C::NT + r;
      if (n >= p.N || bytes <= 0) continue;
      // every address stays inside the row's range [lo, lo + bytes)
      const uintptr_t lo = reinterpret_cast<uintptr_t>(Wq + n * rw + static_cast<int64_t>(g_lo) * C::GW);
      uintptr_t a = (lo & ~static_cast<uintptr_t>(127)) + 128 * static_cast<uintptr_t>(u - r * lines);
      if (a < lo) a = lo;
      if (a < lo + bytes) prefetch_l2(reinterpret_cast<const void*>(a));
    }
    for (int r = tid; r < C::NT; r += C::THREADS) {
      const int n = tile * C::NT + r;
      if (n < p.N && g_lo < g_hi) {
        if constexpr (MX) {
          prefetch_l2(p.S8 + static_cast<int64_t>(n) * p.G + g_lo);
        } else {
          prefetch_l2(Sg + static_cast<int64_t>(n) * p.G + g_lo);
          prefetch_l2(Bg + static_cast<int64_t>(n) * p.G + g_lo);
        }
      }
    }
  }
  griddep_wait();
  if (gathered) {
    tile = blockIdx.x % p.tiles;
    int e = 0;
    if (!gather_setup<C::THREADS>(p.lhs, p.rhs, p.P, p.T, p.E, blockIdx.x / p.tiles, C::MP, g_row, g_out, &e, &M))
      return;
    Wq += e * p.w_stride;
    Sg += e * p.m_stride;
    Bg += e * p.m_stride;
  }
  auto xrow = [&](int m) { return static_cast<int64_t>(gathered ? g_row[m] : m); };
  auto yrow = [&](int m) { return static_cast<int64_t>(gathered ? g_out[m] : m); };

  const int n0 = tile * C::NT;
  const int split = blockIdx.y;
  const int cta_g0 = split * p.gpc;
  int cta_g1 = cta_g0 + p.gpc;
  if (cta_g1 > p.G) cta_g1 = p.G;
  const int64_t row_words = static_cast<int64_t>(p.K) / C::VPW;

  // Word of the group this thread loads (first of LW), in words from the group start.
  const int wofs = (C::TPW == 1) ? t * C::LW : t / C::TPW;

  // Row pointers of this thread's 2R weight rows (null for rows past N).
  const uint32_t* wrow[R][2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = n0 + wn * 16 * R + 16 * r + 8 * h + g;
      wrow[r][h] = (n < p.N) ? Wq + static_cast<int64_t>(n) * row_words + wofs : nullptr;
    }

  float acc[R][NB][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][nb][i] = 0.f;

  for (int c0 = cta_g0; c0 < cta_g1; c0 += p.chunk) {
    const int nch = (cta_g1 - c0 < p.chunk) ? cta_g1 - c0 : p.chunk;
    __syncthreads();  // previous chunk fully consumed

    // ---- stage X (permuted into unpack order) and per-group sums of X ----
    for (int u = tid; u < C::MP * nch; u += C::THREADS) {
      const int m = u / nch;
      const int jl = u - m * nch;
      const int64_t k0 = static_cast<int64_t>(c0 + jl) * GS;
      uint16_t* dst = Xs + m * L.rsx + jl * GS;
      float s = 0.f;
      if constexpr (E8) {
        // 8-bit codes as virtual nibbles: word wc holds real codes 4wc..4wc+3
        // of the group; stage (x0, x2), (16x0, 16x2), (x1, x3), (16x1, 16x3)
        // and sum the real activations (see qmm_group.cuh).
#pragma unroll
        for (int wc = 0; wc < C::GW; ++wc) {
          uint2 v = make_uint2(0, 0);
          if (m < M) v = ld_nc_v2(p.X + xrow(m) * (p.K / 2) + k0 / 2 + 4 * wc);
          const uint32_t h0 = bf16x2_times16(v.x), h1 = bf16x2_times16(v.y);
          s += bf16_lo(v.x) + bf16_hi(v.x) + bf16_lo(v.y) + bf16_hi(v.y);
          uint2* d2 = reinterpret_cast<uint2*>(dst + wc * C::VPW);
          d2[0] = make_uint2(prmt_lo(v.x, v.y), prmt_lo(h0, h1));
          d2[1] = make_uint2(prmt_hi(v.x, v.y), prmt_hi(h0, h1));
        }
      } else if constexpr (BITS == 8) {
        // native 8-bit codes: word wc holds codes 4wc..4wc+3; stage (x0, x2), (x1, x3)
#pragma unroll
        for (int wc = 0; wc < C::GW; ++wc) {
          uint2 v = make_uint2(0, 0);
          if (m < M) v = ld_nc_v2(p.X + xrow(m) * p.K + k0 + 4 * wc);
          s += bf16_lo(v.x) + bf16_hi(v.x) + bf16_lo(v.y) + bf16_hi(v.y);
          *reinterpret_cast<uint2*>(dst + wc * C::VPW) = make_uint2(prmt_lo(v.x, v.y), prmt_hi(v.x, v.y));
        }
      } else {
#pragma unroll
        for (int wc = 0; wc < C::GW; ++wc) {
          uint4 v[C::VPW / 8];
#pragma unroll
          for (int q = 0; q < C::VPW / 8; ++q) {
            if (m < M) v[q] = ld_nc_v4(p.X + xrow(m) * p.K + k0 + wc * C::VPW + 8 * q);
            else v[q] = make_uint4(0, 0, 0, 0);
          }
          const uint32_t* e = reinterpret_cast<const uint32_t*>(v);  // VPW/2 words of bf16 pairs
          uint32_t out[C::HALF];
#pragma unroll
          for (int i = 0; i < C::HALF; ++i) {
            // out[i] = (x[i], x[i + HALF]); x[j] lives in e[j/2], half j%2.
            const uint32_t a = e[i / 2];
            const uint32_t b = e[(i + C::HALF) / 2];
            out[i] = (i % 2 == 0) ? prmt_lo(a, b) : prmt_hi(a, b);
          }
#pragma unroll
          for (int j = 0; j < C::VPW / 2; ++j) s += bf16_lo(e[j]) + bf16_hi(e[j]);
          uint2* d2 = reinterpret_cast<uint2*>(dst + wc * C::VPW);
#pragma unroll
          for (int i = 0; i < C::HALF / 2; ++i) d2[i] = make_uint2(out[2 * i], out[2 * i + 1]);
        }
      }
      xsum[m * p.chunk + jl] = s;
    }
    // ---- stage (scale, bias - offset * scale) per row and group; offset 128, or 2176 for 8-bit ----
    for (int u = tid; u < C::NT * nch; u += C::THREADS) {
      const int rl = u / nch;
      const int jl = u - rl * nch;
      const int n = n0 + rl;
      float2 sb = make_float2(0.f, 0.f);
      if (n < p.N) {
        const int64_t idx = static_cast<int64_t>(n) * p.G + c0 + jl;
        if constexpr (MX) {
          const uint32_t b = p.S8[idx];  // no bias, no offset to remove
          sb = make_float2(CODES == kCodesNv4 ? e4m3_to_float(b) : e8m0_to_float(b), 0.f);
        } else {
          const float sc = __half2float(__ushort_as_half(Sg[idx]));
          const float bi = __half2float(__ushort_as_half(Bg[idx]));
          sb = make_float2(sc, fmaf(E8 ? -2176.f : -128.f, sc, bi));
        }
      }
      meta[rl * p.chunk + jl] = sb;
    }
    __syncthreads();

    // ---- main loop: groups wk, wk + WK, ... of this chunk ----
    uint32_t wcur[R][2][C::LW];
    auto load_group = [&](uint32_t (&w)[R][2][C::LW], int jl) {
      const int64_t off = static_cast<int64_t>(c0 + jl) * C::GW;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (wrow[r][h] != nullptr) {
            ld_stream<C::LW>(w[r][h], wrow[r][h] + off);
          } else {
#pragma unroll
            for (int i = 0; i < C::LW; ++i) w[r][h][i] = 0u;
          }
        }
    };

    int jl = wk;
    if (jl < nch) load_group(wcur, jl);
    for (; jl < nch; jl += WK) {
      uint32_t wnxt[R][2][C::LW];
      if (jl + WK < nch) load_group(wnxt, jl + WK);

      float tmp[R][NB][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) tmp[r][nb][i] = 0.f;

#pragma unroll
      for (int st = 0; st < C::STEPS; ++st) {
        const int lwi = (C::TPW == 1) ? st / C::SPW : 0;
        const int s = (C::TPW == 1) ? st % C::SPW : (t % C::TPW) * (C::SPW / C::TPW) + st;
        const int wi = (C::TPW == 1) ? t * C::LW + lwi : t / C::TPW;
        const int koff = (jl * C::GW + wi) * C::VPW + 4 * s;
        uint2 xb[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          xb[nb] = *reinterpret_cast<const uint2*>(Xs + (8 * nb + g) * L.rsx + koff);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          uint32_t a[4];
          auto unpack = [&](uint32_t w, int i) {
            if constexpr (CODES == kCodesMx4 || CODES == kCodesNv4) return unpack_fp4_pair(w, i);
            else if constexpr (CODES == kCodesMx8) return unpack_fp8_pair(w, i);
            else return unpack_pair<BITS>(w, i, magic);
          };
          a[0] = unpack(wcur[r][0][lwi], 2 * s);
          a[1] = unpack(wcur[r][1][lwi], 2 * s);
          a[2] = unpack(wcur[r][0][lwi], 2 * s + 1);
          a[3] = unpack(wcur[r][1][lwi], 2 * s + 1);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(tmp[r][nb], a, xb[nb].x, xb[nb].y);
        }
      }

      // fold the group's scale and bias
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const float x0 = xsum[(8 * nb + 2 * t) * p.chunk + jl];
        const float x1 = xsum[(8 * nb + 2 * t + 1) * p.chunk + jl];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int rl = wn * 16 * R + 16 * r + g;
          const float2 lo = meta[rl * p.chunk + jl];
          const float2 hi = meta[(rl + 8) * p.chunk + jl];
          acc[r][nb][0] = fmaf(lo.x, tmp[r][nb][0], fmaf(lo.y, x0, acc[r][nb][0]));
          acc[r][nb][1] = fmaf(lo.x, tmp[r][nb][1], fmaf(lo.y, x1, acc[r][nb][1]));
          acc[r][nb][2] = fmaf(hi.x, tmp[r][nb][2], fmaf(hi.y, x0, acc[r][nb][2]));
          acc[r][nb][3] = fmaf(hi.x, tmp[r][nb][3], fmaf(hi.y, x1, acc[r][nb][3]));
        }
      }

#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < C::LW; ++i) wcur[r][h][i] = wnxt[r][h][i];
    }
  }

  // ---- reduce across the WK warps (fixed order) ----
  __syncthreads();  // staging buffers are dead; `red` aliases them
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int rl = wn * 16 * R + 16 * r + g;
      const int m = 8 * nb + 2 * t;
      float* base = red + (wk * C::MP) * C::NT;
      base[m * C::NT + rl] = acc[r][nb][0];
      base[(m + 1) * C::NT + rl] = acc[r][nb][1];
      base[m * C::NT + rl + 8] = acc[r][nb][2];
      base[(m + 1) * C::NT + rl + 8] = acc[r][nb][3];
    }
  __syncthreads();

  const int E = M * C::NT;  // only rows m < M are reduced and written
  const int splits = gridDim.y;
  if (splits == 1) {
    for (int e = tid; e < E; e += C::THREADS) {
      float v = red[e];
#pragma unroll
      for (int w = 1; w < WK; ++w) v += red[w * C::MP * C::NT + e];
      const int m = e / C::NT;
      const int n = n0 + (e - m * C::NT);
      if (n < p.N) {
        const int64_t o = yrow(m) * p.N + n;
        store_y(p.Y, p.R, o, v, p.out_f32);
      }
    }
    return;
  }

  for (int e = tid; e < E; e += C::THREADS) {
    float v = red[e];
#pragma unroll
    for (int w = 1; w < WK; ++w) v += red[w * C::MP * C::NT + e];
    part[e] = v;
  }
  cluster_sync_all();  // every CTA's partial tile is complete and visible
  const uint32_t rank = cluster_ctarank();
  const int e0 = static_cast<int>((static_cast<int64_t>(E) * rank) / splits);
  const int e1 = static_cast<int>((static_cast<int64_t>(E) * (rank + 1)) / splits);
  for (int e = e0 + tid; e < e1; e += C::THREADS) {
    float v = 0.f;
    for (int q = 0; q < splits; ++q) v += ld_dsmem_f32(part + e, static_cast<uint32_t>(q));
    const int m = e / C::NT;
    const int n = n0 + (e - m * C::NT);
    if (n < p.N) {
      const int64_t o = yrow(m) * p.N + n;
      store_y(p.Y, p.R, o, v, p.out_f32);
    }
  }
  cluster_sync_all();  // keep this CTA's shared memory alive until all peers have read it
}

}  // namespace qmm
