// Warp-specialized TMA kernel family ("tma") of libqmm: the production path.
//
// Same arithmetic as the register-streaming kernel (qmm_mma.cuh): codes are
// unpacked once to the exact bf16 value 128 + q, fed as the 16-row A operand
// of bf16 m16n8k16 MMAs against the <= 16 activation rows, and each group's
// scale and bias are applied once to the group's fp32 tile ("MLX
// quantized_matmul small-M verify kernels", facts "Fix family 1", "Fix family
// 2" and "qmv_wide tuning").  What changes is how the weights reach the SM
// and how work is spread over it:
//
//  * Persistent clusters.  The grid is a set of thread-block clusters of C
//    CTAs, as many as the GPU co-schedules.  Cluster q owns a contiguous,
//    balanced range of 16-row tiles of W; CTA r of the cluster owns K-piece r
//    (groups [r*G/C, (r+1)*G/C)) of every one of those tiles.  The split of K
//    across the CTAs of a block group follows "Fix family 2" (split K across
//    the simdgroups) one level up.
//  * Producer warp.  One warp streams tile after tile into a ring of S
//    shared-memory stages: the tile's packed words through a 2-D TMA copy
//    (cp.async.bulk.tensor), its fp16 scales and biases through 4-byte
//    cp.async, both completing on the stage's "full" mbarrier.  Weights are
//    read once per call whatever M is ("Stock qmv streams the weight matrix
//    once per input row": the fix is to stream it once).
//  * Consumer warps.  Each takes every wact-th tile of the cluster's range
//    (wact = the largest divisor of S that is <= W; warp w owns the stages
//    congruent to w mod wact, S/wact of them, as its private buffers),
//    computes the tile's partial Y for its K-piece from the stage, releases
//    the stage ("empty" mbarrier) and parks the partial in shared memory.
//    The activations of the CTA's K-piece are staged once per kernel, in
//    unpack order, with their per-group sums.
//  * Reduction.  After the last tile, one cluster barrier; CTA r then sums
//    the C partials of tiles r, r+C, ... over distributed shared memory in
//    rank order and writes Y.  Deterministic, no atomics, no global scratch.
//  * Programmatic dependent launch.  The producer starts streaming weights
//    before griddepcontrol.wait; activations are read and Y is written only
//    after it, so a chain of calls overlaps one call's tail with the next
//    call's weight stream.
//
// Every mbarrier wait is bounded in time (mbar_wait); a wait that gives up
// sets a flag in the device status word instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm_device.cuh"
#include "qmm_geometry.h"

namespace qmm {

struct TmaParams {
  const uint16_t* __restrict__ X;
  const uint16_t* __restrict__ S;
  const uint16_t* __restrict__ B;
  void* __restrict__ Y;
  int M, N, K;
  int G;          // groups per row
  int gp;         // groups per K-piece (G / C), even
  int pw;         // packed words per row and K-piece
  int box_words;  // TMA box width (pw = nbox * box_words)
  int nbox;
  int tiles;      // 16-row tiles of W
  int ncl;        // clusters in the grid
  int rt;         // tiles per reduction round
  int stages;     // ring depth (<= template maximum)
  int wact;       // consumer warps that take tiles (<= stages, see below)
  int out_f32;
};

template <int BITS, int GS, int NB, int W, int SMAX>
struct TmaCfg {
  static constexpr int VPW = 32 / BITS;
  static constexpr int HALF = VPW / 2;
  static constexpr int GW = GS / VPW;
  static constexpr int STEPS = GS / 16;
  static constexpr int SPW = VPW / 4;
  static constexpr int LW = (GW >= 4) ? GW / 4 : 1;
  static constexpr int TPW = (GW >= 4) ? 1 : 4 / GW;
  static constexpr int MP = 8 * NB;
  static constexpr int THREADS = 32 * (W + 1);
  static constexpr int STAGES = SMAX;
  static constexpr int CONSUMER_THREADS = 32 * W;
};

template <int BITS, int GS, int NB, int W, int SMAX>
__global__ void __launch_bounds__(32 * (W + 1), 1)
qmm_tma_kernel(const __grid_constant__ CUtensorMap tmap, const TmaParams p) {
  using C = TmaCfg<BITS, GS, NB, W, SMAX>;
  static_assert(2 * SMAX * 8 <= 128, "mbarriers must fit below the stages");
  const int S = p.stages;
  extern __shared__ __align__(128) unsigned char tma_smem[];
  unsigned char* smem = tma_smem;
  const TmaLayout L(p.pw, p.gp, GS, C::MP, p.stages, p.rt);
  const uint32_t sbase = smem_addr(smem);
  auto full_bar = [&](int s) { return sbase + 8u * s; };
  auto empty_bar = [&](int s) { return sbase + 8u * (SMAX + s); };
  uint16_t* Xs = reinterpret_cast<uint16_t*>(smem + L.x_off);
  float* xsum = reinterpret_cast<float*>(smem + L.xs_off);
  float* part = reinterpret_cast<float*>(smem + L.part_off);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int csize = static_cast<int>(gridDim.x);  // CTAs per cluster (cluster spans x)
  const int rank = static_cast<int>(blockIdx.x);
  const int q = static_cast<int>(blockIdx.y);
  const int t_begin = static_cast<int>((static_cast<int64_t>(p.tiles) * q) / p.ncl);
  const int t_end = static_cast<int>((static_cast<int64_t>(p.tiles) * (q + 1)) / p.ncl);
  const int nt = t_end - t_begin;
  const int nrounds = (nt + p.rt - 1) / p.rt;
  const int g0 = rank * p.gp;  // first group of this CTA's K-piece

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == W) {
    // ------------------------------------------------------------ producer
    if (lane == 0) prefetch_tmap(&tmap);
    const int meta_copies = 16 * p.gp;  // 4-byte words: 16 rows x (gp/2) x {scales, biases}
    const int words_per_row = p.gp / 2;
    int done_round = 0;
    for (int i = 0; i < nt; ++i) {
      // Before running S tiles into the next round, take part in the
      // reduction barriers of the round just issued.
      while (done_round < nrounds - 1 && i >= (done_round + 1) * p.rt + S) {
        cluster_sync_all();  // partials of round done_round complete
        cluster_sync_all();  // and reduced
        ++done_round;
      }
      const int s = i % S;
      if (i >= S) mbar_wait(empty_bar(s), ((i / S) - 1) & 1, kStatusTimeoutEmpty);
      const int n0 = (t_begin + i) * 16;
      unsigned char* stage = smem + L.stage_off + s * L.stage_bytes;
      const uint32_t meta_dst = smem_addr(stage + L.w_bytes);
      for (int c = lane; c < meta_copies; c += 32) {
        const int arr = c / (8 * p.gp);          // 0: scales, 1: biases
        const int rem = c - arr * 8 * p.gp;
        const int row = rem / words_per_row;
        const int wd = rem - row * words_per_row;
        const int n = n0 + row;
        if (n < p.N) {
          const uint16_t* src = (arr ? p.B : p.S) + static_cast<int64_t>(n) * p.G + g0 + 2 * wd;
          cp_async_4(meta_dst + 4u * (arr * 8 * p.gp + row * words_per_row + wd), src);
        }
      }
      cp_async_mbar_arrive(full_bar(s));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(L.w_bytes));
        const uint32_t wdst = smem_addr(stage);
        for (int b = 0; b < p.nbox; ++b)
          tma_load_2d(wdst + static_cast<uint32_t>(b * p.box_words * 4 * 16), &tmap,
                      rank * p.pw + b * p.box_words, n0, full_bar(s));
      }
    }
    // Drain: every copy this warp issued has landed before the CTA can exit
    // (the consumers wait on the same phases; this only matters if one of
    // them gave up).
    if (lane == 0) {
      const int first = nt > S ? nt - S : 0;
      for (int i = first; i < nt; ++i) mbar_wait(full_bar(i % S), (i / S) & 1, kStatusTimeoutDrain);
    }
    __syncwarp();
    while (done_round < nrounds) {
      cluster_sync_all();
      cluster_sync_all();
      ++done_round;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();  // X may be the previous call's output; Y may still be read by it
  const int cthreads = C::CONSUMER_THREADS;
  // Stage this CTA's K-piece of X in unpack order, with per-group sums.
  for (int u = tid; u < C::MP * p.gp; u += cthreads) {
    const int m = u / p.gp;
    const int jl = u - m * p.gp;
    const int64_t k0 = static_cast<int64_t>(g0 + jl) * GS;
    uint16_t* dst = Xs + m * L.rsx + jl * GS;
    float sum = 0.f;
#pragma unroll
    for (int wc = 0; wc < C::GW; ++wc) {
      uint4 v[C::VPW / 8];
#pragma unroll
      for (int qq = 0; qq < C::VPW / 8; ++qq) {
        if (m < p.M) v[qq] = ld_nc_v4(p.X + static_cast<int64_t>(m) * p.K + k0 + wc * C::VPW + 8 * qq);
        else v[qq] = make_uint4(0, 0, 0, 0);
      }
      const uint32_t* e = reinterpret_cast<const uint32_t*>(v);
      uint32_t out[C::HALF];
#pragma unroll
      for (int i = 0; i < C::HALF; ++i) {
        const uint32_t a = e[i / 2];
        const uint32_t b = e[(i + C::HALF) / 2];
        out[i] = (i % 2 == 0) ? prmt_lo(a, b) : prmt_hi(a, b);
      }
#pragma unroll
      for (int j = 0; j < C::VPW / 2; ++j) sum += bf16_lo(e[j]) + bf16_hi(e[j]);
      uint2* d2 = reinterpret_cast<uint2*>(dst + wc * C::VPW);
#pragma unroll
      for (int i = 0; i < C::HALF / 2; ++i) d2[i] = make_uint2(out[2 * i], out[2 * i + 1]);
    }
    xsum[m * p.gp + jl] = sum;
  }
  asm volatile("bar.sync 1, %0;" :: "r"(cthreads) : "memory");  // consumers only

  const int g = lane >> 2;
  const int t = lane & 3;
  const int wofs = (C::TPW == 1) ? t * C::LW : t / C::TPW;

  for (int round = 0; round < nrounds; ++round) {
    const int i_lo = round * p.rt;
    const int i_hi = (i_lo + p.rt < nt) ? i_lo + p.rt : nt;
    // Tile i goes to warp i % wact and stage i % S, and wact divides S: warp
    // w owns the stages congruent to w mod wact, so the previous phase of the
    // stage it waits on was its own earlier tile, already complete.  (An
    // mbarrier parity wait cannot tell a phase from the one two ahead.)
    for (int i = i_lo + warp; warp < p.wact && i < i_hi; i += p.wact) {
      const int s = i % S;
      mbar_wait(full_bar(s), (i / S) & 1, kStatusTimeoutFull);
      const unsigned char* stage = smem + L.stage_off + s * L.stage_bytes;
      // Stage layout of the packed words: [box][16 rows][box_words]; a group
      // never straddles two boxes (box_words is a multiple of the group's words).
      const uint32_t* wbase = reinterpret_cast<const uint32_t*>(stage) + g * p.box_words + wofs;
      const int gpb = p.box_words / C::GW;  // groups per box
      const uint16_t* sc = reinterpret_cast<const uint16_t*>(stage + L.w_bytes);
      const uint16_t* bi = sc + 16 * p.gp;

      float acc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;

      for (int jl = 0; jl < p.gp; ++jl) {
        const int bj = jl / gpb;
        const uint32_t* wlo = wbase + bj * 16 * p.box_words + (jl - bj * gpb) * C::GW;
        const uint32_t* whi = wlo + 8 * p.box_words;
        uint32_t wl[C::LW], wh[C::LW];
        ld_shared_words<C::LW>(wl, wlo);
        ld_shared_words<C::LW>(wh, whi);
        float tmp[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e) tmp[nb][e] = 0.f;
#pragma unroll
        for (int st = 0; st < C::STEPS; ++st) {
          const int lwi = (C::TPW == 1) ? st / C::SPW : 0;
          const int sub = (C::TPW == 1) ? st % C::SPW : (t % C::TPW) * (C::SPW / C::TPW) + st;
          const int wi = (C::TPW == 1) ? t * C::LW + lwi : t / C::TPW;
          const int koff = (jl * C::GW + wi) * C::VPW + 4 * sub;
          uint32_t a[4];
          a[0] = unpack_pair<BITS>(wl[lwi], 2 * sub);
          a[1] = unpack_pair<BITS>(wh[lwi], 2 * sub);
          a[2] = unpack_pair<BITS>(wl[lwi], 2 * sub + 1);
          a[3] = unpack_pair<BITS>(wh[lwi], 2 * sub + 1);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const uint2 xb = *reinterpret_cast<const uint2*>(Xs + (8 * nb + g) * L.rsx + koff);
            mma_bf16_16816(tmp[nb], a, xb.x, xb.y);
          }
        }
        const float s_lo = __half2float(__ushort_as_half(sc[g * p.gp + jl]));
        const float s_hi = __half2float(__ushort_as_half(sc[(g + 8) * p.gp + jl]));
        const float b_lo = fmaf(-128.f, s_lo, __half2float(__ushort_as_half(bi[g * p.gp + jl])));
        const float b_hi = fmaf(-128.f, s_hi, __half2float(__ushort_as_half(bi[(g + 8) * p.gp + jl])));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const float x0 = xsum[(8 * nb + 2 * t) * p.gp + jl];
          const float x1 = xsum[(8 * nb + 2 * t + 1) * p.gp + jl];
          acc[nb][0] = fmaf(s_lo, tmp[nb][0], fmaf(b_lo, x0, acc[nb][0]));
          acc[nb][1] = fmaf(s_lo, tmp[nb][1], fmaf(b_lo, x1, acc[nb][1]));
          acc[nb][2] = fmaf(s_hi, tmp[nb][2], fmaf(b_hi, x0, acc[nb][2]));
          acc[nb][3] = fmaf(s_hi, tmp[nb][3], fmaf(b_hi, x1, acc[nb][3]));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      // partial tile: part[slot][m][row]
      float* pt = part + (i - i_lo) * (C::MP * 16);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m = 8 * nb + 2 * t;
        pt[m * 16 + g] = acc[nb][0];
        pt[(m + 1) * 16 + g] = acc[nb][1];
        pt[m * 16 + g + 8] = acc[nb][2];
        pt[(m + 1) * 16 + g + 8] = acc[nb][3];
      }
    }

    cluster_sync_all();  // every CTA's partials of this round are complete
    // CTA `rank` reduces tiles rank, rank + C, ... of the round.
    const int per_tile = p.M * 16;
    for (int i = i_lo + rank; i < i_hi; i += csize) {
      const int slot = i - i_lo;
      for (int e = tid; e < per_tile; e += cthreads) {
        const int m = e >> 4;
        const int row = e & 15;
        const float* src = part + slot * (C::MP * 16) + m * 16 + row;
        float v = 0.f;
        for (int r2 = 0; r2 < csize; ++r2) v += ld_dsmem_f32(src, static_cast<uint32_t>(r2));
        const int n = (t_begin + i) * 16 + row;
        if (n < p.N) {
          const int64_t o = static_cast<int64_t>(m) * p.N + n;
          if (p.out_f32) static_cast<float*>(p.Y)[o] = v;
          else static_cast<__nv_bfloat16*>(p.Y)[o] = __float2bfloat16_rn(v);
        }
      }
    }
    cluster_sync_all();  // peers are done reading this CTA's partials
  }
}

}  // namespace qmm
