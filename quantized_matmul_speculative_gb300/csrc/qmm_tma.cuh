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
//  * Producer warp.  One elected thread streams tile after tile into a ring
//    of S shared-memory stages with 2-D TMA copies (cp.async.bulk.tensor):
//    the tile's packed words, and its fp16 scales and biases (a box from the
//    CTA's first group rounded down to 16 bytes; the overlap with the
//    neighbouring rank is served by L2), all completing on the stage's
//    "full" mbarrier.  Weights are
//    read once per call whatever M is ("Stock qmv streams the weight matrix
//    once per input row": the fix is to stream it once).
//  * Consumer warps.  Tiles are taken in windows of ws <= S/2 tiles (the
//    next window streams in meanwhile); a window's (tile, group) work is cut
//    into W equal contiguous ranges, one per consumer warp, so every warp
//    does the same number of whole groups (two at a time: two independent
//    MMA chains).  Each warp parks its partial of every
//    tile it meets in that tile's slot for it.  Every warp walks every stage
//    in order and releases it ("empty" mbarrier, W arrivals).  The
//    activations of the CTA's K-piece are staged once per kernel, in unpack
//    order, with their per-group sums.
//  * Reduction.  After the last tile, the partials of each tile are summed in
//    slot (warp) order; one cluster barrier; CTA r then sums the C
//    partials of tiles r, r+C, ... over distributed shared memory in rank
//    order and writes Y.  Deterministic, no atomics, no global scratch.
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
#include "qmm_gather.cuh"
#include "qmm_geometry.h"
#include "qmm_group.cuh"

namespace qmm {

struct TmaParams {
  const uint16_t* __restrict__ X;
  const uint16_t* __restrict__ S;
  const uint16_t* __restrict__ B;
  void* __restrict__ Y;
  const void* R;  // residual added to Y (Y's dtype, [M, N]), may be Y itself; null: none
  int M, N, K;
  int G;          // groups per row
  int gp;         // groups per K-piece (G / C), even
  unsigned long long gp_magic;  // ceil(2^32 / gp): u / gp = (u * gp_magic) >> 32 for u * gp < 2^32
  int pw;         // packed words per row and K-piece
  int box_words;  // TMA box width (pw = nbox * box_words)
  int nbox;
  int tiles;      // 16-row tiles of W
  int ncl;        // clusters in the grid
  int rt;         // tiles per reduction round
  int stages;     // ring depth (<= template maximum)
  int slots;      // partial-tile slots per tile (most warps that can meet one tile)
  int ws;         // tiles per work window (the warps split each window's groups evenly)
  int single;     // 1: every tile has a stage of its own (no stage is reused): a warp
                  // waits only on the tiles it computes and never releases a stage
  int push;       // 1: one reduction round, partials pushed to their owner (st.async)
  int recv_tiles; // tiles one CTA owns in the push reduction
  int mbw;        // scale/bias TMA box width in halves
  int out_f32;
  unsigned long long wait_ns;  // limit of the waits on tile data (kWaitLimitNs; shorter only under test)
  int inject;     // test only: the first tile of cluster 0 declares 16 bytes more than its copies
                  // deliver, so that its phase never completes and the waits on it give up
  // Gathered form (rhs null: a plain call).  The tensor maps span the whole
  // stack (E*N rows); tile tau is row tile tau % tpe of the expert in union
  // slot tau / tpe; every token row (M = T) is computed against it and the
  // entries naming (token, expert) receive the result.  `tiles` is then the
  // largest union's tile count; the kernel splits the actual union's tiles.
  const int32_t* lhs;
  const int32_t* rhs;
  int P, E;
  int tpe;        // 16-row tiles per matrix of the stack
  int gather_off; // byte offset of the gathered lists' shared scratch
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

template <int BITS, int GS, int NB, int W, int SMAX, bool E8, bool GATHER>
__global__ void __launch_bounds__(32 * (W + 1), (W <= 8) ? 2 : 1)
qmm_tma_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_s,
               const __grid_constant__ CUtensorMap tmap_b, const TmaParams p) {
  using C = TmaCfg<BITS, GS, NB, W, SMAX>;
  using GM = GroupMath<BITS, GS, NB, E8 ? kCodesAffine8 : kCodesAffine>;
  static_assert((2 * SMAX + 1) * 8 <= 512, "mbarriers must fit below the stages");
  const int S = p.stages;
  extern __shared__ __align__(128) unsigned char tma_smem[];
  unsigned char* smem = tma_smem;
  const TmaLayout L(p.pw, p.gp, GS, C::MP, p.stages, p.rt, p.slots, p.mbw, p.recv_tiles, static_cast<int>(gridDim.x));
  const uint32_t sbase = smem_addr(smem);
  auto full_bar = [&](int s) { return sbase + 8u * s; };
  auto empty_bar = [&](int s) { return sbase + 8u * (SMAX + s); };
  const uint32_t recv_bar = sbase + 8u * (2 * SMAX);
  uint16_t* Xs = reinterpret_cast<uint16_t*>(smem + L.x_off);
  float* xsum = reinterpret_cast<float*>(smem + L.xs_off);
  float* part = reinterpret_cast<float*>(smem + L.part_off);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int csize = static_cast<int>(gridDim.x);  // CTAs per cluster (cluster spans x)
  const int rank = static_cast<int>(blockIdx.x);
  const int q = static_cast<int>(blockIdx.y);
  // this cluster's tiles (computed before the barrier below, which hides the
  // 64-bit divisions; a gathered call recomputes them for its actual union)
  int t_begin = cluster_tile_begin(p.tiles, p.ncl, q);
  int t_end = cluster_tile_begin(p.tiles, p.ncl, q + 1);
  const int g0 = rank * p.gp;  // first group of this CTA's K-piece

  QMM_TRACE_POINT(0);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), W);  // every consumer warp reads every stage
    }
    mbar_init(recv_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Gathered form: the index lists may be the previous call's output, so they
  // are read after the dependency wait (the weights of a gathered call cannot
  // stream before it: which experts to read is not known yet).
  constexpr bool gathered = GATHER;
  GatherLists gl;
  if constexpr (GATHER) {
    griddep_wait();
    gl = gather_lists<C::THREADS>(p.lhs, p.rhs, p.P, p.M, p.E, reinterpret_cast<int*>(smem + p.gather_off));
    const int tiles = gl.u * p.tpe;
    t_begin = cluster_tile_begin(tiles, p.ncl, q);
    t_end = cluster_tile_begin(tiles, p.ncl, q + 1);
  }
  // first weight row (of the tensor maps) of tile tau, and its first output row within its matrix
  auto tile_row = [&](int tau) {
    if constexpr (GATHER) return gl.expert[tau / p.tpe] * p.N + (tau % p.tpe) * 16;
    else return tau * 16;
  };
  auto tile_n0 = [&](int tau) {
    if constexpr (GATHER) return (tau % p.tpe) * 16;
    else return tau * 16;
  };
  // Y[m, n] of tile tau: the plain store, or one store per entry naming (token m, the tile's expert)
  auto store_tile = [&](int tau, int m, int n, float v) {
    if constexpr (!GATHER) {
      store_y(p.Y, p.R, static_cast<int64_t>(m) * p.N + n, v, p.out_f32);
    } else {
      const int sl = tau / p.tpe;
      for (int j = gl.start[sl]; j < gl.start[sl + 1]; ++j)
        if (gl.token[j] == m) store_y(p.Y, nullptr, static_cast<int64_t>(gl.entry[j]) * p.N + n, v, p.out_f32);
    }
  };
  const int nt = t_end - t_begin;
  const int nrounds = (nt + p.rt - 1) / p.rt;
  // Push reduction: tell the cluster this CTA's barriers exist (the matching
  // wait comes after the activations are staged).
  if (p.push) cluster_arrive();
  griddep_launch_dependents();

  if (warp == W) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmap);
      prefetch_tmap(&tmap_s);
      prefetch_tmap(&tmap_b);
    }
    const int mx0 = (g0 / 8) * 8;  // first scale/bias column of the box (16-byte aligned)
    const uint32_t tx_bytes = static_cast<uint32_t>(L.w_bytes + L.meta_bytes);
    const bool inject = p.inject && q == 0;
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
      if (lane == 0) {
        if (i >= S) mbar_wait(empty_bar(s), ((i / S) - 1) & 1, kStatusTimeoutEmpty);
        const int n0 = tile_row(t_begin + i);
        const uint32_t dst = smem_addr(smem + L.stage_off + s * L.stage_bytes);
        mbar_arrive_expect_tx(full_bar(s), tx_bytes + ((inject && i == 0) ? 16u : 0u));
        for (int b = 0; b < p.nbox; ++b)
          tma_load_2d(dst + static_cast<uint32_t>(b * p.box_words * 4 * 16), &tmap, rank * p.pw + b * p.box_words,
                      n0, full_bar(s));
        tma_load_2d(dst + L.w_bytes, &tmap_s, mx0, n0, full_bar(s));
        tma_load_2d(dst + L.w_bytes + L.meta_bytes / 2, &tmap_b, mx0, n0, full_bar(s));
      }
      __syncwarp();
    }
    // Drain: every copy this warp issued has landed before the CTA can exit
    // (the consumers wait on the same phases; this only matters if one of
    // them gave up).
    if (lane == 0) {
      const int first = nt > S ? nt - S : 0;
      for (int i = first; i < nt; ++i) mbar_wait(full_bar(i % S), (i / S) & 1, kStatusTimeoutDrain, p.wait_ns);
      QMM_TRACE_POINT(33);
    }
    __syncwarp();
    if (p.push) {
      cluster_wait();
      return;
    }
    while (done_round < nrounds) {
      cluster_sync_all();
      cluster_sync_all();
      ++done_round;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();  // X may be the previous call's output; Y may still be read by it
  QMM_TRACE_POINT(1);
  const int cthreads = C::CONSUMER_THREADS;
  // This CTA's K-piece of X in unpack order, with its per-group sums.
  GM::stage_x(p.X, p.K, p.M, g0, p.gp, p.gp_magic, Xs, L.rsx, xsum, tid, cthreads);
  asm volatile("bar.sync 1, %0;" :: "r"(cthreads) : "memory");  // consumers only
  // Push reduction: every CTA of the cluster has initialized its barriers
  // (waited for here, long before the first remote store, while the tiles
  // are still landing).
  if (p.push) cluster_wait();
  QMM_TRACE_POINT(2);

  const typename GM::Lane ln = GM::lane_geometry(lane);
  const int g = ln.g;
  const int t = ln.t;
  const int wofs = ln.wofs;
  const uint16_t* xrow = GM::x_row(Xs, L.rsx, ln);
  const int gpb = p.box_words / C::GW;  // groups per TMA box

  // MMAs of group j (packed words of this thread's rows at wp) into tmp (fresh per group).
  auto group_mma = [&](const uint32_t* wp, int j, float (&tmp)[NB][4]) {
    uint32_t wl[C::LW], wh[C::LW];
    GM::load_words(wp, p.box_words, wl, wh);
    GM::mma(wl, wh, xrow + j * GS, L.rsx, ln.tsub, tmp, ln.magic);
  };
  // Fold group j's scale and bias into acc.
  auto group_fold = [&](const uint16_t* meta, int j, const float (&tmp)[NB][4], float (&acc)[NB][4]) {
    GM::fold(meta + j, p.mbw, 16 * p.mbw, xsum + j * C::MP, t, tmp, acc);
  };

  int s = 0, ph = 0;  // stage and phase parity of tile i
  for (int round = 0; round < nrounds; ++round) {
    const int i_lo = round * p.rt;
    const int i_hi = (i_lo + p.rt < nt) ? i_lo + p.rt : nt;
    // The round's tiles are processed in windows of ws tiles (ws <= S/2, so
    // the next window streams in while this one is computed).  A window's
    // work, flattened to units (tile, group) in tile-major order, is cut into
    // W contiguous, equal ranges; warp w takes [ua, ub).  A tile is computed
    // by the warps whose ranges meet it; warp w parks its partial of the tile
    // in slot w - (first warp meeting the tile).
    for (int w0 = i_lo; w0 < i_hi; w0 += p.ws) {
      const int w1 = (w0 + p.ws < i_hi) ? w0 + p.ws : i_hi;
      const int U = (w1 - w0) * p.gp;
      const int ua = warp * U / W;
      const int ub = (warp + 1) * U / W;
      for (int i = w0; i < w1; ++i) {
        const int t0u = (i - w0) * p.gp;
        const int ja = (ua > t0u ? ua : t0u) - t0u;
        const int jb = (ub < t0u + p.gp ? ub : t0u + p.gp) - t0u;
        if (p.single && ja >= jb) {  // a stage of its own that this warp does not read
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
          continue;
        }
        // With stage reuse, every consumer warp waits on every stage in tile
        // order and arrives on it, so a wait is never more than one phase
        // ahead of its stage.
        QMM_TRACE_POINT(40);
        mbar_wait(full_bar(s), ph, kStatusTimeoutFull, p.wait_ns);
        QMM_TRACE_POINT(20);
        if (ja < jb) {
          const unsigned char* stage = smem + L.stage_off + s * L.stage_bytes;
          // Stage layout of the packed words: [box][16 rows][box_words]; a group
          // never straddles two boxes (box_words is a multiple of the group's words).
          const uint32_t* wstage = reinterpret_cast<const uint32_t*>(stage) + g * p.box_words + wofs;
          // scale/bias boxes: [16 rows][mbw halves] each, the piece starting at column g0 % 8;
          // meta[j] = scale(row g), meta[8 mbw + j] = scale(row g+8), then the biases.
          const uint16_t* meta = reinterpret_cast<const uint16_t*>(stage + L.w_bytes) + g * p.mbw + (g0 % 8);

          float acc[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;
          // word pointer of group j, advanced group by group across the boxes
          int bj = ja / gpb, jj = ja - (ja / gpb) * gpb;
          auto next_words = [&]() {
            const uint32_t* wp = wstage + bj * 16 * p.box_words + jj * C::GW;
            if (++jj == gpb) {
              jj = 0;
              ++bj;
            }
            return wp;
          };
          int j = ja;
          // Four independent MMA chains per step with one activation tile, two
          // with two tiles (register budget).
          for (; NB == 1 && j + 3 < jb; j += 4) {
            float tmp0[NB][4], tmp1[NB][4], tmp2[NB][4], tmp3[NB][4];
            const uint32_t* wp0 = next_words();
            const uint32_t* wp1 = next_words();
            const uint32_t* wp2 = next_words();
            const uint32_t* wp3 = next_words();
            group_mma(wp0, j, tmp0);
            group_mma(wp1, j + 1, tmp1);
            group_mma(wp2, j + 2, tmp2);
            group_mma(wp3, j + 3, tmp3);
            group_fold(meta, j, tmp0, acc);
            group_fold(meta, j + 1, tmp1, acc);
            group_fold(meta, j + 2, tmp2, acc);
            group_fold(meta, j + 3, tmp3, acc);
          }
          for (; j + 1 < jb; j += 2) {
            float tmp0[NB][4], tmp1[NB][4];
            const uint32_t* wp0 = next_words();
            const uint32_t* wp1 = next_words();
            group_mma(wp0, j, tmp0);
            group_mma(wp1, j + 1, tmp1);
            group_fold(meta, j, tmp0, acc);
            group_fold(meta, j + 1, tmp1, acc);
          }
          if (j < jb) {
            float tmp0[NB][4];
            group_mma(next_words(), j, tmp0);
            group_fold(meta, j, tmp0, acc);
          }
          QMM_TRACE_POINT(41);
          // slot of this warp in the tile: warps before it that meet the tile
          int first = warp;
          while (first > 0 && (first * U / W) > t0u) --first;
          float* pt = part + ((i - i_lo) * p.slots + (warp - first)) * (C::MP * 16);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int m = 8 * nb + 2 * t;
            pt[m * 16 + g] = acc[nb][0];
            pt[(m + 1) * 16 + g] = acc[nb][1];
            pt[m * 16 + g + 8] = acc[nb][2];
            pt[(m + 1) * 16 + g + 8] = acc[nb][3];
          }
        }
        if (!p.single) {
          __syncwarp();
          if (lane == 0) mbar_arrive(empty_bar(s));
        }
        QMM_TRACE_POINT(8);
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
    }

    // Sum the partials of each tile of the round in slot order (4 elements at
    // a time); with the push reduction, send the sum straight to the tile's
    // owner (CTA slot % C of the cluster), else park it in slot 0.
    asm volatile("bar.sync 1, %0;" :: "r"(cthreads) : "memory");
    QMM_TRACE_POINT(9);
    const int per_tile = p.M * 16;
    const int nslots = i_hi - i_lo;
    QMM_TRACE_POINT(10);
    for (int e4 = tid; e4 < nslots * (per_tile / 4); e4 += cthreads) {
      const int slot = e4 / (per_tile / 4);
      const int r = (e4 - slot * (per_tile / 4)) * 4;  // m * 16 + row
      // the tile's window and its units
      const int w0 = (slot / p.ws) * p.ws;
      const int w1 = (w0 + p.ws < nslots) ? w0 + p.ws : nslots;
      const int U = (w1 - w0) * p.gp;
      const int t0u = (slot - w0) * p.gp;
      // owner of the tile's first unit: the last warp whose range starts at or before it
      int first = W - 1;
      while (first > 0 && (first * U / W) > t0u) --first;
      float* base = part + slot * p.slots * (C::MP * 16) + r;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int w2 = first; w2 < W; ++w2) {
        const int a2 = w2 * U / W, b2 = (w2 + 1) * U / W;
        if (a2 >= t0u + p.gp) break;
        if (a2 < b2) {
          const float4 x4 = *reinterpret_cast<const float4*>(base + (w2 - first) * C::MP * 16);
          v.x += x4.x;
          v.y += x4.y;
          v.z += x4.z;
          v.w += x4.w;
        }
      }
      if (p.push) {
        const uint32_t q = static_cast<uint32_t>(slot % csize);
        const int o = slot / csize;
        const uint32_t dst = smem_addr(smem + L.recv_off) + 4u * static_cast<uint32_t>((o * csize + rank) * C::MP * 16 + r);
        st_async_v4(mapa_shared(dst, q), v, mapa_shared(recv_bar, q));
      } else {
        *reinterpret_cast<float4*>(base) = v;
      }
    }
    if (p.push) {
      // Owned tiles: slot % C == rank.  Wait for every peer's bytes, sum the
      // C partials in rank order, write Y.
      const int owned = (nslots > rank) ? (nslots - rank + csize - 1) / csize : 0;
      if (tid == 0) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(owned * csize * per_tile * 4));
      // (never the test's short limit: peers still push into this CTA)
      QMM_TRACE_POINT(11);
      if (owned > 0) mbar_wait(recv_bar, 0, kStatusTimeoutFull);
      QMM_TRACE_POINT(12);
      const float* recv = reinterpret_cast<const float*>(smem + L.recv_off);
      for (int e = tid; e < owned * per_tile; e += cthreads) {
        const int o = e / per_tile;
        const int r = e - o * per_tile;
        float v = 0.f;
        for (int r2 = 0; r2 < csize; ++r2) v += recv[(o * csize + r2) * C::MP * 16 + r];
        const int i = i_lo + o * csize + rank;
        const int m = r >> 4;
        const int n = tile_n0(t_begin + i) + (r & 15);
        if (n < p.N) store_tile(t_begin + i, m, n, v);
      }
      QMM_TRACE_POINT(6);
      return;  // one round only
    }
    QMM_TRACE_POINT(3);
    cluster_sync_all();  // every CTA's partials of this round are complete
    QMM_TRACE_POINT(4);
    // CTA `rank` reduces tiles rank, rank + C, ... of the round.
    for (int i = i_lo + rank; i < i_hi; i += csize) {
      const int slot = i - i_lo;
      for (int e = tid; e < per_tile; e += cthreads) {
        const float* src = part + slot * p.slots * (C::MP * 16) + e;
        float v = 0.f;
        for (int r2 = 0; r2 < csize; ++r2) v += ld_dsmem_f32(src, static_cast<uint32_t>(r2));
        const int m = e >> 4;
        const int n = tile_n0(t_begin + i) + (e & 15);
        if (n < p.N) store_tile(t_begin + i, m, n, v);
      }
    }
    QMM_TRACE_POINT(5);
    cluster_sync_all();  // peers are done reading this CTA's partials
    QMM_TRACE_POINT(6);
  }
}

}  // namespace qmm
