// Warp-owned TMA kernel family ("own"): every consumer warp streams its own
// work through a private ring of shared-memory stages, filled by 2-D TMA
// copies that the warp issues itself.
//
// Work.  A cluster of C CTAs takes a contiguous range of 16-row tiles of W;
// CTA `rank` of the cluster covers the K-piece of groups [rank*gp, (rank+1)*gp)
// for all of them.  Within the CTA, a tile's K-piece is cut into kp parts of
// gq groups; the (tile, part) units, tile-major, are split into W contiguous,
// equal ranges, one per warp.  A warp loads its units one by one (the copies
// of its first D-1 units are issued before the kernel waits for the previous
// call on the stream: the weights never depend on it) and keeps the running
// sum of the tile it is in.
//
// Reduction.  Tile i of the cluster belongs to CTA i mod C and, there, to warp
// (i div C) mod W.  When a warp leaves a tile it pushes its partial sums (the
// m16n8 accumulator fragments, 16 bytes per lane per activation tile) into a
// slot of the owner's receive area with st.async, which counts the bytes on the
// owner's mbarrier for that tile.  The owner waits for exactly the bytes of all
// contributors (every CTA of the cluster, every warp whose range meets the
// tile), adds the slots in a fixed order (CTA rank, then warp order) and
// writes Y.  A tile with a single contributor in a cluster of one is written
// directly.  No atomics: results are deterministic for a given launch shape.
//
// Every wait is bounded (mbar_wait); one that gives up sets a flag in the
// device status word instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm_device.cuh"
#include "qmm_gather.cuh"
#include "qmm_geometry.h"
#include "qmm_group.cuh"

namespace qmm {

struct OwnParams {
  const uint16_t* __restrict__ X;
  void* __restrict__ Y;
  const void* R;  // residual added to Y (Y's dtype, [M, N]), may be Y itself; null: none
  int M, N, K;
  int gp;                       // groups per CTA K-piece (G / C)
  unsigned long long gp_magic;  // ceil(2^32 / gp), for u / gp = (u * gp_magic) >> 32
  int kp;                       // parts per tile K-piece
  int gq;                       // groups per part (gp / kp)
  int bw, nbox;                 // weight box width (words) and boxes per unit: nbox * bw = gq * words per group
  int mbw;                      // scale/bias box width (halves); G with meta_tile
  int bofs;                     // halves from a stage's scales to its biases: 16 * mbw, or with
                                // meta_tile 16 * G rounded up to 128 bytes
  int meta_tile;                // 1: a stage holds its tile's scales and biases for all G groups
                                // ([16 rows][G] each), copied through a [rows*G/8, 8] view of the
                                // [rows, G] arrays: their rows are not 16-byte strided (G % 8 != 0);
                                // microscaling: the scale bytes, through a [rows*G/16, 16] view
  int swz;                      // 1: weight boxes are 32-word (128-byte) rows copied with the 128-byte
                                // swizzle (16-byte chunk c of box row r at c ^ (r & 7)), bw = 32
  int tiles;                    // 16-row tiles of W
  int ncl;                      // clusters in the grid
  int maxw;                     // receive slots per (tile, CTA): most warps that meet one tile
  int owned_max;                // most tiles one CTA owns
  int out_f32;
  // Gathered form (GATHER kernels): as in the TMA family, the tensor maps span
  // the stack (E*N rows), tile tau is row tile tau % tpe of the expert in
  // union slot tau / tpe, every token row (M = T) is computed against it and
  // the entries naming (token, expert) receive the result; `tiles` is the
  // largest union's tile count and the kernel splits the actual union's.
  const int32_t* lhs;
  const int32_t* rhs;
  int P, E;
  int tpe;                      // 16-row tiles per matrix of the stack
  int gather_off;               // byte offset of the gathered lists' shared scratch
};

// Shared-memory layout of one CTA (bytes).  Only the M staged activation
// rows are reserved: the MMA fragments of rows M..mp-1 read whatever lies
// after them (still inside the CTA's shared memory, which `total` guarantees),
// and those rows only feed output columns that are never stored.
struct OwnLayout {
  int x_off, xs_off, ring_off, w_bytes, stage_bytes, recv_off, slot_bytes, total, rsx;
  // meta_row: shared-memory bytes of scale/bias data per weight row of a unit
  // (affine: fp16 scales and biases, (bofs + 16 mbw) / 8, i.e. 4 mbw unless the
  // biases are placed further; microscaling: mbw scale bytes).
  // swz: swizzled weight boxes, whose destinations must be 1024-byte aligned:
  // the ring starts and every stage spans a multiple of 1024 bytes from a base
  // that the kernel aligns itself (`total` keeps 1024 bytes of slack for it).
  __host__ __device__ OwnLayout(int W, int D, int gp, int gs, int mp, int nb, int nbox, int bw, int meta_row,
                                int owned_max, int csize, int maxw, int m, int swz = 0) {
    const int nbar = W * D + owned_max;  // full barriers of the rings, then one per owned tile
    const int al = swz ? 1023 : 127;
    rsx = gp * gs + 4;                   // X row stride (halves): 8 bytes past a 16-byte multiple
    x_off = (8 * nbar + 127) & ~127;
    xs_off = (x_off + m * rsx * 2 + 15) & ~15;
    ring_off = (xs_off + gp * mp * 4 + al) & ~al;
    w_bytes = nbox * 16 * bw * 4;
    stage_bytes = (w_bytes + 16 * meta_row + al) & ~al;
    recv_off = ring_off + W * D * stage_bytes;
    slot_bytes = 32 * 16 * nb;  // 32 lanes x 4 floats x activation tiles
    total = recv_off + owned_max * csize * maxw * slot_bytes;
    const int x_end = x_off + mp * rsx * 2;  // the reads of all mp rows stay inside
    if (total < x_end) total = x_end;
    if (swz) total += 1024;
  }
};

// With W <= 8 two CTAs must fit an SM (the "2cta" shared-memory budget and
// the next call's CTAs under PDL), which caps registers at 128 per thread.
template <int BITS, int GS, int NB, int W, int D, int CODES, bool GATHER>
__global__ void __launch_bounds__(32 * W, (W <= 8) ? 2 : 1)
qmm_own_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_s,
               const __grid_constant__ CUtensorMap tmap_b, const OwnParams p) {
  using GM = GroupMath<BITS, GS, NB, CODES>;
  constexpr bool MX = GM::MX;  // one scale byte per (row, group), no bias
  constexpr int MP = GM::MP;
  constexpr int GW = GM::GW;
  extern __shared__ __align__(128) unsigned char own_smem[];
  // Swizzled weight boxes need 1024-byte aligned destinations: align the base.
  unsigned char* smem = own_smem + (p.swz ? ((1024u - (smem_addr(own_smem) & 1023u)) & 1023u) : 0u);
  const int csize = static_cast<int>(gridDim.x);  // CTAs per cluster (cluster spans x)
  const int rank = static_cast<int>(blockIdx.x);
  const int q = static_cast<int>(blockIdx.y);
  // shared memory per weight row of a stage for its metadata (bytes), and the bytes the copies deliver
  const int meta_row = MX ? p.mbw : (p.bofs + 16 * p.mbw) / 8;
  const OwnLayout L(W, D, p.gp, GS, MP, NB, p.nbox, p.bw, meta_row, p.owned_max, csize, p.maxw, p.M, p.swz);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  auto full_bar = [&](int s) { return sbase + 8u * static_cast<uint32_t>(warp * D + s); };
  auto recv_bar = [&](int o) { return sbase + 8u * static_cast<uint32_t>(W * D + o); };
  uint16_t* Xs = reinterpret_cast<uint16_t*>(smem + L.x_off);
  float* xsum = reinterpret_cast<float*>(smem + L.xs_off);

  // Gathered form: the index lists may be the previous call's output, so they
  // (and every weight copy, whose expert they decide) wait for it.
  GatherLists gl;
  int tiles = p.tiles;
  if constexpr (GATHER) {
    griddep_wait();
    gl = gather_lists<32 * W>(p.lhs, p.rhs, p.P, p.M, p.E, reinterpret_cast<int*>(smem + p.gather_off));
    tiles = gl.u * p.tpe;
  }
  auto tile_row = [&](int tau) {  // first row of tile tau in the weight tensor maps
    if constexpr (GATHER) return gl.expert[tau / p.tpe] * p.N + (tau % p.tpe) * 16;
    else return tau * 16;
  };
  auto tile_n0 = [&](int tau) {  // first output column of tile tau
    if constexpr (GATHER) return (tau % p.tpe) * 16;
    else return tau * 16;
  };
  const int t_begin = cluster_tile_begin(tiles, p.ncl, q);
  const int t_end = cluster_tile_begin(tiles, p.ncl, q + 1);
  const int nt = t_end - t_begin;
  const int g0 = rank * p.gp;
  const int U = nt * p.kp;
  const int ua = own_unit_begin(warp, U, W);
  const int nu = own_unit_begin(warp + 1, U, W) - ua;
  const int owned = (nt > rank) ? (nt - rank + csize - 1) / csize : 0;
  // Receive slots per (owned tile, CTA): the plan's, or (gathered: the tile
  // count is only known here) the most contributors any of this cluster's
  // tiles has, found by each warp over its lanes.  The planner reserved room
  // for every possible tile count.
  int maxw = p.maxw;
  if constexpr (GATHER) {
    int mw = 1;
    for (int i = lane; i < nt; i += 32) {
      int sl;
      const int n = own_contributors(i, p.kp, nt * p.kp, W, -1, &sl);
      mw = n > mw ? n : mw;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const int other = __shfl_xor_sync(0xffffffffu, mw, o);
      mw = other > mw ? other : mw;
    }
    maxw = mw;
  }
  const uint32_t unit_bytes = static_cast<uint32_t>(L.w_bytes + (MX ? 16 * p.mbw : 64 * p.mbw));

  QMM_TRACE_POINT(0);
  if (lane == 0)
    for (int s = 0; s < D; ++s) mbar_init(full_bar(s), 1);
  if (tid == 0)
    for (int o = 0; o < owned; ++o) mbar_init(recv_bar(o), 1);
  fence_mbar_init();
  __syncthreads();
  // Expected bytes of every owned tile, before any peer can push (peers push
  // only after the cluster barrier below).
  if (tid == 0) {
    for (int o = 0; o < owned; ++o) {
      int sl;
      const int n = own_contributors(o * csize + rank, p.kp, U, W, -1, &sl);
      if (!(csize == 1 && n == 1))
        mbar_arrive_expect_tx(recv_bar(o), static_cast<uint32_t>(csize * n * L.slot_bytes));
    }
  }
  cluster_arrive();
  griddep_launch_dependents();

  // Copy the unit at the issue cursor (tile ii, part ip: unit qq of this
  // warp's range) into stage qq mod D, then advance the cursor.
  int ii = ua / p.kp, ip = ua - (ua / p.kp) * p.kp;
  auto issue = [&](int qq) {
    const int i = ii;
    const int part = ip;
    if (++ip == p.kp) {
      ip = 0;
      ++ii;
    }
    const int n0 = tile_row(t_begin + i);
    const int gs0 = g0 + part * p.gq;
    const int s = qq % D;
    const uint32_t dst = sbase + static_cast<uint32_t>(L.ring_off + (warp * D + s) * L.stage_bytes);
    mbar_arrive_expect_tx(full_bar(s), unit_bytes);
    for (int b = 0; b < p.nbox; ++b)
      tma_load_2d(dst + static_cast<uint32_t>(b * 16 * p.bw * 4), &tmap, gs0 * GW + b * p.bw, n0, full_bar(s));
    if constexpr (MX) {
      if (p.meta_tile) {  // rows n0 .. n0+15 are the G view rows from n0*G/16
        const int vr = static_cast<int>((static_cast<int64_t>(n0) * p.mbw) >> 4);
        tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes), &tmap_s, 0, vr, full_bar(s));
      } else {
        const int mx0 = (gs0 / 16) * 16;  // 16-byte aligned start of the scale-byte box
        tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes), &tmap_s, mx0, n0, full_bar(s));
      }
    } else if (p.meta_tile) {
      // rows n0 .. n0+15 of a [rows, G] array are the 2G view rows from n0*G/8 (n0*G is a multiple of 8)
      const int vr = static_cast<int>((static_cast<int64_t>(n0) * p.mbw) >> 3);
      tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes), &tmap_s, 0, vr, full_bar(s));
      tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes + 2 * p.bofs), &tmap_b, 0, vr, full_bar(s));
    } else {
      const int mx0 = (gs0 / 8) * 8;  // 16-byte aligned start of the scale/bias box
      tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes), &tmap_s, mx0, n0, full_bar(s));
      tma_load_2d(dst + static_cast<uint32_t>(L.w_bytes + 2 * p.bofs), &tmap_b, mx0, n0, full_bar(s));
    }
  };
  if (lane == 0) {
    if (warp == 0) {
      prefetch_tmap(&tmap);
      prefetch_tmap(&tmap_s);
      prefetch_tmap(&tmap_b);
    }
    for (int qq = 0; qq < D - 1 && qq < nu; ++qq) issue(qq);
  }
  __syncwarp();

  griddep_wait();  // X may be the previous call's output; Y may still be read by it
  QMM_TRACE_POINT(1);
  GM::stage_x(p.X, p.K, p.M, g0, p.gp, p.gp_magic, Xs, L.rsx, xsum, tid, 32 * W);
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has initialized its barriers
  QMM_TRACE_POINT(2);

  const typename GM::Lane ln = GM::lane_geometry(lane);
  // Swizzled boxes (p.swz): GPB groups per 128-byte box row; this lane's words
  // of group jj of a box start at word sw[jj] of its row (16-byte chunk index
  // XOR the row's low three bits; rows g and g + 8 share them).  Only for
  // groups of 4..16 words per row, where a lane's words of a group lie in one
  // 16-byte chunk.
  constexpr bool SWZ_OK = GW >= 4 && GW <= 16 && 32 % GW == 0;
  constexpr int GPB = SWZ_OK ? 32 / GW : 1;
  int sw[GPB];
#pragma unroll
  for (int jj = 0; jj < GPB; ++jj) {
    const int wd = jj * GW + ln.wofs;
    sw[jj] = (((wd >> 2) ^ (ln.g & 7)) << 2) | (wd & 3);
  }
  const uint16_t* xrow = GM::x_row(Xs, L.rsx, ln);
  const int gpb = p.bw / GW;  // groups per weight box

  // Y[m, n] for this lane's fragment of tile i (gathered: one store per entry
  // naming (token m, the tile's expert)).
  auto write_y = [&](int i, const float (&v)[NB][4]) {
    const int n_lo = tile_n0(t_begin + i) + ln.g;
    const int n_hi = n_lo + 8;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 8 * nb + 2 * ln.t + (e & 1);
        const int n = (e < 2) ? n_lo : n_hi;
        if (m < p.M && n < p.N) {
          if constexpr (GATHER) {
            const int sl = (t_begin + i) / p.tpe;
            for (int j = gl.start[sl]; j < gl.start[sl + 1]; ++j)
              if (gl.token[j] == m)
                store_y(p.Y, nullptr, static_cast<int64_t>(gl.entry[j]) * p.N + n, v[nb][e], p.out_f32);
          } else {
            store_y(p.Y, p.R, static_cast<int64_t>(m) * p.N + n, v[nb][e], p.out_f32);
          }
        }
      }
    }
  };
  // Tiles strictly inside this warp's range have no other contributor.
  const int first_tile = (nu > 0) ? ua / p.kp : 0;
  const int last_tile = (nu > 0) ? (ua + nu - 1) / p.kp : -1;
  // Hand this warp's partial of tile i to the tile's owner.
  auto push = [&](int i, const float (&acc)[NB][4]) {
    int slot = 0;
    const int n = (i > first_tile && i < last_tile) ? 1 : own_contributors(i, p.kp, U, W, warp, &slot);
    if (csize == 1 && n == 1) {
      write_y(i, acc);
      return;
    }
    const uint32_t owner = static_cast<uint32_t>(i % csize);
    const int o = i / csize;
    const uint32_t dst = sbase + static_cast<uint32_t>(L.recv_off + ((o * csize + rank) * maxw + slot) * L.slot_bytes +
                                                        lane * 16 * NB);
    const uint32_t rbar = mapa_shared(recv_bar(o), owner);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
      st_async_v4(mapa_shared(dst + 16u * nb, owner), make_float4(acc[nb][0], acc[nb][1], acc[nb][2], acc[nb][3]),
                  rbar);
  };

  float acc[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;
  int cur = -1;
  bool waits_ok = true;
  int ci = ua / p.kp, cp = ua - (ua / p.kp) * p.kp;  // compute cursor: tile and part of unit qq
  for (int qq = 0; qq < nu; ++qq) {
    const int i = ci;
    const int part = cp;
    if (++cp == p.kp) {
      cp = 0;
      ++ci;
    }
    if (i != cur) {
      if (cur >= 0) {
        push(cur, acc);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;
      }
      cur = i;
    }
    // Refill the stage of unit qq - 1 with unit qq + D - 1: every lane's reads
    // of it were consumed by its MMAs before the __syncwarp that closed unit
    // qq - 1, and this lane issues the copy after that point.
    if (lane == 0 && qq + D - 1 < nu) issue(qq + D - 1);
    const int s = qq % D;
    QMM_TRACE_POINT(40);
    waits_ok = mbar_wait(full_bar(s), static_cast<uint32_t>((qq / D) & 1), kStatusTimeoutFull) && waits_ok;
    QMM_TRACE_POINT(20);
    const unsigned char* stage = smem + L.ring_off + (warp * D + s) * L.stage_bytes;
    // Weights: [box][16 rows][bw words]; a group never straddles two boxes.
    const uint32_t* wst = reinterpret_cast<const uint32_t*>(stage) + ln.g * p.bw + ln.wofs;
    // Scales then biases: [16 rows][mbw halves] each, from group (g0 + part*gq) rounded down to 8
    // (meta_tile: from group 0).
    const int gs0 = g0 + part * p.gq;
    const uint16_t* meta =
        reinterpret_cast<const uint16_t*>(stage + L.w_bytes) + ln.g * p.mbw + (p.meta_tile ? gs0 : gs0 % 8);
    // (microscaling: [16 rows][mbw scale bytes], from group gs0 rounded down to 16, or from group 0)
    const uint8_t* meta8 = stage + L.w_bytes + ln.g * p.mbw + (p.meta_tile ? gs0 : gs0 % 16);
    const int jr = part * p.gq;  // the unit's first group within the K-piece
    const uint16_t* xu = xrow + jr * GS;
    const float* xsu = xsum + jr * MP;
    // word pointer of the next group, advanced group by group across the boxes
    int bj = 0, jj = 0;
    auto next_words = [&]() {
      const uint32_t* wp = wst + bj * 16 * p.bw + jj * GW;
      if (++jj == gpb) {
        jj = 0;
        ++bj;
      }
      return wp;
    };
    auto group = [&](int j, float (&tmp)[NB][4]) {
      uint32_t wl[GM::LW], wh[GM::LW];
      GM::load_words(next_words(), p.bw, wl, wh);
      GM::mma(wl, wh, xu + j * GS, L.rsx, ln.tsub, tmp, ln.magic);
    };
    auto fold = [&](int j, const float (&tmp)[NB][4]) {
      if constexpr (MX) GM::fold_mx(meta8 + j, p.mbw, tmp, acc);
      else GM::fold(meta + j, p.mbw, p.bofs, xsu + j * MP, ln.t, tmp, acc);
    };
    int j = 0;
    if (SWZ_OK && p.swz) {
      // whole boxes of GPB groups each, the groups' word offsets known at compile time
      auto sgroup = [&](const uint32_t* bp, const int jj, int jg, float (&tmp)[NB][4]) {
        uint32_t wl[GM::LW], wh[GM::LW];
        GM::load_words(bp + sw[jj], 32, wl, wh);
        GM::mma(wl, wh, xu + jg * GS, L.rsx, ln.tsub, tmp, ln.magic);
      };
      const uint32_t* wrow = reinterpret_cast<const uint32_t*>(stage) + ln.g * 32;
      for (int b = 0; b < p.nbox; ++b) {
        const uint32_t* bp = wrow + b * 512;
        const int jb = b * GPB;
        if constexpr (NB == 1 && GPB >= 4) {
#pragma unroll
          for (int c = 0; c < GPB; c += 4) {
            float t0[NB][4], t1[NB][4], t2[NB][4], t3[NB][4];
            sgroup(bp, c, jb + c, t0);
            sgroup(bp, c + 1, jb + c + 1, t1);
            sgroup(bp, c + 2, jb + c + 2, t2);
            sgroup(bp, c + 3, jb + c + 3, t3);
            fold(jb + c, t0);
            fold(jb + c + 1, t1);
            fold(jb + c + 2, t2);
            fold(jb + c + 3, t3);
          }
        } else if constexpr (GPB >= 2) {
#pragma unroll
          for (int c = 0; c < GPB; c += 2) {
            float t0[NB][4], t1[NB][4];
            sgroup(bp, c, jb + c, t0);
            sgroup(bp, c + 1, jb + c + 1, t1);
            fold(jb + c, t0);
            fold(jb + c + 1, t1);
          }
        } else {
          float t0[NB][4];
          sgroup(bp, 0, jb, t0);
          fold(jb, t0);
        }
      }
      j = p.gq;
    }
    for (; NB == 1 && j + 3 < p.gq; j += 4) {  // four independent MMA chains
      float t0[NB][4], t1[NB][4], t2[NB][4], t3[NB][4];
      group(j, t0);
      group(j + 1, t1);
      group(j + 2, t2);
      group(j + 3, t3);
      fold(j, t0);
      fold(j + 1, t1);
      fold(j + 2, t2);
      fold(j + 3, t3);
    }
    for (; j + 1 < p.gq; j += 2) {
      float t0[NB][4], t1[NB][4];
      group(j, t0);
      group(j + 1, t1);
      fold(j, t0);
      fold(j + 1, t1);
    }
    if (j < p.gq) {
      float t0[NB][4];
      group(j, t0);
      fold(j, t0);
    }
    QMM_TRACE_POINT(41);
    __syncwarp();
  }
  if (cur >= 0) push(cur, acc);
  QMM_TRACE_POINT(3);
  // A wait that gave up may leave copies in flight: wait (bounded) for every
  // copy this warp issued before the CTA can exit.
  if (!waits_ok && lane == 0) {
    const int first = nu > D ? nu - D : 0;
    for (int qq = first; qq < nu; ++qq)
      mbar_wait(full_bar(qq % D), static_cast<uint32_t>((qq / D) & 1), kStatusTimeoutDrain);
  }
  __syncwarp();

  // Owned tiles: wait for every contributor's bytes, add the slots in order.
  for (int o = warp; o < owned; o += W) {
    const int i = o * csize + rank;
    int sl;
    const int n = own_contributors(i, p.kp, U, W, -1, &sl);
    if (csize == 1 && n == 1) continue;  // written by its only contributor
    mbar_wait(recv_bar(o), 0, kStatusTimeoutFull);
    const float* rv = reinterpret_cast<const float*>(smem + L.recv_off) +
                      static_cast<int64_t>(o * csize * maxw) * (L.slot_bytes / 4) + lane * 4 * NB;
    float v[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[nb][e] = 0.f;
    for (int r2 = 0; r2 < csize; ++r2)
      for (int k = 0; k < n; ++k) {
        const float* src = rv + (r2 * maxw + k) * (L.slot_bytes / 4);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const float4 x4 = *reinterpret_cast<const float4*>(src + 4 * nb);
          v[nb][0] += x4.x;
          v[nb][1] += x4.y;
          v[nb][2] += x4.z;
          v[nb][3] += x4.w;
        }
      }
    write_y(i, v);
  }
  QMM_TRACE_POINT(6);
}

}  // namespace qmm
