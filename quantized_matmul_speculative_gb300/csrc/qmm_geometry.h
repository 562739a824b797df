// Shape constraints of the TMA kernel family, shared by the launcher and the
// dispatcher.
#pragma once

#ifdef __CUDACC__
#define QMM_HD __host__ __device__
#else
#define QMM_HD
#endif

namespace qmm {

// Shared-memory wavefronts of one warp's load of its weight fragment words
// from a stage whose rows are `bw` words apart, for `gw` words per group: lane
// (g = lane / 4, t = lane % 4) reads row g, lw = max(1, gw / 4) consecutive
// words at word t * lw (or word t / (4 / gw) when several lanes share a word).
// A 4-, 8- or 16-byte load is served 32, 16 or 8 lanes at a time; each such
// phase takes as many wavefronts as the most distinct words on one bank.
inline int tma_box_wavefronts(int bw, int gw) {
  const int lw = gw >= 4 ? gw / 4 : 1;
  const int tpw = gw >= 4 ? 1 : 4 / gw;
  const int per_phase = 32 / lw;
  int total = 0;
  for (int p0 = 0; p0 < 32; p0 += per_phase) {
    int words[32 * 4];
    int n = 0;
    for (int lane = p0; lane < p0 + per_phase; ++lane) {
      const int g = lane >> 2, t = lane & 3;
      const int w0 = g * bw + (tpw == 1 ? t * lw : t / tpw);
      for (int k = 0; k < lw; ++k) {
        bool seen = false;
        for (int i = 0; i < n; ++i) seen = seen || words[i] == w0 + k;
        if (!seen) words[n++] = w0 + k;
      }
    }
    int worst = 0;
    for (int bank = 0; bank < 32; ++bank) {
      int c = 0;
      for (int i = 0; i < n; ++i) c += (words[i] % 32 == bank);
      worst = c > worst ? c : worst;
    }
    total += worst;
  }
  return total;
}

// Whether (K, bits, gs, csize) fits the TMA family's constraints: G = K/gs is
// a multiple of 8 (the fp16 scale/bias rows are 16-byte strided for TMA) and
// of csize; the piece of each CTA (gp = G/csize groups) splits its packed
// words into equal TMA boxes of <= 256 words, 16-byte multiples, each holding
// whole groups.  *mbw = width in halves of the scale/bias TMA box: it starts
// at the CTA's first group rounded down to 8 halves (16 bytes) and covers the
// whole piece for every rank.
inline bool tma_geometry(int K, int bits, int gs, int csize, int* gp, int* pw, int* box_words, int* nbox,
                         int* mbw) {
  const int G = K / gs;
  if (G % 8 != 0 || G % csize != 0) return false;
  *gp = G / csize;
  const int gw = gs * bits / 32;
  *pw = *gp * gw;
  int lead = 0;  // largest (first group mod 8) over the ranks
  for (int r = 0; r < csize; ++r) {
    const int l = (r * *gp) % 8;
    if (l > lead) lead = l;
  }
  *mbw = (lead + *gp + 7) / 8 * 8;
  if (*mbw > 256) return false;
  // Among the box widths, take the one whose weight-fragment loads need the
  // fewest shared-memory wavefronts (fewer boxes on ties).
  int best = 0, best_cost = 1 << 30;
  for (int nb = 1; nb <= *gp; ++nb) {
    if (*gp % nb != 0) continue;
    const int bw = *pw / nb;
    if (bw > 256 || bw % 4 != 0) continue;
    const int cost = tma_box_wavefronts(bw, gw);
    if (cost < best_cost) {
      best_cost = cost;
      best = nb;
    }
  }
  if (best == 0) return false;
  *nbox = best;
  *box_words = *pw / best;
  return true;
}

// First 16-row tile of cluster q when `tiles` tiles are split over ncl
// clusters: every cluster gets floor(tiles / ncl) or one more, and the ones
// with one more come first.  In a chain of dependent calls the clusters are
// launched in index order as the previous call's CTAs leave, so the last
// ones start last, with the least time before the dependency wait to stream
// their weights: they get the lighter share.
QMM_HD inline int cluster_tile_begin(int tiles, int ncl, int q) {
  const int base = tiles / ncl;
  const int rem = tiles - base * ncl;
  return q * base + (q < rem ? q : rem);
}

// First unit of warp w when U units are split into W contiguous ranges.
QMM_HD inline int own_unit_begin(int w, int U, int W) {
  return static_cast<int>((static_cast<long long>(w) * U) / W);
}

// Warps whose (non-empty) unit range meets tile i (units [i*kp, (i+1)*kp)),
// and the position of warp w among them in *slot (-1 if w is not one).
QMM_HD inline int own_contributors(int i, int kp, int U, int W, int w, int* slot) {
  const int lo = i * kp, hi = (i + 1) * kp;
  if (U >= W) {
    // Every range is non-empty: the warp holding unit u is ((u + 1) W - 1) / U
    // (the largest w with floor(w U / W) <= u), and the contributors are the
    // warps from the one holding lo to the one holding hi - 1.
    const int wl = static_cast<int>((static_cast<long long>(lo + 1) * W - 1) / U);
    const int wh = static_cast<int>((static_cast<long long>(hi) * W - 1) / U);
    *slot = (w >= wl && w <= wh) ? w - wl : -1;
    return wh - wl + 1;
  }
  int n = 0;
  *slot = -1;
  for (int v = 0; v < W; ++v) {
    const int a = own_unit_begin(v, U, W), b = own_unit_begin(v + 1, U, W);
    if (a < b && a < hi && b > lo) {
      if (v == w) *slot = n;
      ++n;
    }
  }
  return n;
}

// Shared-memory layout of one CTA of the TMA family (bytes); the kernel and
// the launcher both use it.  `mp` = activation rows held (8 or 16), `rt` =
// tiles per reduction round, `slots` = partial tiles kept per tile.
struct TmaLayout {
  int stage_bytes, w_bytes, meta_bytes, rsx;
  int stage_off, x_off, xs_off, part_off, recv_off, total;
  // `recv_tiles` = tiles one CTA owns in the push reduction (0 = not used),
  // `csize` = CTAs per cluster.
  __host__ __device__ TmaLayout(int pw, int gp, int gs, int mp, int stages, int rt, int slots, int mbw,
                                int recv_tiles = 0, int csize = 1) {
    w_bytes = 16 * pw * 4;
    meta_bytes = 2 * 16 * mbw * 2;  // scales then biases, 16 rows x mbw halves each
    stage_bytes = (w_bytes + meta_bytes + 127) & ~127;
    rsx = gp * gs + 4;
    stage_off = 512;  // mbarriers live below
    x_off = stage_off + stages * stage_bytes;
    xs_off = (x_off + mp * rsx * 2 + 15) & ~15;
    part_off = (xs_off + gp * mp * 4 + 15) & ~15;
    recv_off = (part_off + rt * slots * mp * 16 * 4 + 15) & ~15;
    total = recv_off + recv_tiles * csize * mp * 16 * 4;
  }
};

// Launch plan of the row-stacking TMA family for clusters of csize CTAs that
// get nt_min..nt_max tiles each: a stage per tile (single shot) when every
// tile of a cluster fits, else a ring of up to 8 stages worked in windows of
// half the ring, reduction rounds of rt tiles (one round preferred, stages
// given up down to 4 for it), partial-tile slots for every window the kernel
// forms of the smallest cluster, and the push reduction when one round covers
// every cluster and its receive buffer still fits.  smax is the kernel's
// most stages, w its consumer warps, budget the shared memory the layout may
// take.  Returns false if no ring fits.
struct TmaPlan {
  int single, stages, ws, rt, slots, push, recv_tiles;
};

inline int tma_slots(int tiles, int gp, int w);

inline bool tma_plan(int pw, int gp, int gs, int mp, int mbw, int w, int smax, int csize, int nt_max, int nt_min,
                     int budget, TmaPlan* pl) {
  const TmaLayout base(pw, gp, gs, mp, 0, 0, 0, mbw);
  // partial slots per tile for rounds of rt tiles cut into windows of ws
  // tiles: full windows and the remainders of the smallest cluster
  auto round_slots = [&](int ws, int rt) {
    int sl = 0;
    for (int n : {ws < rt ? ws : rt, rt % ws, nt_min % rt % ws, (nt_min % rt ? nt_min % rt : rt) % ws}) {
      if (n <= 0) continue;
      const int x = tma_slots(n, gp, w);
      sl = x > sl ? x : sl;
    }
    return sl;
  };
  int stages = 0, rt = 0, slots = 0, ws = 1, single = 0;
  if (nt_max <= smax) {
    const int sl = round_slots(nt_max, nt_max);
    if (TmaLayout(pw, gp, gs, mp, nt_max, nt_max, sl, mbw).total <= budget) {
      single = 1;
      stages = nt_max;
      ws = nt_max;
      rt = nt_max;
      slots = sl;
    }
  }
  if (!single) {
    for (stages = smax < 8 ? smax : 8; stages >= 2; --stages) {
      ws = stages / 2 > 0 ? stages / 2 : 1;
      const int room = budget - base.total - stages * base.stage_bytes;
      for (rt = nt_max; rt >= 1; --rt) {
        slots = round_slots(ws, rt);
        if (rt * slots * mp * 16 * 4 <= room) break;
      }
      if (rt >= 1 && (rt == nt_max || stages <= 4)) break;
    }
    if (stages < 2 || rt < 1) return false;
  }
  pl->single = single;
  pl->stages = stages;
  pl->ws = ws;
  pl->rt = rt;
  pl->slots = slots;
  pl->push = 0;
  pl->recv_tiles = 0;
  if (rt == nt_max) {
    const int recv_tiles = (rt + csize - 1) / csize;
    if (TmaLayout(pw, gp, gs, mp, stages, rt, slots, mbw, recv_tiles, csize).total <= budget) {
      pl->push = 1;
      pl->recv_tiles = recv_tiles;
    }
  }
  return true;
}

// Partial-tile slots per tile: with units = tiles * gp groups cut into w equal
// ranges, a tile (gp units) meets at most ceil(gp / floor(units / w)) + 1
// ranges, and never more than w.
inline int tma_slots(int tiles, int gp, int w) {
  const int per = (tiles * gp) / w;
  if (per < 1) return w;
  const int s = (gp + per - 1) / per + 1;
  return s < w ? s : w;
}

// Shared memory one CTA may use when `ctas_per_sm` share an SM of
// `smem_per_sm` bytes: the hardware reserves 1 KB per CTA, and the rest is
// rounded down to 8 KB so that the co-residency the occupancy calculator
// reports is the one intended (at the exact half, two CTAs do not fit).  A
// CTA alone on its SM takes everything up to the per-block opt-in limit.
inline int tma_smem_budget(int smem_per_sm, int optin, int ctas_per_sm) {
  int b = smem_per_sm / ctas_per_sm - 1024;
  if (ctas_per_sm > 1) b = (b / 8192) * 8192;
  return b < optin ? b : optin;
}

}  // namespace qmm
