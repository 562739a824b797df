// Shape constraints of the TMA kernel family, shared by the launcher and the
// dispatcher.
#pragma once

namespace qmm {

// Whether (K, bits, gs, csize) fits the TMA family's constraints: the K-piece
// of each CTA holds an even number of groups, G is even, and the piece's
// packed words split into equal TMA boxes of <= 256 words, 16-byte multiples,
// each holding whole groups.
inline bool tma_geometry(int K, int bits, int gs, int csize, int* gp, int* pw, int* box_words, int* nbox) {
  const int G = K / gs;
  if (G % 2 != 0 || G % csize != 0) return false;
  *gp = G / csize;
  if (*gp % 2 != 0) return false;
  const int gw = gs * bits / 32;
  *pw = *gp * gw;
  for (int nb = 1; nb <= *gp; ++nb) {
    if (*gp % nb != 0) continue;
    const int bw = *pw / nb;
    if (bw <= 256 && bw % 4 == 0) {
      *nbox = nb;
      *box_words = bw;
      return true;
    }
  }
  return false;
}

// Shared-memory layout of one CTA of the TMA family (bytes); the kernel and
// the launcher both use it.  `mp` = activation rows held (8 or 16), `rt` =
// partial tiles held for one reduction round.
struct TmaLayout {
  int stage_bytes, w_bytes, rsx;
  int stage_off, x_off, xs_off, part_off, total;
  __host__ __device__ TmaLayout(int pw, int gp, int gs, int mp, int stages, int rt) {
    w_bytes = 16 * pw * 4;
    stage_bytes = (w_bytes + 16 * gp * 2 * 2 + 127) & ~127;  // + scales and biases, 16 rows x gp halves each
    rsx = gp * gs + 4;
    stage_off = 128;  // the 2 * stages mbarriers live below
    x_off = stage_off + stages * stage_bytes;
    xs_off = (x_off + mp * rsx * 2 + 15) & ~15;
    part_off = (xs_off + mp * gp * 4 + 15) & ~15;
    total = part_off + rt * mp * 16 * 4;
  }
};

// Shared memory one CTA may use when `ctas_per_sm` share an SM of
// `smem_per_sm` bytes (1 KB per CTA is reserved by the hardware), capped at
// the per-block opt-in limit.
inline int tma_smem_budget(int smem_per_sm, int optin, int ctas_per_sm) {
  int b = smem_per_sm / ctas_per_sm - 1024;
  return b < optin ? b : optin;
}

}  // namespace qmm
