"""Host-side geometry of the TMA kernel family, checked on the CPU.

The launcher sizes the kernel from ``csrc/qmm_geometry.h``: the K-piece of
each CTA, the TMA box widths, the shared-memory layout and the number of
partial-tile slots.  A slot count that is too small would make two warps
write the same partial tile, so it is checked here against brute force over
every way the kernel cuts a window's (tile, group) units among its warps.
The header is compiled with g++ into a small driver that prints one JSON
object per case.
"""
from __future__ import annotations

import json
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
CSRC = ROOT / "quantized_matmul_speculative_gb300" / "csrc"

DRIVER = r"""
#include <cstdio>
#include <initializer_list>
#define __host__
#define __device__
#include "qmm_geometry.h"
using namespace qmm;
int main() {
  // tma_geometry for every supported (bits, gs) and cluster size over a few K
  for (int bits : {2, 4}) for (int gs : {32, 64, 128}) for (int K : {512, 1024, 4096, 5120, 8192, 12288, 17408})
    for (int c : {1, 2, 4, 8, 16}) {
      int gp = 0, pw = 0, bw = 0, nb = 0, mbw = 0;
      const bool ok = tma_geometry(K, bits, gs, c, &gp, &pw, &bw, &nb, &mbw);
      int best = 1 << 30;
      if (ok)
        for (int n = 1; n <= gp; ++n)
          if (gp % n == 0 && pw / n <= 256 && (pw / n) % 4 == 0) {
            const int w = tma_box_wavefronts(pw / n, gs * bits / 32);
            best = w < best ? w : best;
          }
      printf("{\"kind\":\"geom\",\"bits\":%d,\"gs\":%d,\"K\":%d,\"c\":%d,\"ok\":%d,\"gp\":%d,\"pw\":%d,"
             "\"bw\":%d,\"nb\":%d,\"mbw\":%d,\"wf\":%d,\"best_wf\":%d}\n",
             bits, gs, K, c, ok ? 1 : 0, gp, pw, bw, nb, mbw, ok ? tma_box_wavefronts(bw, gs * bits / 32) : 0,
             ok ? best : 0);
    }
  // tma_slots against brute force: a window of `tiles` tiles of gp groups cut
  // into w ranges [u*U/w, (u+1)*U/w); the most ranges meeting one tile.
  for (int w : {4, 8, 12, 16}) for (int gp = 1; gp <= 96; ++gp) for (int tiles = 1; tiles <= 20; ++tiles) {
    const int U = tiles * gp;
    int worst = 0;
    for (int t = 0; t < tiles; ++t) {
      int meet = 0;
      for (int u = 0; u < w; ++u) {
        const int a = u * U / w, b = (u + 1) * U / w;
        if (a < b && a < (t + 1) * gp && b > t * gp) ++meet;
      }
      worst = meet > worst ? meet : worst;
    }
    const int s = tma_slots(tiles, gp, w);
    if (s < worst) printf("{\"kind\":\"slots_bad\",\"w\":%d,\"gp\":%d,\"tiles\":%d,\"slots\":%d,\"need\":%d}\n", w, gp, tiles, s, worst);
  }
  // layout: regions in order, aligned, no overlap
  for (int mp : {8, 16}) for (int st : {2, 9, 16}) for (int rt : {1, 9}) for (int recv : {0, 3}) {
    const TmaLayout L(160, 20, 64, mp, st, rt, 3, 24, recv, 4);
    printf("{\"kind\":\"layout\",\"mp\":%d,\"stages\":%d,\"rt\":%d,\"recv\":%d,\"stage_bytes\":%d,\"w_bytes\":%d,"
           "\"meta_bytes\":%d,\"stage_off\":%d,\"x_off\":%d,\"xs_off\":%d,\"part_off\":%d,\"recv_off\":%d,\"total\":%d,\"rsx\":%d}\n",
           mp, st, rt, recv, L.stage_bytes, L.w_bytes, L.meta_bytes, L.stage_off, L.x_off, L.xs_off, L.part_off,
           L.recv_off, L.total, L.rsx);
  }
  printf("{\"kind\":\"budget\",\"one\":%d,\"two\":%d}\n", tma_smem_budget(233472, 232448, 1), tma_smem_budget(233472, 232448, 2));
  // cluster split: begins from 0 to tiles, non-decreasing, every cluster within one tile of
  // the even share, the larger shares first
  int bad_split = 0, splits = 0;
  for (int tiles = 1; tiles <= 2400; tiles += 7) for (int ncl = 1; ncl <= 160; ++ncl) {
    ++splits;
    bool ok = cluster_tile_begin(tiles, ncl, 0) == 0 && cluster_tile_begin(tiles, ncl, ncl) == tiles;
    int prev = tiles;
    for (int q = 0; q < ncl; ++q) {
      const int n = cluster_tile_begin(tiles, ncl, q + 1) - cluster_tile_begin(tiles, ncl, q);
      ok = ok && n >= tiles / ncl && n <= (tiles + ncl - 1) / ncl && n <= prev;
      prev = n;
    }
    bad_split += ok ? 0 : 1;
  }
  printf("{\"kind\":\"split\",\"checked\":%d,\"bad\":%d}\n", splits, bad_split);
  // tma_slots never grows with the window's tile count (the gathered planner
  // sizes for one-tile windows as the worst case)
  int bad_mono = 0, mono = 0;
  for (int w : {4, 8, 12, 16}) for (int gp = 1; gp <= 128; ++gp) for (int n = 1; n < 64; ++n) {
    ++mono;
    bad_mono += tma_slots(n + 1, gp, w) > tma_slots(n, gp, w) ? 1 : 0;
  }
  printf("{\"kind\":\"slots_mono\",\"checked\":%d,\"bad\":%d}\n", mono, bad_mono);
  // tma_plan: every window the kernel forms gets enough partial-tile slots.  A
  // cluster of nc tiles runs rounds of rt tiles, each cut into windows of ws;
  // the warps meeting a tile of a window of n tiles are at most
  // tma_slots(n, gp, w).  Plain calls: clusters of nt_min or nt_max tiles (the
  // split gives floor or ceil); gathered calls: any count up to nt_max.  A
  // one-tile window may be met by more warps than planned only where its
  // extra partials stay in the round's own slot region past its last tile.
  long plans = 0, windows_checked = 0, bad_plan = 0, spills = 0;
  for (int gathered = 0; gathered < 2; ++gathered)
  for (int bits : {2, 4}) for (int gs : {32, 64, 128}) for (int K : {1024, 2048, 4096, 5120, 8192, 17408})
  for (int N : {64, 136, 1024, 1536, 4096, 5120, 7168, 8192, 24576, 34816})
  for (int c : {1, 2, 4, 8, 16}) for (int wcfg = 0; wcfg < 4; ++wcfg) for (int mp : {8, 16}) {
    const int w = wcfg == 0 ? 4 : (wcfg == 3 ? 16 : 8), cps = wcfg < 2 ? 2 : 1;
    int gp = 0, pw = 0, bw = 0, nb = 0, mbw = 0;
    if (!tma_geometry(K, bits, gs, c, &gp, &pw, &bw, &nb, &mbw)) continue;
    const int tiles = (N + 15) / 16 * (gathered ? 8 : 1);
    int ncl = (148 * cps) / c;
    if (ncl > tiles) ncl = tiles;
    const int nt_max = (tiles + ncl - 1) / ncl;
    const int nt_min = gathered ? 1 : tiles / ncl;
    const int budget = tma_smem_budget(233472, 232448, cps) - (gathered ? (6 * 256 + 34) * 4 : 0);
    TmaPlan pl;
    if (!tma_plan(pw, gp, gs, mp, mbw, w, 16, c, nt_max, nt_min, budget, &pl)) continue;
    ++plans;
    for (int nc = gathered ? 1 : nt_min; nc <= nt_max; ++nc) {
      if (!gathered && nc != nt_min && nc != nt_max) continue;
      for (int r0 = 0; r0 < nc; r0 += pl.rt) {
        const int r1 = r0 + pl.rt < nc ? r0 + pl.rt : nc;
        for (int w0 = r0; w0 < r1; w0 += pl.ws) {
          const int w1 = w0 + pl.ws < r1 ? w0 + pl.ws : r1;
          const int n = w1 - w0, need = tma_slots(n, gp, w);
          ++windows_checked;
          if (need <= pl.slots) continue;
          const bool contained = n == 1 && w1 == r1 && (w1 - 1 - r0) * pl.slots + need <= pl.rt * pl.slots;
          if (contained && !gathered) ++spills; else ++bad_plan;
        }
      }
    }
  }
  printf("{\"kind\":\"plan\",\"plans\":%ld,\"windows\":%ld,\"bad\":%ld,\"spills\":%ld}\n", plans, windows_checked,
         bad_plan, spills);
  // warp-owned split: contributors of every tile against the definition
  // (warps with a non-empty range [begin(w), begin(w+1)) meeting the tile's units)
  int bad_contrib = 0, checked = 0;
  for (int W : {4, 8, 12, 16}) for (int kp = 1; kp <= 9; ++kp) for (int nt = 1; nt <= 40; ++nt) {
    const int U = nt * kp;
    for (int i = 0; i < nt; ++i) {
      int n_def = 0;
      int slot_def[16];
      for (int v = 0; v < W; ++v) {
        const int a = own_unit_begin(v, U, W), b2 = own_unit_begin(v + 1, U, W);
        slot_def[v] = -1;
        if (a < b2 && a < (i + 1) * kp && b2 > i * kp) slot_def[v] = n_def++;
      }
      for (int v = -1; v < W; ++v) {
        int sl;
        const int n = own_contributors(i, kp, U, W, v, &sl);
        ++checked;
        if (n != n_def || (v >= 0 && sl != slot_def[v]) || (v < 0 && sl != -1)) ++bad_contrib;
      }
    }
  }
  printf("{\"kind\":\"contrib\",\"checked\":%d,\"bad\":%d}\n", checked, bad_contrib);
  return 0;
}
"""


@pytest.fixture(scope="module")
def records(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("geom")
    src = d / "geom.cpp"
    src.write_text(DRIVER)
    exe = d / "geom"
    subprocess.run([gxx, "-std=c++17", "-O1", f"-I{CSRC}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return [json.loads(line) for line in out.splitlines() if line.strip()]


def test_geometry_invariants(records):
    geo = [r for r in records if r["kind"] == "geom"]
    assert geo
    for r in geo:
        G = r["K"] // r["gs"]
        supported = G % 8 == 0 and G % r["c"] == 0
        if not supported:
            assert not r["ok"], r
            continue
        gw = r["gs"] * r["bits"] // 32
        gp, pw = G // r["c"], (G // r["c"]) * gw
        lead = max((rank * gp) % 8 for rank in range(r["c"]))
        box_ok = any(gp % n == 0 and pw // n <= 256 and (pw // n) % 4 == 0 for n in range(1, gp + 1))
        if not r["ok"]:
            # refused only when the scale/bias box would exceed 256 halves or
            # no box of whole groups is a 16-byte multiple of <= 256 words
            assert (lead + gp + 7) // 8 * 8 > 256 or not box_ok, r
            continue
        assert r["gp"] * r["c"] == G
        assert r["pw"] == r["gp"] * gw
        assert r["bw"] * r["nb"] == r["pw"]
        assert r["bw"] <= 256 and r["bw"] % 4 == 0
        assert r["bw"] % gw == 0, "a group must not straddle two boxes"
        assert r["mbw"] % 8 == 0 and r["mbw"] <= 256
        assert r["mbw"] >= lead + r["gp"], "scale/bias box must cover every rank's piece"
        assert r["wf"] == r["best_wf"], "box width must minimise fragment-load wavefronts"


def test_slot_bound_covers_brute_force(records):
    bad = [r for r in records if r["kind"] == "slots_bad"]
    assert not bad, bad[:5]


def test_layout_regions_ordered_and_aligned(records):
    lay = [r for r in records if r["kind"] == "layout"]
    assert lay
    for r in lay:
        assert r["stage_bytes"] % 128 == 0 and r["stage_bytes"] >= r["w_bytes"] + r["meta_bytes"]
        assert r["stage_off"] >= (2 * 16 + 1) * 8, "mbarriers of up to 16 stages live below the stages"
        assert r["x_off"] == r["stage_off"] + r["stages"] * r["stage_bytes"]
        assert r["xs_off"] >= r["x_off"] + r["mp"] * r["rsx"] * 2
        assert r["part_off"] >= r["xs_off"] + 20 * r["mp"] * 4
        assert r["recv_off"] >= r["part_off"] + r["rt"] * 3 * r["mp"] * 16 * 4
        assert r["total"] == r["recv_off"] + r["recv"] * 4 * r["mp"] * 16 * 4
        for k in ("x_off", "xs_off", "part_off", "recv_off"):
            assert r[k] % 16 == 0, k
        # rows of X are 16-byte aligned modulo 8 bytes: the uint2 stores and
        # 8-byte fragment loads stay aligned, and rows fall on different banks
        assert (r["rsx"] * 2) % 16 == 8


def test_warp_owned_contributors(records):
    """The closed form of the warp-owned split's contributor set (used when
    every warp has work) equals its definition, and so does the fallback."""
    r = [r for r in records if r["kind"] == "contrib"][0]
    assert r["checked"] > 10000 and r["bad"] == 0, r


def test_budget(records):
    """Two CTAs per SM: each gets half the SM less the 1 KB the hardware
    reserves, rounded down to 8 KB, and two such fit; a CTA alone gets the
    whole per-block opt-in limit."""
    b = [r for r in records if r["kind"] == "budget"][0]
    assert b["one"] == 232448 and b["two"] == 114688
    assert 2 * (b["two"] + 1024) <= 233472


def test_cluster_split(records):
    """The tiles of a call split over its clusters cover every tile once,
    give each cluster floor or ceil of the even share, larger shares first."""
    r = [r for r in records if r["kind"] == "split"][0]
    assert r["checked"] > 10000 and r["bad"] == 0, r


def test_slots_never_grow_with_tiles(records):
    """A window of more tiles never needs more partial-tile slots: the one-tile
    window is the worst case the gathered planner sizes for."""
    r = [r for r in records if r["kind"] == "slots_mono"][0]
    assert r["checked"] > 10000 and r["bad"] == 0, r


def test_plan_gives_every_window_its_slots(records):
    """The row-stacking family's planner (tma_plan) gives every window the
    kernel can form enough partial-tile slots: all windows of gathered calls
    (any union), and all windows of plain calls except one-tile remainder
    windows whose extra partials stay inside their round's slot region."""
    r = [r for r in records if r["kind"] == "plan"][0]
    assert r["plans"] > 1000 and r["windows"] > 10000 and r["bad"] == 0, r
