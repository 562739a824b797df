"""The dispatch-table generator (tuning/make_table.py), checked on small
synthetic sweeps: the fastest measurement wins, `_half` variants stay out of
the isolated table, chain-tuned entries override, and the microscaling table
keeps only warp-owned choices, keyed by format."""
from __future__ import annotations

import json

from quantized_matmul_speculative_gb300.tuning import make_table as mt


def _row(M, variant, vid, splits, us, N=5120, K=5120, bits=4, gs=64):
    return json.dumps({"M": M, "N": N, "K": K, "bits": bits, "gs": gs, "variant": variant, "variant_id": vid,
                       "splits": splits, "us": us})


def test_fastest_wins_and_half_variants_are_left_out():
    lines = [_row(1, "tma_w8_2cta", 3, 4, 7.5), _row(1, "tma_w4_2cta", 4, 4, 7.2),
             _row(1, "tma_own_w8_d3_half", 15, 2, 6.9), _row(8, "tma_w16_1cta", 6, 2, 8.0)]
    best = mt.best_entries(lines)
    assert best[(1, 5120, 5120, 4, 64)]["variant"] == "tma_w4_2cta"
    assert best[(8, 5120, 5120, 4, 64)]["splits"] == 2
    text = mt.render(best)
    assert text.splitlines()[4] == "{0, 0, 0, 0, 0, -1, -1},"  # the sentinel
    assert "{1, 5120, 5120, 4, 64, 4, 4},  // tma_w4_2cta 7.2 us" in text


def test_chain_entries_override():
    best = mt.best_entries([_row(2, "tma_w8_2cta", 3, 4, 7.3)])
    chain = [json.dumps({"M": 2, "N": 5120, "K": 5120, "bits": 4, "gs": 64, "variant": "tma_own_w8_d2_2cta",
                         "variant_id": 13, "splits": 2, "source": "chain", "step_ms": 1.5})]
    best.update(mt.chain_overrides(chain))
    assert "{2, 5120, 5120, 4, 64, 13, 2},  // tma_own_w8_d2_2cta chain-tuned, step 1.5 ms" in mt.render(best)


def test_mx_table_keeps_warp_owned_choices_by_format():
    lines = [json.dumps({"N": 5120, "K": 5120, "format": "nvfp4", "M": 1,
                         "best": [[9.0, "mma_r2_wn2_wk4", 1], [9.5, "tma_own_w8_d3_2cta", 2]]}),
             json.dumps({"N": 5120, "K": 5120, "format": "mxfp4", "M": 8,
                         "best": [[11.4, "tma_own_w8_d2_2cta", 2], [11.5, "tma_own_w8_d2_2cta", 4]]}),
             json.dumps({"N": 2880, "K": 2880, "format": "mxfp8", "M": 1, "best": [[7.0, "mma_r2_wn2_wk4", 2]]})]
    ids = {"tma_own_w8_d3_2cta": 9, "tma_own_w8_d2_2cta": 13, "mma_r2_wn2_wk4": 0}
    text = mt.render_mx(lines, ids)
    body = [l for l in text.splitlines() if l.startswith("{")]
    assert body[0] == "{0, 0, 0, 0, -1, -1},"
    assert "{2, 1, 5120, 5120, 9, 2},  // tma_own_w8_d3_2cta 9.5 us" in body  # nvfp4 = 2, mma skipped
    assert "{0, 8, 5120, 5120, 13, 2},  // tma_own_w8_d2_2cta 11.4 us" in body  # mxfp4 = 0
    assert len(body) == 3  # no warp-owned choice for the mxfp8 row: no entry
