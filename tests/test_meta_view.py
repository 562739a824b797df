"""Whole-tile metadata copies (CPU): where the [rows, G] scale and bias arrays
have rows that are not 16-byte strided, the warp-owned kernels copy a tile's
metadata as one box of a view with 16-byte rows.  This models that box
(elements x view rows from the tile's first view row, zero past the end) and
checks it against the arrays' definition for every tile, for the planner's
acceptance conditions: fp16 [rows*G/8, 8] boxes of 2G view rows (N*G a
multiple of 8, G <= 128), byte [rows*G/16, 16] boxes of G view rows for
microscaling scales (N*G a multiple of 16, G <= 256), tiles of a gathered
stack starting at expert*N + 16j, and the bias block placed 128-byte aligned
after the scales."""
import numpy as np
import pytest


def view_box(flat, inner, vrow0, vrows):
    """A TMA box of `inner` elements x `vrows` rows of the [len/inner, inner]
    view of `flat`, from view row vrow0; rows past the view read as 0."""
    nrows_view = len(flat) // inner
    out = np.zeros((vrows, inner), dtype=flat.dtype)
    for r in range(vrows):
        if vrow0 + r < nrows_view:
            out[r] = flat[(vrow0 + r) * inner:(vrow0 + r + 1) * inner]
    return out.reshape(-1)


def accepted(n, e, g, inner, gmax):
    rows = e * n
    return g <= gmax and (rows * g) % inner == 0 and (n * g) % inner == 0


@pytest.mark.parametrize("inner,gmax", [(8, 128), (16, 256)], ids=["fp16", "bytes"])
def test_tile_box_is_the_tile(inner, gmax):
    rng = np.random.default_rng(3)
    checked = 0
    for g in list(range(1, 40)) + [45, 60, 84, 90, 100, 120, 128, 130, 180, 256, 257]:
        for n in (1, 7, 16, 17, 18, 40, 48, 64, 72, 200):
            for e in (1, 3):
                if g % inner == 0 or not accepted(n, e, g, inner, gmax):
                    continue
                a = rng.integers(1, 1 << 15, size=(e * n, g)).astype(np.uint16)
                flat = a.reshape(-1)
                tiles = (n + 15) // 16
                for ex in range(e):
                    for j in range(tiles):
                        n0 = ex * n + 16 * j  # first row of the tile in the stacked tensor map
                        assert (n0 * g) % inner == 0, "a tile must start on a view row"
                        vrows = 16 * g // inner
                        assert 16 * g % inner == 0 and vrows <= 256, "one box per tile"
                        box = view_box(flat, inner, n0 * g // inner, vrows).reshape(16, g)
                        # rows of this expert's tile; rows past the stack read 0, rows of the
                        # next expert are read but feed outputs that are never stored
                        for r in range(16):
                            row = n0 + r
                            if row < e * n:
                                assert np.array_equal(box[r], a[row])
                            else:
                                assert not box[r].any()
                        checked += 1
    assert checked > 500


def test_acceptance_matches_the_conditions():
    """The planner's rule is exactly: every element in the view, every tile
    (and stacked matrix) on a view row, one box per tile."""
    for inner, gmax in ((8, 128), (16, 256)):
        for g in range(1, 300):
            for n in range(1, 70):
                for e in (1, 2, 5):
                    whole_view = (e * n * g) % inner == 0
                    starts = all(((ex * n + 16 * j) * g) % inner == 0
                                 for ex in range(e) for j in range((n + 15) // 16))
                    one_box = 16 * g // inner <= 256
                    assert accepted(n, e, g, inner, gmax) == (whole_view and starts and one_box
                                                              and g <= gmax), (inner, g, n, e)


def test_bias_block_offset():
    """The bias block starts 16*G halves or more after the scales, on a 128-byte
    boundary of the stage (the scale block starts on one)."""
    for g in range(1, 129):
        bofs = (16 * g + 63) // 64 * 64
        assert bofs >= 16 * g and (2 * bofs) % 128 == 0 and bofs - 16 * g < 64
