"""The GPU tests' allowance for a bf16 output: one round to nearest even into
bf16 moves a value by at most qmm_harness.bf16_half_ulp of the result, and
that allowance is tight (CPU only; torch's CPU conversion rounds to nearest
even)."""
import numpy as np
import torch

from qmm_harness import assert_within, bf16_half_ulp


def test_half_ulp_bounds_round_to_nearest_even():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-40, 40, size=200000))).astype(np.float32)
    r = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    err = np.abs(r - v.astype(np.float64))
    hu = bf16_half_ulp(r)
    assert np.all(err <= hu)
    assert (err / hu).max() > 0.99  # tight: some values sit next to a midpoint


def test_half_ulp_values():
    # 1.0: ulp 2^-7; the largest value of the binade below 2 has the same ulp; 2.0: 2^-6
    assert bf16_half_ulp(np.array([1.0, 1.9921875, 2.0, -3.0, 0.0])).tolist() == [2.0**-8, 2.0**-8, 2.0**-7,
                                                                                   2.0**-7, 0.0]
    # a midpoint between 1 and 1 + 2^-7 rounds to even (1.0), exactly half an ulp away
    mid = np.float32(1.0 + 2.0**-8)
    r = torch.tensor([mid]).to(torch.bfloat16).to(torch.float64).numpy()
    assert r[0] == 1.0 and abs(r[0] - float(mid)) == bf16_half_ulp(r)[0]


def test_bf16_allowance_only_when_asked():
    y_ref = np.array([2.0863660270879336])
    a_ref = np.array([3.66])
    y = np.array([2.09375])  # its bf16 rounding, 0.0074 away: outside 2e-3 * 3.66 + 1e-5
    try:
        assert_within(y, y_ref, a_ref, "fp32 bound")
    except AssertionError:
        pass
    else:
        raise AssertionError("the fp32 bound must reject a bf16 rounding error this large")
    assert_within(y, y_ref, a_ref, "bf16 output", bf16=True)
