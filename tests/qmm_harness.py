"""Shared helpers of the GPU tests: upload a synthetic problem through the
library's own packer, run it through the C ABI, and judge it against the
oracle with the acceptance bound |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-5."""
from __future__ import annotations

import numpy as np

from oracle import oracle
from quantized_matmul_speculative_gb300 import binding, synth

REL_TOL = 2e-3
ABS_TOL = 1e-5


class DeviceProblem:
    """A synth.Problem with its tensors resident on the GPU (product packing)."""

    def __init__(self, p: synth.Problem, device="cuda"):
        import torch

        self.p = p
        wq = binding.pack(p.q, p.bits)
        self.wq = torch.from_numpy(wq.view(np.int32)).to(device)
        self.s = torch.from_numpy(p.scales.view(np.float16)).to(device)
        self.b = torch.from_numpy(p.biases.view(np.float16)).to(device)
        self.x = torch.from_numpy(p.x.view(np.int16)).to(device).view(torch.bfloat16)
        self.device = device

    def run(self, M: int, out_dtype=None, variant: int = -1, splits: int = -1, out=None, allow_unsupported=False):
        """Run through the C ABI.  With ``allow_unsupported``, a forced
        (variant, splits) pair the shape cannot use returns None."""
        import torch

        out_dtype = out_dtype or torch.bfloat16
        x = self.x[:M].contiguous()
        try:
            return binding.small_m(x, self.wq, self.s, self.b, self.p.bits, self.p.group_size, out=out,
                                   out_dtype=out_dtype, variant=variant, splits=splits)
        except binding.QmmError as e:
            if allow_unsupported and e.status == 3:
                return None
            raise


def to_f64(y) -> np.ndarray:
    import torch

    return y.detach().to(torch.float64).cpu().numpy()


class OracleRef:
    """Oracle results for one problem (the oracle packs the codes itself)."""

    def __init__(self, p: synth.Problem):
        self.p = p
        self.lib = oracle.load()
        self.wq = self.lib.pack(p.q, p.bits)
        self._full = None

    def full(self, M: int = synth.MAX_ROWS):
        if self._full is None or self._full[0].shape[0] < M:
            self._full = self.lib.qmm(self.p.x_rows(M), self.wq, self.p.scales, self.p.biases, self.p.bits,
                                      self.p.group_size)
        y, a = self._full
        return y[:M], a[:M]

    def sampled(self, M: int, ms, ns):
        return self.lib.qmm_sampled(self.p.x_rows(M), self.wq, self.p.scales, self.p.biases, self.p.bits,
                                    self.p.group_size, ms, ns)


def bf16_half_ulp(y) -> np.ndarray:
    """Half a bf16 ulp at each value of ``y`` (values that are bf16 numbers):
    2^(e-8) for |y| in [2^e, 2^(e+1)), i.e. the most that one round to nearest
    even into bf16 moves a real number that rounds to y.  0 at y = 0."""
    y = np.abs(np.asarray(y, dtype=np.float64))
    _, ex = np.frexp(y)  # y = f * 2^ex, f in [0.5, 1)
    return np.where(y > 0, np.ldexp(1.0, ex - 9), 0.0)


def assert_within(y, y_ref, a_ref, what: str, bf16: bool = False):
    """|y - y_ref| <= 2e-3 * a_ref + 1e-5 per output.  With ``bf16`` the
    outputs were stored as bf16: the bound applies to the fp32 result, and the
    one rounding of the store adds at most half a bf16 ulp of the output."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = REL_TOL * a_ref + ABS_TOL
    if bf16:
        bound = bound + bf16_half_ulp(y)
    bad = ~(err <= bound)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; first at {idx}: "
                             f"gpu={y[idx]!r} ref={y_ref[idx]!r} bound={bound[idx]!r}; "
                             f"max err/bound={float((err / bound).max()):.3f}")
    return float((err / bound).max()) if err.size else 0.0


def check(y, y_ref, a_ref, what: str, at=None):
    """assert_within for a GPU output tensor (bf16 or fp32), optionally at
    sampled positions ``at`` = (rows, columns)."""
    import torch

    v = to_f64(y)
    if at is not None:
        v = v[at]
    return assert_within(v, y_ref, a_ref, what, bf16=y.dtype == torch.bfloat16)


def sample_positions(M: int, N: int, count: int, seed: int = 0):
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, size=count)
    ns = rng.integers(0, N, size=count)
    # always include the corners and the last row tile
    ms = np.concatenate([ms, [0, M - 1, 0, M - 1]])
    ns = np.concatenate([ns, [0, 0, N - 1, N - 1]])
    return ms, ns
