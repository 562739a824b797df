"""Python access to the fp64 CPU oracle in ``qmm_oracle.cpp``.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Nothing here imports the CUDA library
and the CUDA library never imports this module.

The oracle is built with the system C++ compiler as a plain shared object and
loaded with ctypes.  ``build()`` is idempotent; ``load()`` builds on demand.
``OracleLib`` can load any build of the source, which is how the mutation test
checks that the pins catch planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "qmm_oracle.cpp"
LIBRARY = HERE / "liboracle.so"
CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def compile_source(source: Path, output: Path, extra_flags=()) -> Path:
    """Compile one oracle source file to a shared object."""
    cmd = ["g++", *CXXFLAGS, *extra_flags, "-o", str(output), str(source)]
    subprocess.run(cmd, check=True)
    return output


def build(force: bool = False) -> Path:
    """Build liboracle.so next to its source unless it is up to date."""
    if force or not LIBRARY.exists() or LIBRARY.stat().st_mtime < SOURCE.stat().st_mtime:
        tmp = LIBRARY.with_name(f"liboracle.{os.getpid()}.tmp.so")
        compile_source(SOURCE, tmp)
        os.replace(tmp, LIBRARY)
    return LIBRARY


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


class OracleLib:
    """ctypes view of one build of the oracle."""

    def __init__(self, path: Path):
        self.path = Path(path)
        lib = ctypes.CDLL(str(self.path))
        i64, vp, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_pack.argtypes = [vp, i64, i64, c_int, vp]
        lib.oracle_unpack.argtypes = [vp, i64, i64, c_int, vp]
        lib.oracle_qmm.argtypes = [vp, vp, vp, vp, i64, i64, i64, c_int, i64, vp, vp]
        lib.oracle_qmm_sampled.argtypes = [vp, vp, vp, vp, i64, i64, i64, c_int, i64, vp, vp, i64, vp, vp]
        lib.oracle_dequant.argtypes = [vp, vp, vp, i64, i64, c_int, i64, vp]
        lib.oracle_qmm_residual.argtypes = [vp, vp, vp, vp, vp, c_int, i64, i64, i64, c_int, i64, vp, vp]
        lib.oracle_gather_qmm.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, i64, vp, vp]
        lib.oracle_ggml_dequant.argtypes = [c_int, vp, i64, i64, vp]
        lib.oracle_ggml_qmm.argtypes = [c_int, vp, vp, i64, i64, i64, vp, vp]
        lib.oracle_mx_dequant.argtypes = [c_int, vp, vp, i64, i64, vp]
        lib.oracle_mx_qmm.argtypes = [c_int, vp, vp, vp, i64, i64, i64, vp, vp]
        for name in ("oracle_fp4_e2m1", "oracle_fp8_e4m3", "oracle_e8m0"):
            getattr(lib, name).argtypes = [ctypes.c_uint]
            getattr(lib, name).restype = ctypes.c_double
        for name in ("oracle_pack", "oracle_unpack", "oracle_qmm", "oracle_qmm_sampled", "oracle_dequant",
                     "oracle_qmm_residual", "oracle_gather_qmm", "oracle_ggml_dequant", "oracle_ggml_qmm",
                     "oracle_mx_dequant", "oracle_mx_qmm"):
            getattr(lib, name).restype = c_int
        self.lib = lib

    # -- scalar decoders -------------------------------------------------
    def half_to_double(self, bits: int) -> float:
        return self.lib.oracle_half_to_double(int(bits) & 0xFFFF)

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits) & 0xFFFF)

    # -- packing ---------------------------------------------------------
    def pack(self, q: np.ndarray, bits: int) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.uint8)
        n, k = q.shape
        out = np.empty((n, k * bits // 32), dtype=np.uint32)
        rc = self.lib.oracle_pack(_ptr(q), n, k, bits, _ptr(out))
        if rc:
            raise OracleError(f"oracle_pack rc={rc}")
        return out

    def unpack(self, wq: np.ndarray, k: int, bits: int) -> np.ndarray:
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        n = wq.shape[0]
        out = np.empty((n, k), dtype=np.uint8)
        rc = self.lib.oracle_unpack(_ptr(wq), n, k, bits, _ptr(out))
        if rc:
            raise OracleError(f"oracle_unpack rc={rc}")
        return out

    # -- the product -----------------------------------------------------
    def qmm(self, x_bits, wq, s_bits, b_bits, bits: int, group_size: int):
        """Return (Y, A) in fp64; inputs are raw bf16/fp16 bit patterns (uint16)."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        m, k = x.shape
        n = wq.shape[0]
        y = np.empty((m, n), dtype=np.float64)
        a = np.empty((m, n), dtype=np.float64)
        rc = self.lib.oracle_qmm(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), m, n, k, bits, group_size, _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_qmm rc={rc}")
        return y, a

    def qmm_residual(self, x_bits, wq, s_bits, b_bits, r, bits: int, group_size: int):
        """Return (Y, A) of Y = R + X . W^T in fp64.  ``r``: [M, N] bf16 bit
        patterns (uint16) or float32 values."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        r = np.ascontiguousarray(r)
        if r.dtype not in (np.uint16, np.float32):
            raise OracleError("r must be uint16 (bf16 bits) or float32")
        m, k = x.shape
        n = wq.shape[0]
        if r.shape != (m, n):
            raise OracleError("r must be [M, N]")
        y = np.empty((m, n), dtype=np.float64)
        a = np.empty((m, n), dtype=np.float64)
        rc = self.lib.oracle_qmm_residual(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), _ptr(r), int(r.dtype == np.float32),
                                          m, n, k, bits, group_size, _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_qmm_residual rc={rc}")
        return y, a

    def gather_qmm(self, x_bits, wq, s_bits, b_bits, lhs, rhs, bits: int, group_size: int):
        """Return (Y, A) [P, N] of Y[i] = X[lhs[i]] . W[rhs[i]]^T in fp64.
        ``wq``: [E, N, K*bits/32]; ``s_bits``, ``b_bits``: [E, N, K/g]."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        lhs = np.ascontiguousarray(lhs, dtype=np.int32)
        rhs = np.ascontiguousarray(rhs, dtype=np.int32)
        t, k = x.shape
        e, n = wq.shape[0], wq.shape[1]
        p = len(lhs)
        y = np.empty((p, n), dtype=np.float64)
        a = np.empty((p, n), dtype=np.float64)
        rc = self.lib.oracle_gather_qmm(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), _ptr(lhs), _ptr(rhs), p, t, e, n, k,
                                        bits, group_size, _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_gather_qmm rc={rc}")
        return y, a

    GGML_TYPES = {"q4_0": (0, 18), "q4_1": (1, 20), "q8_0": (2, 34)}

    def ggml_dequant(self, kind: str, blocks, n: int, k: int) -> np.ndarray:
        """fp64 W[N, K] from ggml blocks (uint8, N * K/32 blocks, row-major)."""
        t, nbytes = self.GGML_TYPES[kind]
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        if blocks.size != n * (k // 32) * nbytes:
            raise OracleError("block buffer size does not match N, K")
        w = np.empty((n, k), dtype=np.float64)
        rc = self.lib.oracle_ggml_dequant(t, _ptr(blocks), n, k, _ptr(w))
        if rc:
            raise OracleError(f"oracle_ggml_dequant rc={rc}")
        return w

    def ggml_qmm(self, kind: str, x_bits, blocks, n: int):
        """(Y, A) of X . W^T for W [N, K] in ggml blocks."""
        t, nbytes = self.GGML_TYPES[kind]
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        m, k = x.shape
        if blocks.size != n * (k // 32) * nbytes:
            raise OracleError("block buffer size does not match N, K")
        y = np.empty((m, n), dtype=np.float64)
        a = np.empty((m, n), dtype=np.float64)
        rc = self.lib.oracle_ggml_qmm(t, _ptr(x), _ptr(blocks), m, n, k, _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_ggml_qmm rc={rc}")
        return y, a

    MX_FORMATS = {"mxfp4": (0, 4), "mxfp8": (1, 8), "nvfp4": (2, 4)}

    def mx_decoders(self):
        """The element and scale decoders: (fp4 e2m1, fp8 e4m3, e8m0) callables."""
        return self.lib.oracle_fp4_e2m1, self.lib.oracle_fp8_e4m3, self.lib.oracle_e8m0

    def mx_dequant(self, fmt: str, wq, s, k: int) -> np.ndarray:
        f, bits = self.MX_FORMATS[fmt]
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s, dtype=np.uint8)
        n = wq.shape[0]
        w = np.empty((n, k), dtype=np.float64)
        rc = self.lib.oracle_mx_dequant(f, _ptr(wq), _ptr(s), n, k, _ptr(w))
        if rc:
            raise OracleError(f"oracle_mx_dequant rc={rc}")
        return w

    def mx_qmm(self, fmt: str, x_bits, wq, s):
        f, bits = self.MX_FORMATS[fmt]
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s, dtype=np.uint8)
        m, k = x.shape
        n = wq.shape[0]
        y = np.empty((m, n), dtype=np.float64)
        a = np.empty((m, n), dtype=np.float64)
        rc = self.lib.oracle_mx_qmm(f, _ptr(x), _ptr(wq), _ptr(s), m, n, k, _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_mx_qmm rc={rc}")
        return y, a

    def qmm_sampled(self, x_bits, wq, s_bits, b_bits, bits: int, group_size: int, ms, ns):
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        m, k = x.shape
        n = wq.shape[0]
        y = np.empty(len(ms), dtype=np.float64)
        a = np.empty(len(ms), dtype=np.float64)
        rc = self.lib.oracle_qmm_sampled(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), m, n, k, bits, group_size,
                                         _ptr(ms), _ptr(ns), len(ms), _ptr(y), _ptr(a))
        if rc:
            raise OracleError(f"oracle_qmm_sampled rc={rc}")
        return y, a

    def dequant(self, wq, s_bits, b_bits, k: int, bits: int, group_size: int) -> np.ndarray:
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        n = wq.shape[0]
        w = np.empty((n, k), dtype=np.float64)
        rc = self.lib.oracle_dequant(_ptr(wq), _ptr(s), _ptr(b), n, k, bits, group_size, _ptr(w))
        if rc:
            raise OracleError(f"oracle_dequant rc={rc}")
        return w


_LOADED: OracleLib | None = None


def load() -> OracleLib:
    """Build (if needed) and load the oracle."""
    global _LOADED
    if _LOADED is None:
        _LOADED = OracleLib(build())
    return _LOADED
