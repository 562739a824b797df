"""ctypes binding of libqmm (C ABI in ``include/qmm.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libqmm.so``.  PyTorch supplies device memory and the current
stream.  If the library has not been built, the first call raises
``RuntimeError``; there is no fallback.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

LIBRARY = Path(__file__).resolve().parent / "libqmm.so"

STATUS = {
    0: "QMM_OK",
    1: "QMM_ERR_NULL",
    2: "QMM_ERR_SHAPE",
    3: "QMM_ERR_UNSUPPORTED",
    4: "QMM_ERR_ALIGN",
    5: "QMM_ERR_CUDA",
    6: "QMM_ERR_TABLE",
}
OUT_BF16 = 0
OUT_F32 = 1

# Every function the header declares, with its ctypes signature.
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
SIGNATURES = {
    "qmm_small_m": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "qmm_small_m_ex": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _i32, _i32, _i32, _vp]),
    "qmm_small_m_residual": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _i32, _i32, _i32,
                                    _vp]),
    "qmm_gather_small_m": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp,
                                  _i32, _i32, _i32, _vp]),
    "qmm_from_ggml": (_i32, [_i32, _vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    "qmm_small_m_mx": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _i32, _i32, _vp]),
    "qmm_packed_words": (ctypes.c_size_t, [_i64, _i64, _i32]),
    "qmm_pack": (_i32, [_vp, _i64, _i64, _i32, _vp]),
    "qmm_unpack": (_i32, [_vp, _i64, _i64, _i32, _vp]),
    "qmm_repack": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp]),
    "qmm_unrepack": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp]),
    "qmm_select_variant": (_i32, [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32)]),
    "qmm_num_variants": (_i32, []),
    "qmm_variant_name": (ctypes.c_char_p, [_i32]),
    "qmm_status_string": (ctypes.c_char_p, [_i32]),
    "qmm_last_cuda_error": (_i32, []),
    "qmm_device_status": (ctypes.c_uint, [_i32]),
    "qmm_version": (ctypes.c_char_p, []),
}


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {name}{(' (' + detail + ')') if detail else ''}")


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not LIBRARY.exists():
            raise RuntimeError(f"{LIBRARY.name} is not built; run __graft_entry__.build() "
                               "or quantized_matmul_speculative_gb300/build.py")
        handle = ctypes.CDLL(str(LIBRARY))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(rc: int, where: str):
    if rc != 0:
        detail = ""
        if rc == 5:
            detail = f"cudaError {lib().qmm_last_cuda_error()}"
        raise QmmError(rc, where, detail)


# ---------------------------------------------------------------- host helpers
def packed_words(N: int, K: int, bits: int) -> int:
    return int(lib().qmm_packed_words(N, K, bits))


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack uint8 codes [N, K] into uint32 words [N, K*bits/32] (host)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    out = np.empty((N, K * bits // 32), dtype=np.uint32)
    _check(lib().qmm_pack(q.ctypes.data, N, K, bits, out.ctypes.data), "qmm_pack")
    return out


def unpack(wq: np.ndarray, K: int, bits: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    N = wq.shape[0]
    out = np.empty((N, K), dtype=np.uint8)
    _check(lib().qmm_unpack(wq.ctypes.data, N, K, bits, out.ctypes.data), "qmm_unpack")
    return out


def repack(wq, bits: int, out=None, inverse: bool = False, stream=None):
    """Canonical -> native packed layout on the device (inverse: native ->
    canonical).  ``wq``: CUDA int32/uint32 [N, K*bits/32]."""
    import torch

    if not wq.is_cuda or not wq.is_contiguous():
        raise ValueError("wq must be a contiguous CUDA tensor")
    N, words = wq.shape
    K = words * 32 // bits
    if out is None:
        out = torch.empty_like(wq)
    if stream is None:
        stream = torch.cuda.current_stream(wq.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    fn = lib().qmm_unrepack if inverse else lib().qmm_repack
    _check(fn(wq.data_ptr(), N, K, bits, out.data_ptr(), handle), "qmm_unrepack" if inverse else "qmm_repack")
    return out


GGML_TYPES = {"q4_0": (0, 18, 4), "q4_1": (1, 20, 4), "q8_0": (2, 34, 8)}
MX_FORMATS = {"mxfp4": (0, 4, 32), "mxfp8": (1, 8, 32), "nvfp4": (2, 4, 16)}


def small_m_mx(x, wq, scales, fmt: str, out=None, out_dtype=None, variant: int = -1, splits: int = -1,
               stream=None):
    """Y = X . W^T for microscaled W: ``wq`` int32 [N, K*bits/32] (E2M1 or
    E4M3 codes), ``scales`` uint8 [N, K/32] (E8M0) or [N, K/16] (nvfp4: E4M3);
    CUDA tensors."""
    import torch

    f, bits, g = MX_FORMATS[fmt]
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    M, K = x.shape
    N = wq.shape[0]
    if wq.shape[1] * 32 != K * bits or tuple(scales.shape) != (N, K // g) or scales.dtype != torch.uint8:
        raise ValueError("wq / scales do not match K and the format")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib().qmm_small_m_mx(x.data_ptr(), wq.data_ptr(), scales.data_ptr(), M, N, K, f, out.data_ptr(),
                                OUT_F32 if out_dtype == torch.float32 else OUT_BF16, variant, splits, handle),
           "qmm_small_m_mx")
    return out


def from_ggml(kind: str, blocks, N: int, K: int, stream=None):
    """ggml blocks (CUDA uint8 tensor of N*K/32 blocks) -> (wq, scales, biases)
    in the affine layout with group size 32; returns the code width too."""
    import torch

    t, nbytes, bits = GGML_TYPES[kind]
    if not blocks.is_cuda or not blocks.is_contiguous() or blocks.numel() != N * (K // 32) * nbytes:
        raise ValueError("blocks must be a contiguous CUDA buffer of N*K/32 blocks")
    dev = blocks.device
    wq = torch.empty((N, K * bits // 32), dtype=torch.int32, device=dev)
    s = torch.empty((N, K // 32), dtype=torch.float16, device=dev)
    b = torch.empty((N, K // 32), dtype=torch.float16, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib().qmm_from_ggml(t, blocks.data_ptr(), N, K, wq.data_ptr(), s.data_ptr(), b.data_ptr(), handle),
           "qmm_from_ggml")
    return wq, s, b, bits


def select_variant(M: int, N: int, K: int, bits: int, group_size: int):
    s = ctypes.c_int(0)
    v = lib().qmm_select_variant(M, N, K, bits, group_size, ctypes.byref(s))
    return (v, s.value) if v >= 0 else (None, None)


def device_status(clear: bool = True) -> int:
    """OR of the kernels' device status words (0 = no bounded wait gave up)."""
    return int(lib().qmm_device_status(1 if clear else 0))


def variant_names():
    L = lib()
    return [L.qmm_variant_name(i).decode() for i in range(L.qmm_num_variants())]


# ---------------------------------------------------------------- device call
def small_m_ptr(x_ptr: int, wq_ptr: int, s_ptr: int, b_ptr: int, M: int, N: int, K: int, bits: int,
                group_size: int, y_ptr: int, out_dtype: int = OUT_BF16, variant: int = -1, splits: int = -1,
                stream: int = 0) -> None:
    """Raw-pointer call of qmm_small_m_ex (device pointers, cudaStream_t as int)."""
    rc = lib().qmm_small_m_ex(x_ptr, wq_ptr, s_ptr, b_ptr, M, N, K, bits, group_size, y_ptr,
                              out_dtype, variant, splits, stream)
    _check(rc, "qmm_small_m_ex")


def small_m_residual_ptr(x_ptr: int, wq_ptr: int, s_ptr: int, b_ptr: int, r_ptr: int, M: int, N: int, K: int,
                         bits: int, group_size: int, y_ptr: int, out_dtype: int = OUT_BF16, variant: int = -1,
                         splits: int = -1, stream: int = 0) -> None:
    """Raw-pointer call of qmm_small_m_residual: Y = R + X . dequant(W)^T."""
    rc = lib().qmm_small_m_residual(x_ptr, wq_ptr, s_ptr, b_ptr, r_ptr, M, N, K, bits, group_size, y_ptr,
                                    out_dtype, variant, splits, stream)
    _check(rc, "qmm_small_m_residual")


def gather_small_m_ptr(x_ptr: int, wq_ptr: int, s_ptr: int, b_ptr: int, lhs_ptr: int, rhs_ptr: int, P: int, T: int,
                       E: int, N: int, K: int, bits: int, group_size: int, y_ptr: int, out_dtype: int = OUT_BF16,
                       variant: int = -1, splits: int = -1, stream: int = 0) -> None:
    """Raw-pointer call of qmm_gather_small_m: Y[i] = X[lhs[i]] . W[rhs[i]]^T."""
    rc = lib().qmm_gather_small_m(x_ptr, wq_ptr, s_ptr, b_ptr, lhs_ptr, rhs_ptr, P, T, E, N, K, bits, group_size,
                                  y_ptr, out_dtype, variant, splits, stream)
    _check(rc, "qmm_gather_small_m")


def gather_small_m(x, wq, scales, biases, lhs, rhs, bits: int, group_size: int, out=None, out_dtype=None,
                   variant: int = -1, splits: int = -1, stream=None):
    """Y[i] = X[lhs[i]] . dequant(W[rhs[i]])^T over an expert stack.

    ``x``: bf16 [T, K]; ``wq``: int32 [E, N, K*bits/32]; ``scales``, ``biases``:
    fp16 [E, N, K/group_size]; ``lhs``, ``rhs``: int32 [P]; all contiguous CUDA
    tensors.  Returns ``out`` [P, N] (bf16 or fp32).
    """
    import torch

    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    for name, t in (("x", x), ("wq", wq), ("scales", scales), ("biases", biases), ("lhs", lhs), ("rhs", rhs)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if lhs.dtype != torch.int32 or rhs.dtype != torch.int32 or lhs.shape != rhs.shape or lhs.dim() != 1:
        raise TypeError("lhs and rhs must be int32 vectors of one length")
    T, K = x.shape
    E, N = wq.shape[0], wq.shape[1]
    if wq.shape[2] * 32 != K * bits or tuple(scales.shape) != (E, N, K // group_size):
        raise ValueError("wq / scales shapes do not match K, bits and group_size")
    P = lhs.shape[0]
    if out is None:
        out = torch.empty((P, N), dtype=out_dtype, device=x.device)
    elif tuple(out.shape) != (P, N) or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [P, N] tensor of out_dtype")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    gather_small_m_ptr(x.data_ptr(), wq.data_ptr(), scales.data_ptr(), biases.data_ptr(), lhs.data_ptr(),
                       rhs.data_ptr(), P, T, E, N, K, bits, group_size, out.data_ptr(),
                       OUT_F32 if out_dtype == torch.float32 else OUT_BF16, variant, splits, handle)
    return out


def small_m(x, wq, scales, biases, bits: int, group_size: int, out=None, out_dtype=None,
            variant: int = -1, splits: int = -1, stream=None, residual=None):
    """Y = X . dequant(Wq, scales, biases)^T on the GPU (+ ``residual``).

    ``x``: bf16 [M, K]; ``wq``: int32/uint32 [N, K*bits/32]; ``scales``,
    ``biases``: fp16 [N, K/group_size]; all CUDA tensors, contiguous.  Returns
    ``out`` (bf16 or fp32 [M, N]), allocated by torch if not given.  With
    ``residual`` (a contiguous [M, N] tensor of the output dtype, which may be
    ``out`` itself) the kernels store residual + product.
    """
    import torch

    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if x.dtype != torch.bfloat16 or scales.dtype != torch.float16 or biases.dtype != torch.float16:
        raise TypeError("x must be bfloat16, scales and biases float16")
    if wq.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32)):
        raise TypeError("wq must hold 32-bit words (int32 or uint32)")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out dtype must be bfloat16 or float32")
    for name, t in (("x", x), ("wq", wq), ("scales", scales), ("biases", biases)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    M, K = x.shape
    N = wq.shape[0]
    if wq.shape[1] * 32 != K * bits:
        raise ValueError("wq shape does not match K and bits")
    if tuple(scales.shape) != (N, K // group_size) or tuple(biases.shape) != (N, K // group_size):
        raise ValueError("scales/biases must be [N, K/group_size]")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    elif tuple(out.shape) != (M, N) or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    od = OUT_F32 if out_dtype == torch.float32 else OUT_BF16
    if residual is None:
        small_m_ptr(x.data_ptr(), wq.data_ptr(), scales.data_ptr(), biases.data_ptr(), M, N, K, bits, group_size,
                    out.data_ptr(), od, variant, splits, handle)
        return out
    if (not residual.is_cuda or not residual.is_contiguous() or tuple(residual.shape) != (M, N)
            or residual.dtype != out_dtype):
        raise ValueError("residual must be a contiguous CUDA [M, N] tensor of the output dtype")
    small_m_residual_ptr(x.data_ptr(), wq.data_ptr(), scales.data_ptr(), biases.data_ptr(), residual.data_ptr(),
                         M, N, K, bits, group_size, out.data_ptr(), od, variant, splits, handle)
    return out
