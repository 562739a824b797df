"""Small-M affine-quantized matmul for speculative-decoding verify, on GB300 (sm_103a).

``Y[M,N] = X[M,K] . dequant(Wq, scales, biases)[N,K]^T`` for M = 1..16, with
4- or 2-bit codes packed low-bits-first into uint32 words, one fp16 scale and
one fp16 bias per group of K, bf16 activations, fp32 accumulation and bf16 or
fp32 output.  All compute runs in the CUDA library ``libqmm.so`` (C ABI in
``include/qmm.h``); :mod:`.binding` is a thin ctypes layer over it.

Importing this package does not load the CUDA library; the first call through
:mod:`.binding` does, and fails loudly if it is missing.
"""

__all__ = ["binding", "synth", "workloads"]
