"""Seeded synthetic inputs for the small-M affine-quantized matmul.

This module only draws random numbers and rounds them to their storage
formats (fp16 for scales and biases, bf16 for activations).  It holds none of
the method's arithmetic: it does not pack, dequantize or multiply.  Both the
CUDA path and the CPU oracle take their inputs from here and nowhere else.

Recipe (one numpy PCG64 stream per tensor, keyed by ``(seed, stream)``):

* codes ``q ~ Uniform{0 .. 2^bits - 1}``, uint8 ``[N, K]``;
* ``scale = fp16(0.002 * |N(0,1)| + 1e-4)`` per (row, group);
* ``bias  = fp16(-(2^bits - 1)/2 * scale)``, i.e. ``-7.5 * scale`` at 4 bits
  and ``-1.5 * scale`` at 2 bits (the scale is taken after its fp16 rounding);
* ``X = bf16(N(0,1))`` drawn for 16 rows; an M-row problem uses the first M
  rows, so every M of a sweep sees the same leading rows;
* a residual ``R = N(0,1)`` per output element, stored as bf16 bit patterns
  or as float32 (the output dtype it is added in);
* mixture-of-experts stacks: E matrices drawn as above (codes, scales and
  biases of the whole stack from one stream each), and a routing in which
  each of T tokens picks k distinct experts with probabilities
  ``softmax(1.5 * z)``, ``z ~ N(0,1)`` per expert (a few popular experts, so
  the tokens of a verify step share some of theirs).

Rounding to fp16 is numpy's (round to nearest even); rounding binary32 to
bf16 is round to nearest even on the bit pattern.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

MAX_ROWS = 16

STREAM_CODES = 0
STREAM_SCALES = 1
STREAM_X = 2
STREAM_RESIDUAL = 3
STREAM_ROUTING = 4
STREAM_GGML = 5
STREAM_MX = 6
GGML_BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34}


def rng_for(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to binary32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f64_to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


@dataclass
class Problem:
    """One weight matrix with its metadata and 16 rows of activations.

    ``q``: uint8 codes [N, K]; ``scales``/``biases``: fp16 bit patterns
    [N, K/group_size]; ``x``: bf16 bit patterns [16, K].
    """

    N: int
    K: int
    bits: int
    group_size: int
    q: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    x: np.ndarray
    seed: int

    def x_rows(self, M: int) -> np.ndarray:
        return np.ascontiguousarray(self.x[:M])


def make_codes(seed: int, N: int, K: int, bits: int) -> np.ndarray:
    return rng_for(seed, STREAM_CODES).integers(0, 1 << bits, size=(N, K), dtype=np.uint8)


def make_scales_biases(seed: int, N: int, groups: int, bits: int):
    z = rng_for(seed, STREAM_SCALES).standard_normal(size=(N, groups))
    scale_bits = f64_to_fp16_bits(0.002 * np.abs(z) + 1e-4)
    scale = scale_bits.view(np.float16).astype(np.float64)
    bias_bits = f64_to_fp16_bits(-((1 << bits) - 1) / 2.0 * scale)
    return scale_bits, bias_bits


def make_x(seed: int, K: int, rows: int = MAX_ROWS) -> np.ndarray:
    z = rng_for(seed, STREAM_X).standard_normal(size=(rows, K), dtype=np.float32)
    return f32_to_bf16_bits(z)


def make_residual(seed: int, M: int, N: int, f32: bool = False) -> np.ndarray:
    """R[M, N]: bf16 bit patterns (uint16), or float32 values if ``f32``."""
    z = rng_for(seed, STREAM_RESIDUAL).standard_normal(size=(M, N), dtype=np.float32)
    return z if f32 else f32_to_bf16_bits(z)


@dataclass
class MoeProblem:
    """A stack of E expert matrices and a routing of T tokens to k experts each.

    ``q``: uint8 [E, N, K]; ``scales``/``biases``: fp16 bits [E, N, K/g];
    ``x``: bf16 bits [16, K]; ``experts``: int32 [T, k] (distinct per token).
    The gathered list is entry i = t * k + j: lhs[i] = t, rhs[i] = experts[t, j].
    """

    E: int
    N: int
    K: int
    bits: int
    group_size: int
    q: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    x: np.ndarray
    experts: np.ndarray
    seed: int

    def lists(self):
        T, k = self.experts.shape
        lhs = np.repeat(np.arange(T, dtype=np.int32), k)
        return lhs, np.ascontiguousarray(self.experts.reshape(-1), dtype=np.int32)


def make_routing(seed: int, T: int, k: int, E: int) -> np.ndarray:
    rng = rng_for(seed, STREAM_ROUTING)
    z = rng.standard_normal(size=E)
    p = np.exp(1.5 * (z - z.max()))
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def make_moe(seed: int, E: int, N: int, K: int, bits: int, group_size: int, T: int, k: int) -> MoeProblem:
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    q = make_codes(seed, E * N, K, bits).reshape(E, N, K)
    scales, biases = make_scales_biases(seed, E * N, K // group_size, bits)
    return MoeProblem(E=E, N=N, K=K, bits=bits, group_size=group_size, q=q,
                      scales=scales.reshape(E, N, -1), biases=biases.reshape(E, N, -1), x=make_x(seed, K),
                      experts=make_routing(seed, T, k, E), seed=seed)


def make_ggml_blocks(seed: int, N: int, K: int, kind: str) -> np.ndarray:
    """Random ggml blocks (uint8 [N * K/32, bytes]) for a [N, K] matrix: the
    fp16 d (and Q4_1's m = fp16(-7.5 d)) drawn like the affine scales and
    biases, every code byte uniform.  Only random draws and fp16 rounding: the
    block layout (d first, little-endian) is the format's."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nblk = N * (K // 32)
    rng = rng_for(seed, STREAM_GGML)
    d_bits = f64_to_fp16_bits(0.002 * np.abs(rng.standard_normal(nblk)) + 1e-4)
    head = [d_bits.view(np.uint8).reshape(nblk, 2)]
    if kind == "q4_1":
        m_bits = f64_to_fp16_bits(-7.5 * d_bits.view(np.float16).astype(np.float64))
        head.append(m_bits.view(np.uint8).reshape(nblk, 2))
    nq = 32 if kind == "q8_0" else 16
    codes = rng.integers(0, 256, size=(nblk, nq), dtype=np.uint8)
    out = np.concatenate(head + [codes], axis=1)
    assert out.shape[1] == GGML_BLOCK_BYTES[kind]
    return np.ascontiguousarray(out)


def make_mx(seed: int, N: int, K: int, fmt: str):
    """Microscaled weights [N, K]: codes (uint8 [N, K]) uniform over the
    format's non-NaN codes (all 16 FP4 E2M1 codes; the 254 FP8 E4M3 codes other
    than 0x7F and 0xFF), and scale bytes: E8M0 (uint8 [N, K/32]) uniform in
    [127 - 12, 127], i.e. 2^-12 .. 1; for nvfp4, E4M3 (uint8 [N, K/16]) with a
    positive normal exponent field in 1..7 and any mantissa, i.e. 2^-6 .. 1.875."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    rng = rng_for(seed, STREAM_MX)
    if fmt in ("mxfp4", "nvfp4"):
        q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    else:
        q = rng.integers(0, 254, size=(N, K), dtype=np.uint8)
        q = np.where(q >= 0x7F, q + 1, q).astype(np.uint8)  # skip 0x7F; 0xFF is never drawn
    if fmt == "nvfp4":
        s = (rng.integers(1, 8, size=(N, K // 16)) << 3 | rng.integers(0, 8, size=(N, K // 16))).astype(np.uint8)
    else:
        s = rng.integers(127 - 12, 128, size=(N, K // 32), dtype=np.uint8)
    return q, s


def make_problem(seed: int, N: int, K: int, bits: int, group_size: int, rows: int = MAX_ROWS) -> Problem:
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    groups = K // group_size
    q = make_codes(seed, N, K, bits)
    scales, biases = make_scales_biases(seed, N, groups, bits)
    x = make_x(seed, K, rows)
    return Problem(N=N, K=K, bits=bits, group_size=group_size, q=q, scales=scales, biases=biases, x=x, seed=seed)
