"""Named synthetic workloads and their algorithmic byte counts.

Every workload is a set of (N, K) weight shapes, a bit width, a group size and
the activation row counts M it is run at.  Shapes stand in for the model
layers the pages benchmark on; no model weights are involved.

Algorithmic bytes of one call (moved once, whatever M is):

    weight bytes   W_B    = N * K * bits / 8
    metadata bytes Meta_B = N * (K / g) * 4      (fp16 scale + fp16 bias)

The "total" count adds the activations (2*M*K) and the output (2 or 4 * M*N).
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Shape:
    name: str
    N: int
    K: int


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple
    bits: int
    group_size: int
    ms: tuple
    seed_base: int
    layers: int = 1
    note: str = ""
    variants: tuple = field(default_factory=tuple)  # extra (bits, group_size) pairs run on the same shapes


def weight_bytes(N: int, K: int, bits: int) -> int:
    return N * K * bits // 8


def meta_bytes(N: int, K: int, group_size: int) -> int:
    return N * (K // group_size) * 4


def call_bytes(N: int, K: int, bits: int, group_size: int) -> int:
    """Weight + metadata bytes one call has to stream (the roofline numerator)."""
    return weight_bytes(N, K, bits) + meta_bytes(N, K, group_size)


def total_bytes(M: int, N: int, K: int, bits: int, group_size: int, out_bytes: int = 2) -> int:
    return call_bytes(N, K, bits, group_size) + 2 * M * K + out_bytes * M * N


SINGLE_LAYER = Workload(
    name="single_layer_1024x1024_4b_g64",
    shapes=(Shape("layer", 1024, 1024),),
    bits=4, group_size=64, ms=(4,), seed_base=1000,
    note="one 1024x1024 layer at M=4; small enough for the full oracle in seconds",
)

M_SWEEP = Workload(
    name="m_sweep_5120x5120_4b_g64",
    shapes=(Shape("square", 5120, 5120),),
    bits=4, group_size=64, ms=tuple(range(1, 17)), seed_base=2000,
    note="M = 1..16 on one 5120x5120 layer",
)

DENSE_27B_LAYER = Workload(
    name="dense27b_layer_4b_g64",
    shapes=(Shape("qkv", 7168, 5120), Shape("o", 5120, 5120),
            Shape("gate_up", 34816, 5120), Shape("down", 5120, 17408)),
    bits=4, group_size=64, ms=(1, 2, 3, 4, 5, 8), seed_base=3000,
    note="projections of a 27B-class dense decoder layer",
)

GROUP_BIT_SWEEP = Workload(
    name="group_bit_sweep_8192x8192",
    shapes=(Shape("square", 8192, 8192),),
    bits=4, group_size=64, ms=tuple(range(1, 17)), seed_base=4000,
    variants=((4, 32), (4, 64), (4, 128), (2, 64)),
    note="4-bit at g32/g64/g128 and 2-bit at g64 on one 8192x8192 layer",
)

VERIFY_STEP = Workload(
    name="verify_step_36x4096_4b_g64",
    shapes=(Shape("qkv", 6144, 4096), Shape("o", 4096, 4096),
            Shape("gate_up", 24576, 4096), Shape("down", 4096, 12288)),
    bits=4, group_size=64, ms=tuple(range(1, 9)), seed_base=5000, layers=36,
    note="36 layers x 4 projections of a 4096-hidden dense stack, back to back on one stream",
)

INT8_AFFINE = Workload(
    name="int8_affine_8b_g64",
    shapes=(Shape("square", 5120, 5120), Shape("gate_up", 15360, 3840)),
    bits=8, group_size=64, ms=tuple(range(1, 17)), seed_base=6000,
    note="8-bit affine g64: the 5120x5120 layer and a 15360x3840 gate/up projection (the shape of the "
         "pages' int8 qmv_wide measurement; 60 groups per row, so its scale rows are not 16-byte strided)",
)

QMV_WIDE_GATE_UP = Workload(
    name="qmv_wide_gate_up_15360x3840_4b_g64",
    shapes=(Shape("gate_up", 15360, 3840),),
    bits=4, group_size=64, ms=tuple(range(1, 17)), seed_base=8000,
    note="the 15360x3840 gate/up projection of the pages' int4 qmv_wide measurement, 4-bit g64, M = 1..16 "
         "(60 groups per row: scale rows not 16-byte strided)",
)

ALL = (SINGLE_LAYER, M_SWEEP, DENSE_27B_LAYER, GROUP_BIT_SWEEP, VERIFY_STEP, INT8_AFFINE, QMV_WIDE_GATE_UP)


@dataclass(frozen=True)
class MoeWorkload:
    """A stack of E expert matrices [N, K] and T tokens routed to k experts each."""

    name: str
    E: int
    N: int
    K: int
    k: int
    bits: int
    group_size: int
    ts: tuple
    seed: int
    note: str = ""


MOE_GATE_UP = MoeWorkload(
    name="moe_gate_up_128x1536x2048_top8_4b_g64",
    E=128, N=1536, K=2048, k=8, bits=4, group_size=64, ts=(1, 2, 4, 8), seed=7000,
    note="gate+up projections of a 128-expert, top-8 MoE layer (2048 hidden, 768 expert width), T verify tokens",
)


def moe_union_bytes(w: MoeWorkload, experts) -> int:
    """Weight + metadata bytes of the distinct experts a routing names."""
    import numpy as np

    return len(np.unique(np.asarray(experts))) * call_bytes(w.N, w.K, w.bits, w.group_size)
BY_NAME = {w.name: w for w in ALL}


def shape_seed(workload: Workload, shape_index: int, layer: int = 0, bits: int | None = None,
               group_size: int | None = None) -> int:
    """Seed of one weight matrix: base + shape index + 4*layer, plus 100 per
    (bits, group) variant index."""
    seed = workload.seed_base + shape_index + 4 * layer
    if bits is not None and group_size is not None and workload.variants:
        seed += 100 * workload.variants.index((bits, group_size))
    return seed
