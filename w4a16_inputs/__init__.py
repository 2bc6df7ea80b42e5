"""Seeded synthetic inputs for the fp16 x int4 group-quantized GEMM.

This module is shared by the tests, the oracle checks and the benchmark. It only
draws random numbers in the shapes and distributions of the workloads described
for the MatMulNBits int4 GEMM (github.com/justinchuby/onnx-genai pull 960,
"Validation": M in {1,2,7,16,33,64}, group in {16,32,64,128}, fp16/fp32 scales,
symmetric and asymmetric zero points; K=5120, N=13824, block 128 timings). It
holds none of the method's arithmetic: the packed weight bytes are drawn as
uniform bytes (two independent uniform nibbles each), the packed zero points
likewise, so no packing or dequantisation happens here.

Distributions:
  A       float32 N(0, 1) rounded to float16, shape [M, K]
  Bq      uint8 uniform 0..255, shape [N, K/2]   (nibbles uniform 0..15)
  scales  float32 uniform [0.005, 0.02], shape [N, K/group], stored as float16
          or float32
  zp      uint8 uniform 0..255, shape [N, ceil(G/2)]  (None when symmetric)
  gamma   float32 uniform [0.5, 1.5] rounded to float16, shape [K] (RMS-norm
          weight; the pages give no distribution)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

SCALE_LO = 0.005
SCALE_HI = 0.02


@dataclasses.dataclass
class W4A16Case:
    """One synthetic problem. Arrays are host numpy arrays."""

    M: int
    N: int
    K: int
    group: int
    A: np.ndarray            # float16 [M, K]
    bq: np.ndarray           # uint8 [N, K//2]
    scales: np.ndarray       # float16 or float32 [N, K//group]
    zp: Optional[np.ndarray]  # uint8 [N, ceil(G/2)] or None (symmetric)

    @property
    def G(self) -> int:
        return self.K // self.group

    @property
    def scale_f32(self) -> bool:
        return self.scales.dtype == np.float32


def draw_activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    return rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)


def draw_weights(rng: np.random.Generator, N: int, K: int, group: int,
                 scale_dtype=np.float16, asym: bool = True):
    """Packed int4 bytes, per-group scales and (optionally) packed zero points."""
    if K % 2 or K % group:
        raise ValueError("K must be even and a multiple of group")
    G = K // group
    bq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.uniform(SCALE_LO, SCALE_HI, size=(N, G)).astype(np.float32)
    scales = scales.astype(scale_dtype)
    zp = rng.integers(0, 256, size=(N, (G + 1) // 2), dtype=np.uint8) if asym else None
    return bq, scales, zp


def draw_norm_weight(rng: np.random.Generator, K: int) -> np.ndarray:
    """RMS-norm weight gamma [K]: float32 uniform [0.5, 1.5] rounded to float16."""
    return rng.uniform(0.5, 1.5, size=K).astype(np.float32).astype(np.float16)


def make_case(M: int, N: int, K: int, group: int, *, seed: int,
              scale_dtype=np.float16, asym: bool = True) -> W4A16Case:
    """Draw weights first (so that cases with the same seed and weight shape share
    weights across M), then activations."""
    rng = np.random.default_rng(seed)
    bq, scales, zp = draw_weights(rng, N, K, group, scale_dtype, asym)
    A = draw_activations(rng, M, K)
    return W4A16Case(M, N, K, group, A, bq, scales, zp)


def make_swiglu_case(M: int, N: int, K: int, group: int, *, seed: int,
                     scale_dtype=np.float16, asym: bool = True):
    """Gate and up weight sets plus shared activations."""
    rng = np.random.default_rng(seed)
    gate = draw_weights(rng, N, K, group, scale_dtype, asym)
    up = draw_weights(rng, N, K, group, scale_dtype, asym)
    A = draw_activations(rng, M, K)
    return (W4A16Case(M, N, K, group, A, *gate), W4A16Case(M, N, K, group, A, *up))


# The five workload families, each with the seed it is drawn with.
WORKLOADS = {
    "tiny": dict(M=2, K=256, N=256, group=32, asym=False, scale_dtype=np.float16, seed=0),
    "decode": dict(Ms=(1, 2, 4, 8), K=4096, N=4096, group=128, asym=True,
                   scale_dtype=np.float16, seed=1),
    "mlp": dict(Ms=(1, 2, 4, 8, 16, 32, 64, 128), K=5120, N=13824, group=128, asym=True,
                scale_dtype=np.float16, seed=2),
    "format": dict(Ms=(1, 2, 7, 16, 33, 64), K=5120, N=5120, groups=(16, 32, 64, 128),
                   scale_dtypes=(np.float16, np.float32), asyms=(False, True), seed=3),
    "gate_up": dict(Ms=(256, 1024, 4096, 8192), K=5120, N=13824, group=128, asym=True,
                    scale_dtype=np.float16, seed=4),
}
