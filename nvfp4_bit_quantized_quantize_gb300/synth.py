"""Seeded synthetic inputs for the NVFP4 linear-layer workloads.

This module only draws random tensors; it holds none of the quantization or
matmul arithmetic.  Both the CUDA path (tests, bench, smoke) and the CPU oracle
receive the same bf16 bytes from here, so the choice of generator cannot affect
parity.

Recipe: NumPy PCG64 seeded with ``seed * 16 + t`` for tensor ``t`` of a
workload; values ~ N(mean, std); an independent Bernoulli(p) mask picks
outliers, multiplied by ``outlier_scale``; the result is rounded to bf16
(round-to-nearest-even) and returned as uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round binary32 to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, seed: int, tensor: int = 0, std: float = 1.0, mean: float = 0.0,
                outlier_frac: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed * 16 + tensor))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < outlier_frac
        x[mask] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


@dataclass(frozen=True)
class Tensor:
    name: str
    rows: int
    cols: int
    std: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0

    def make(self, seed: int, index: int) -> np.ndarray:
        return normal_bf16((self.rows, self.cols), seed, index, self.std, 0.0,
                           self.outlier_frac, self.outlier_scale)


# The five workloads of the NVFP4 linear-layer path (shapes and value
# distributions as specified for this implementation).
WORKLOADS = {
    "tiny_linear_256": dict(seed=0, tensors=[
        Tensor("X", 256, 256, 1.0, 0.005, 50.0),
        Tensor("W", 256, 256, 1.0, 0.005, 50.0)]),
    "quantize_sweep": dict(seed=1, tensors=[
        Tensor("A1024", 1024, 1024, 1.0, 0.001, 100.0),
        Tensor("A4096", 4096, 4096, 1.0, 0.001, 100.0),
        Tensor("A8192", 8192, 8192, 1.0, 0.001, 100.0)]),
    "fprop_w2d_8192x20480x5120": dict(seed=2, tensors=[
        Tensor("W", 20480, 5120, 0.02),
        Tensor("X", 8192, 5120, 1.0, 0.001, 100.0)]),
    "wgrad_rht_sr_16384x5120": dict(seed=3, tensors=[
        Tensor("dY", 16384, 5120, 1e-3),
        Tensor("X", 16384, 5120, 1.0)]),
    "mlp7b_fwd_bwd_h4096_f11008_t8192": dict(seed=4, tensors=[
        Tensor("X", 8192, 4096, 1.0, 0.001, 100.0),
        Tensor("W_up", 11008, 4096, 0.02),
        Tensor("W_down", 4096, 11008, 0.02),
        Tensor("dY_down", 8192, 4096, 1e-3)]),
}


def make_workload(name: str, only=None) -> dict:
    w = WORKLOADS[name]
    out = {}
    for i, t in enumerate(w["tensors"]):
        if only is None or t.name in only:
            out[t.name] = t.make(w["seed"], i)
    return out
