"""Seeded synthetic inputs for the affinity calibration pass.

This module only draws random tensors; it holds none of the method's
arithmetic.  Both the fp64 oracle (through the tests and the bench) and the
CUDA path consume what it returns, so the two always see identical values.

The calibration set of "Affinity-Aware Sharding for Delayed Tensor
Parallelism" (§3, "Affinity scores": 64 sequences x 1024 tokens of web text,
one forward pass of a trained Qwen3-0.6B / Danube3-500M) is not available, so
seeded Gaussian / Student-t tensors of the same shapes stand in for it.

Tensor layout (PyTorch ``nn.Linear`` storage, out x in):
  a   [T, H*dh]   attention head outputs, head h = columns h*dh .. h*dh+dh-1
  x   [T, D]      residual entering the FFN pre-norm
  Wo  [D, H*dh]   attention output projection
  gamma [D]       FFN pre-norm gain
  Wg, Wu [I, D]   gate / up projections (row k = w^g_k, w^u_k)
  Wd  [D, I]      down projection (column k = w^d_k)
  gamma_next [D], Wq_next [H*dh, D], Wk_next / Wv_next [G*dh, D]
                  the next layer's attention pre-norm gain and projections
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import numpy as np

__all__ = ["LayerShape", "CONFIGS", "make_layer", "bf16_round", "bf16_bits"]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    D: int
    H: int
    G: int
    dh: int
    I: int
    dtype: str            # "bf16" or "fp32" operand storage
    w_std: float          # weight std (N(0, w_std))
    x_dist: str           # "normal", "normal_outliers" or "student_t4"
    seed: int
    eps: float = 1e-6

    def scaled(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 layer, a Qwen3-0.6B-shaped layer, a
# Danube3-500M-shaped layer, the 28-layer Qwen3 stack (per-layer seeds
# 3000 + i, see ``stack_layer``) and a Llama-3-8B-shaped stress layer.
CONFIGS: Dict[str, LayerShape] = {
    "tiny": LayerShape("tiny", 256, 64, 4, 2, 16, 128, "fp32", 0.05, "normal", 0),
    "qwen3_0p6b_layer": LayerShape("qwen3_0p6b_layer", 65536, 1024, 16, 8, 128, 3072,
                                   "bf16", 0.02, "normal_outliers", 1),
    "danube3_500m_layer": LayerShape("danube3_500m_layer", 65536, 1536, 16, 8, 96, 4096,
                                     "bf16", 0.02, "normal_outliers", 2),
    "qwen3_0p6b_stack": LayerShape("qwen3_0p6b_stack", 65536, 1024, 16, 8, 128, 3072,
                                   "bf16", 0.02, "normal_outliers", 3),
    "llama3_8b_layer": LayerShape("llama3_8b_layer", 65536, 4096, 32, 8, 128, 14336,
                                  "bf16", 0.02, "student_t4", 4),
}
STACK_LAYERS = 28


def stack_layer(i: int) -> LayerShape:
    """Layer i of the 28-layer Qwen3-shaped stack: same shape, seed 3000 + i."""
    return CONFIGS["qwen3_0p6b_stack"].scaled(name=f"qwen3_0p6b_stack_l{i}", seed=3000 + i)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even);
    return the 16-bit patterns as uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    # NaN stays NaN (never produced by these generators, kept for safety)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 array holding the bfloat16-rounded values of x."""
    return (bf16_bits(x).astype(np.uint32) << 16).view(np.float32)


def _x(rng: np.random.Generator, shape: LayerShape) -> np.ndarray:
    T, D = shape.T, shape.D
    if shape.x_dist == "student_t4":
        return rng.standard_t(4, size=(T, D)).astype(np.float32)
    x = rng.standard_normal((T, D), dtype=np.float32)
    if shape.x_dist == "normal_outliers":
        # four fixed outlier channels scaled by 20
        for c in (0, D // 4, D // 2, 3 * D // 4):
            x[:, c] *= 20.0
    return x


def make_layer(shape: LayerShape, with_next: bool = False) -> Dict[str, np.ndarray]:
    """Draw one layer's inputs.

    Draw order is fixed (a, x, Wo, gamma, Wg, Wu, Wd, then gamma_next,
    Wq_next, Wk_next, Wv_next) from numpy's PCG64 seeded with shape.seed.
    For "bf16" shapes every tensor is rounded to bfloat16 and returned as
    float32 holding the rounded values; ``<name>_bits`` carries the uint16
    patterns to copy to the device.
    """
    rng = np.random.Generator(np.random.PCG64(shape.seed))
    s = shape
    T = s.T
    t: Dict[str, np.ndarray] = {}
    t["a"] = rng.standard_normal((T, s.H * s.dh), dtype=np.float32)
    t["x"] = _x(rng, s)
    w = np.float32(s.w_std)
    t["Wo"] = rng.standard_normal((s.D, s.H * s.dh), dtype=np.float32) * w
    t["gamma"] = (1.0 + 0.1 * rng.standard_normal(s.D, dtype=np.float32)).astype(np.float32)
    t["Wg"] = rng.standard_normal((s.I, s.D), dtype=np.float32) * w
    t["Wu"] = rng.standard_normal((s.I, s.D), dtype=np.float32) * w
    t["Wd"] = rng.standard_normal((s.D, s.I), dtype=np.float32) * w
    if with_next:
        t["gamma_next"] = (1.0 + 0.1 * rng.standard_normal(s.D, dtype=np.float32)).astype(np.float32)
        t["Wq_next"] = rng.standard_normal((s.H * s.dh, s.D), dtype=np.float32) * w
        t["Wk_next"] = rng.standard_normal((s.G * s.dh, s.D), dtype=np.float32) * w
        t["Wv_next"] = rng.standard_normal((s.G * s.dh, s.D), dtype=np.float32) * w
    if s.dtype == "bf16":
        for k in list(t):
            bits = bf16_bits(t[k])
            t[k + "_bits"] = bits
            t[k] = (bits.astype(np.uint32) << 16).view(np.float32)
    return t


def random_small_shape(rng: np.random.Generator, **over) -> LayerShape:
    """A small random-but-valid bf16 layer shape for parity sweeps."""
    G = int(rng.choice([1, 2, 4]))
    H = G * int(rng.choice([1, 2, 3]))
    base = dict(name="rand", T=int(rng.integers(1, 700)), D=int(8 * rng.integers(8, 40)),
                H=H, G=G, dh=int(8 * rng.integers(1, 17)), I=int(8 * rng.integers(4, 60)),
                dtype="bf16", w_std=0.05, x_dist="normal_outliers", seed=int(rng.integers(1 << 30)))
    base.update(over)
    return LayerShape(**base)
