"""Seeded synthetic inputs for the small-M NVFP4 W4A4 decode linear.

This module holds shapes and random draws only -- none of the method's
arithmetic (no scales, no quantisation).  Both the CUDA path's tests and
benchmark and the CPU oracle consume the same arrays from here.

Workloads stand in for the decode layers of the models the ReSET README lists
under "Supported models" (Qwen3 8B / 32B): the pages run real checkpoints,
which are not available here, so weights are Gaussian and activations are
Gaussian with a few large "outlier" channels, all seeded.

Recipe (every draw is ``numpy.random.default_rng(seed)``, PCG64, drawn
directly in float32 with ``standard_normal(dtype=float32)``):

* weights   W[n, k] = std * N(0, 1); std 0.02 (8B shapes) or 0.015 (32B shapes)
* activations X[m, k] = N(0, 1); then ``round(0.005 * k)`` channels, chosen by a
  seeded permutation shared by every row of the layer, are multiplied by 20.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Linear:
    name: str
    n: int  # output features (rows of W)
    k: int  # input features (reduction dim)


# One decoder layer of an 8B-shaped model (hidden 4096, MLP 12288).
LINEARS_8B = (
    Linear("qkv", 6144, 4096),
    Linear("o", 4096, 4096),
    Linear("gate_up", 24576, 4096),
    Linear("down", 4096, 12288),
)

# One decoder layer of a 32B-shaped model (hidden 5120, attn 8192, MLP 25600).
LINEARS_32B = (
    Linear("qkv", 10240, 5120),
    Linear("o", 5120, 8192),
    Linear("gate_up", 51200, 5120),
    Linear("down", 5120, 25600),
)

# The single small GEMV: M=1, K=512, N=256.
TINY = Linear("tiny", 256, 512)

WEIGHT_STD_8B = 0.02
WEIGHT_STD_32B = 0.015
OUTLIER_FRACTION = 0.005
OUTLIER_GAIN = 20.0
DECODE_LAYERS_8B = 36

M_SWEEP_8B = (1, 2, 4, 8)
M_SWEEP_32B = (1, 4)
# batch sizes past the small-M range (tensor-core kernel only): the GEMV /
# tensor-core crossover study of the README's `gemv_max_m` knob
M_SWEEP_WIDE = (12, 16, 24, 32)


def weight_seed(base: int, layer: int, j: int) -> int:
    """Seed of linear j (0..3) of decoder layer ``layer``."""
    return base + 4 * layer + j


def weights(n: int, k: int, std: float, seed: int) -> np.ndarray:
    """W[n, k] float32 ~ N(0, std^2)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, k), dtype=np.float32)
    w *= np.float32(std)
    return w


def outlier_channels(k: int, seed: int) -> np.ndarray:
    """The ``round(0.005 k)`` outlier channel indices for a layer of width k."""
    count = int(round(OUTLIER_FRACTION * k))
    rng = np.random.default_rng(seed + 1_000_003)
    return np.sort(rng.permutation(k)[:count])


def activations(m: int, k: int, seed: int, outliers: bool = True) -> np.ndarray:
    """X[m, k] float32 ~ N(0, 1), with the layer's outlier channels x20."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32)
    if outliers:
        x[:, outlier_channels(k, seed)] *= np.float32(OUTLIER_GAIN)
    return x


def uniform(shape, lo: float, hi: float, seed: int) -> np.ndarray:
    """Uniform float32 draws (edge-case inputs: exercise every E4M3 exponent)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def log_uniform_blocks(rows: int, k: int, seed: int, lo_exp: float = -12.0,
                       hi_exp: float = 4.0) -> np.ndarray:
    """Gaussian rows whose 16-element blocks carry gains 2^u, u ~ U(lo, hi):
    spreads the block amax over many decades so block scales hit E4M3
    subnormals, normals and saturation."""
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((rows, k), dtype=np.float32)
    gains = np.exp2(rng.uniform(lo_exp, hi_exp, size=(rows, k // 16))).astype(np.float32)
    t *= np.repeat(gains, 16, axis=1)
    return t
