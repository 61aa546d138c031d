"""Rotary position embedding, rotate-half pairing (test infrastructure only).

The pages do not print RoPE; the layer workloads fix only its base (1e4 for the
small layer).  Plain definition used: for a head vector x of length D and
absolute position p, each pair (x_i, x_{i+D/2}), i < D/2, is rotated by
theta_i = p * base^(-2i/D):

    x_i'       = x_i * cos(theta_i) - x_{i+D/2} * sin(theta_i)
    x_{i+D/2}' = x_{i+D/2} * cos(theta_i) + x_i * sin(theta_i)

Optional per-head RMSNorm ("QK-norm") is applied before the rotation, without a
bf16 rounding in between; the result is rounded to bf16 once.
"""
from __future__ import annotations

import numpy as np

from . import bf16
from .rmsnorm import rmsnorm_f64


def angles(pos: np.ndarray, dim: int, base: float) -> np.ndarray:
    """theta [len(pos)][dim/2] in fp64."""
    i = np.arange(dim // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope_f64(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """x [T][H][D] fp64, pos [T] -> rotated fp64."""
    d = x.shape[-1]
    th = angles(pos, d, base)[:, None, :]
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope(x_bits, pos, base: float, norm_w_bits=None, eps: float = 1e-6):
    """bf16 [T][H][D] -> bf16, optional QK-norm first."""
    x = bf16.to_f64(x_bits)
    if norm_w_bits is not None:
        x = rmsnorm_f64(x, bf16.to_f64(norm_w_bits), eps)
    return bf16.from_f64(rope_f64(x, np.asarray(pos), base))
