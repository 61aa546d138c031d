"""RMSNorm (test infrastructure only).

Follows "Deterministic and bit-exact inference" (M-0002), *technical*: RMSNorm
is one of the three kernels made batch-invariant.  The pages name the operation
but print no formula; the plain definition (gain form, as in Llama/Qwen-style
decoders) is

    y_i = x_i / sqrt(mean_j(x_j^2) + eps) * w_i

with eps = 1e-6 for the decoder layers used here.  With a residual r the fused
form first forms the new residual stream s = bf16(x + r) (the sum of two bf16
values is exact in fp64, so one rounding), then normalises s.
"""
from __future__ import annotations

import numpy as np

from . import bf16


def rmsnorm_f64(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Unrounded RMSNorm of fp64 rows x [rows][d] with gains w [d]."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rmsnorm(x_bits, w_bits, eps: float = 1e-6, residual_bits=None):
    """bf16 in, bf16 out.  Returns y, or (y, s) when a residual is given."""
    x = bf16.to_f64(x_bits)
    w = bf16.to_f64(w_bits)
    if residual_bits is None:
        return bf16.from_f64(rmsnorm_f64(x, w, eps))
    s_bits = bf16.from_f64(x + bf16.to_f64(residual_bits))
    return bf16.from_f64(rmsnorm_f64(bf16.to_f64(s_bits), w, eps)), s_bits
