"""Layer glue without reductions (test infrastructure only): embedding gather,
residual add (of two bf16 tensors, or of a bf16 tensor and an unrounded
product), SwiGLU.  None of these sums across elements, so each is
batch-invariant by construction; they are here because the decoder step needs
them.  SwiGLU: a = silu(g) * u with silu(g) = g / (1 + e^-g)."""
from __future__ import annotations

import numpy as np

from . import bf16


def embed(table_bits: np.ndarray, ids) -> np.ndarray:
    return table_bits[np.asarray(ids, dtype=np.int64)].copy()


def add(x_bits, y_bits) -> np.ndarray:
    return bf16.from_f64(bf16.to_f64(x_bits) + bf16.to_f64(y_bits))


def add_f64(x_bits, y: np.ndarray) -> np.ndarray:
    """bf16(x + y) for a bf16 x and an unrounded fp64 y: the residual stream
    plus a projection output that is never stored on its own, rounded once."""
    return bf16.from_f64(bf16.to_f64(x_bits) + np.asarray(y, dtype=np.float64))


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu(gu_bits: np.ndarray) -> np.ndarray:
    """gu [M][2F] holds gate in columns [0, F) and up in [F, 2F) (bf16)."""
    return swiglu_f64(bf16.to_f64(gu_bits))


def swiglu_f64(gu: np.ndarray) -> np.ndarray:
    """The same on unrounded fp64 gate/up values (the fused gate/up GEMM keeps
    g and u in its fp32 accumulators and rounds only the product)."""
    f = gu.shape[-1] // 2
    with np.errstate(over="ignore"):
        return bf16.from_f64(silu(gu[..., :f]) * gu[..., f:])
