"""Matrix multiplication C = A . W^T (test infrastructure only).

Follows "Deterministic and bit-exact inference" (trustbutveri.fyi, M-0002),
*technical*: matrix multiplication is one of the three kernels the invariant
route makes batch-invariant.  The plain definition is C[i, j] = sum_k A[i, k] *
W[j, k]; W is stored [N][K] (one row per output feature).  The oracle sums in
fp64 (the GPU accumulates in fp32) and rounds once at the output: to bf16, or to
fp32 when the caller asks for an fp32 result (the LM head's logits).
"""
from __future__ import annotations

import numpy as np

from . import bf16


def gemm(a_bits: np.ndarray, w_bits: np.ndarray, out: str = "bf16") -> np.ndarray:
    """a_bits [M][K] bf16, w_bits [N][K] bf16 -> [M][N] (bf16 bits or float32)."""
    a = bf16.to_f64(a_bits)
    w = bf16.to_f64(w_bits)
    if a.shape[1] != w.shape[1]:
        raise ValueError("inner dimensions differ")
    c = a @ w.T
    if out == "bf16":
        return bf16.from_f64(c)
    if out == "f32":
        return c.astype(np.float32)
    if out == "f64":
        return c
    raise ValueError(out)


def gemm_f64_rows(a_bits: np.ndarray, w_bits: np.ndarray, rows, cols=None) -> np.ndarray:
    """Exact fp64 values of selected outputs (for sampled checks at full size):
    C[rows][:, cols] without forming the whole product."""
    a = bf16.to_f64(a_bits[rows])
    w = bf16.to_f64(w_bits if cols is None else w_bits[cols])
    return a @ w.T


def matmul(a: np.ndarray, w_bits: np.ndarray, out: str = "bf16") -> np.ndarray:
    """The same product for an fp64 left operand that was never rounded to bf16
    (a normalised row that the GPU path keeps inside its projection)."""
    w = bf16.to_f64(w_bits)
    if a.shape[1] != w.shape[1]:
        raise ValueError("inner dimensions differ")
    c = np.asarray(a, dtype=np.float64) @ w.T
    if out == "bf16":
        return bf16.from_f64(c)
    if out == "f32":
        return c.astype(np.float32)
    if out == "f64":
        return c
    raise ValueError(out)
