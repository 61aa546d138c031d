"""bf16 <-> fp64 conversions for the oracle (test infrastructure only).

bf16 keeps fp32's 8-bit exponent and 7 stored fraction bits.  Widening a bf16
bit pattern to fp64 is exact.  Narrowing rounds once, to nearest with ties to
even, directly from fp64 (no intermediate fp32 rounding, which could round
twice).
"""
from __future__ import annotations

import numpy as np

_FRAC_DROP = 52 - 7           # fp64 fraction bits that bf16 does not keep
_HALF = np.uint64((1 << (_FRAC_DROP - 1)) - 1)
_LOW = np.uint64((1 << _FRAC_DROP) - 1)
_TINY = 2.0 ** -126           # below this bf16 is subnormal (spacing 2^-133)


def to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def from_f64(x) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    bits = x.view(np.uint64).copy()
    lsb = (bits >> np.uint64(_FRAC_DROP)) & np.uint64(1)
    bits = (bits + _HALF + lsb) & ~_LOW
    with np.errstate(over="ignore"):
        f32 = bits.view(np.float64).astype(np.float32)   # exact: <= 8 significant bits
    out = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    tiny = np.abs(x) < _TINY
    if tiny.any():
        q = np.rint(x[tiny] / 2.0 ** -133) * 2.0 ** -133    # np.rint rounds half to even
        out[tiny] = (q.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def round_f64(x) -> np.ndarray:
    """fp64 -> the fp64 value of its bf16 rounding."""
    return to_f64(from_f64(x))
