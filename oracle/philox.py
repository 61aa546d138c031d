"""Philox4x32-10 counter-based generator, written from its published definition.

Test infrastructure only (see ``oracle/__init__.py``).

Definition followed: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
easy as 1, 2, 3" (SC'11), the Philox-4x32 bijection with R = 10 rounds.  One
round maps a counter (c0, c1, c2, c3) under a key (k0, k1) to

    (hi0, lo0) = 64-bit product M0 * c0 split in halves
    (hi1, lo1) = 64-bit product M1 * c2 split in halves
    (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)

and between rounds the key is bumped by the Weyl constants (k0 += W0, k1 += W1,
modulo 2^32).  The multipliers and Weyl constants are the ones the paper gives
for Philox-4x32.

Two independent restatements are kept on purpose: ``philox4x32_10`` works on
Python integers one counter at a time, ``philox4x32_10_np`` on NumPy uint64
vectors.  The tests check that they agree and that their output is uniform.

How the sampler uses it (the pages ask for a seeded sampler whose seed is
recorded -- Kinetic "Receipts", *Making a receipt*, the ``sampling.seed``
field): key = (low 32 bits of the request seed, high 32 bits), counter =
(low 32 bits of the request-local step, high 32 bits, 0, 0); the uniform draw is
u = (word0 >> 8) * 2^-24, which is exact in fp32 and fp64.
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
ROUNDS = 10
_MASK = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Scalar Philox-4x32-10 on Python ints: counter is 4 words, key 2 words."""
    c0, c1, c2, c3 = (int(v) & _MASK for v in counter)
    k0, k1 = (int(v) & _MASK for v in key)
    for r in range(ROUNDS):
        if r:
            k0 = (k0 + W0) & _MASK
            k1 = (k1 + W1) & _MASK
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return (c0, c1, c2, c3)


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox-4x32-10: every argument is an array (or scalar) of
    32-bit words; returns four uint32 arrays.  Products are formed in uint64,
    where a 32x32-bit product cannot overflow."""
    c = [np.asarray(v, dtype=np.uint64) & np.uint64(_MASK) for v in (c0, c1, c2, c3)]
    k = [np.asarray(v, dtype=np.uint64) & np.uint64(_MASK) for v in (k0, k1)]
    shape = np.broadcast_shapes(*(a.shape for a in c + k))
    c = [np.broadcast_to(a, shape).copy() for a in c]
    k = [np.broadcast_to(a, shape).copy() for a in k]
    m32 = np.uint64(_MASK)
    for r in range(ROUNDS):
        if r:
            k[0] = (k[0] + np.uint64(W0)) & m32
            k[1] = (k[1] + np.uint64(W1)) & m32
        p0 = np.uint64(M0) * c[0]
        p1 = np.uint64(M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & m32
        hi1, lo1 = p1 >> np.uint64(32), p1 & m32
        c = [hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0]
    return tuple(a.astype(np.uint32) for a in c)


def uniform_from_word(word0) -> float:
    """Top 24 bits of a 32-bit word scaled to [0, 1): exact in fp32 and fp64."""
    return float(int(word0) >> 8) * (1.0 / 16777216.0)


def sampler_uniform(seed: int, step: int) -> float:
    """The one uniform draw the sampler takes for request ``seed`` at its
    request-local token index ``step`` (never the batch slot)."""
    seed &= (1 << 64) - 1
    step &= (1 << 64) - 1
    w = philox4x32_10((step & _MASK, step >> 32, 0, 0), (seed & _MASK, seed >> 32))
    return uniform_from_word(w[0])
