"""Softmax attention for decode and causal prefill (test infrastructure only).

Follows "Deterministic and bit-exact inference" (M-0002), *technical*:
attention is made batch-invariant by cutting the keys into splits of one fixed
length, not into a fixed number of splits.  The split is how the GPU
schedules the sum; the quantity itself is plain softmax attention, so the
oracle computes it unsplit, in fp64:

    o[b, h] = sum_{j < L_b} softmax_j(scale * q[b, h] . k[b, j, g]) * v[b, j, g]

with g = h // (Hq / Hkv) (grouped-query attention, consecutive query heads
share a key/value head) and scale = 1/sqrt(D) unless given.  A sequence with
L_b = 0 has nothing to attend to; its output is zero.  Causal prefill: the
query at absolute position p sees keys 0..p.

``split_merge`` restates the same value as per-split partials (m, l, o) folded
left to right with the log-sum-exp merge; the tests check that it equals the
unsplit form for any split length, which is the identity the GPU's fixed-split
kernels rely on.
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16


def _attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [H][D], k/v [L][H][D] already expanded to query heads -> [H][D]."""
    if k.shape[0] == 0:
        return np.zeros_like(q)
    s = np.einsum("hd,lhd->hl", q, k) * scale
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", p, v)


def _expand(kv: np.ndarray, hq: int) -> np.ndarray:
    """[L][Hkv][D] -> [L][Hq][D] by repeating each kv head Hq/Hkv times."""
    return np.repeat(kv, hq // kv.shape[1], axis=1)


def decode(q_bits, k_cache_bits, v_cache_bits, lengths, scale=None):
    """q [B][Hq][D]; caches [B][Lmax][Hkv][D]; lengths [B] -> bf16 [B][Hq][D]."""
    q = bf16.to_f64(q_bits)
    bsz, hq, d = q.shape
    if hq % k_cache_bits.shape[2]:
        raise ValueError("Hq must be a multiple of Hkv")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = np.zeros_like(q)
    for b in range(bsz):
        n = int(lengths[b])
        k = _expand(bf16.to_f64(k_cache_bits[b, :n]), hq)
        v = _expand(bf16.to_f64(v_cache_bits[b, :n]), hq)
        out[b] = _attend(q[b], k, v, scale)
    return bf16.from_f64(out)


def prefill(q_bits, k_cache_bits, v_cache_bits, p0: int, scale=None):
    """One sequence: q [T][Hq][D] at absolute positions p0..p0+T-1; the cache
    [Lmax][Hkv][D] already holds keys 0..p0+T-1.  Row t sees keys 0..p0+t."""
    q = bf16.to_f64(q_bits)
    t_len, hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    k_all = _expand(bf16.to_f64(k_cache_bits[: p0 + t_len]), hq)
    v_all = _expand(bf16.to_f64(v_cache_bits[: p0 + t_len]), hq)
    out = np.zeros_like(q)
    for t in range(t_len):
        n = p0 + t + 1
        out[t] = _attend(q[t], k_all[:n], v_all[:n], scale)
    return bf16.from_f64(out)


def split_merge(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, split_len: int) -> np.ndarray:
    """fp64 q [H][D], k/v [L][H][D]: partials per split of ``split_len`` keys at
    absolute offsets 0, split_len, ...; each partial is (m, l, o) with m the
    split's max score, l = sum e^(s - m), o = sum e^(s - m) v (unnormalised);
    folded in ascending split order, then o / l."""
    n = k.shape[0]
    h, d = q.shape
    if n == 0:
        return np.zeros_like(q)
    m_acc = np.full(h, -np.inf)
    l_acc = np.zeros(h)
    o_acc = np.zeros((h, d))
    for s0 in range(0, n, split_len):
        ks, vs = k[s0: s0 + split_len], v[s0: s0 + split_len]
        sc = np.einsum("hd,lhd->hl", q, ks) * scale
        m_s = sc.max(axis=1)
        e = np.exp(sc - m_s[:, None])
        l_s = e.sum(axis=1)
        o_s = np.einsum("hl,lhd->hd", e, vs)
        m_new = np.maximum(m_acc, m_s)
        a = np.exp(m_acc - m_new)
        c = np.exp(m_s - m_new)
        l_acc = l_acc * a + l_s * c
        o_acc = o_acc * a[:, None] + o_s * c[:, None]
        m_acc = m_new
    return o_acc / l_acc[:, None]
