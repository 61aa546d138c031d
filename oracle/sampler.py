"""The seeded sampler (test infrastructure only).

Follows Kinetic "Receipts", *Making a receipt*: a receipt records every sampler
setting -- temperature, top_k, top_p, min_p, the repeat, presence and
frequency penalties, logit bias, repeat_last_n -- and the seed; a request without a seed gets a fresh one that is recorded.  The
receipt's example uses temperature 0.8, top_k 50, top_p 0.95, min_p 0.05,
repeat_penalty 1.1, presence_penalty 0, frequency_penalty 0, repeat_last_n 64,
seed 42.

The pages list the settings but not the order in which they act, nor their
exact forms.  The reading taken here (the usual one for these knobs):

0. Logit bias: each (id, b) of the request's list adds b to logit id (fp32,
   in list order; ids outside the vocabulary are ignored).
1. Penalties, once per distinct id among the last ``repeat_last_n`` tokens
   of the request (n < 0: all of them, n = 0: none), c its count there:
   first the repeat penalty, z <- z / r if z > 0 else z * r; then the presence
   and frequency penalties, z <- z - (c * f + p) (f the frequency penalty, p
   the presence penalty; each operation rounded to fp32, skipped when both
   are 0).
2. Temperature <= 0 is greedy: the largest z, lowest id on ties.
3. Candidates: the top_k largest z ordered by (z descending, id ascending);
   top_k <= 0 or >= V keeps every id in that order.
4. s = z / T; e_i = exp(s_i - s_0) (s_0 is the largest, so e_0 = 1).
5. Top-p (only if top_p < 1): keep the shortest prefix whose sum of e reaches
   top_p * sum(e) (at least one candidate).
6. Min-p (only if min_p > 0): keep the candidates with p_i >= min_p * p_max,
   i.e. e_i >= min_p, since e_0 = 1 is the largest.
7. Draw u = Philox4x32-10 word 0 >> 8, times 2^-24, keyed by the request seed,
   counter = the request-local token index; return the first kept candidate
   whose running sum of e exceeds u * (sum of kept e).

Precision: the penalty, the temperature division and the ranking decide
integers (which ids survive, in which order), so they are taken in fp32 with
correctly rounded division and multiplication, as the kernel takes them; those
decisions are then identical on both sides.  The exponentials and sums are
fp64 here and fp32 on the GPU, so a draw or a top-p / min-p cut that falls
within a margin of a boundary is reported as a near tie, and token parity is
not asserted for such a row.  The margin (relative to the sum) bounds the
kernel's fp32 error: a sequential sum of k terms below 1 is off by at most
k * 2^-24 relative, and each exponential by a few units in the last place, so
``tie_tol(k) = 1e-5 + k * 6e-8``.  Over the whole vocabulary (no top-k) the
kernel still forms its running sums over at most 1024 ranked candidates, and
the whole-row total per 128-id block and then in 32 strided runs of blocks,
so k is the candidate count (at most 1024) and the total adds
``whole_sum_tol(V)`` more.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .philox import sampler_uniform


def tie_tol(k: int) -> float:
    return 1e-5 + k * 6e-8


def whole_sum_tol(v: int) -> float:
    """Relative error bound of an fp32 sum of v terms taken as 128-term blocks
    (4 in order per lane, then a 32-lane butterfly) and then 32 strided runs of
    blocks added in order and by a butterfly: one rounding per addition along
    the longest chain."""
    blocks = (v + 127) // 128
    chain = 4 + 5 + (blocks + 31) // 32 + 5
    return chain * 2.0 ** -24


@dataclass
class SamplingParams:
    temperature: float = 0.8
    top_k: int = 50
    top_p: float = 0.95
    min_p: float = 0.05
    repeat_penalty: float = 1.1
    repeat_last_n: int = 64
    seed: int = 42
    presence_penalty: float = 0.0
    frequency_penalty: float = 0.0
    logit_bias: dict = None   # {id: bias}; applied in insertion order


def bias_logits(logits_f32: np.ndarray, p: SamplingParams) -> np.ndarray:
    z = np.array(logits_f32, dtype=np.float32, copy=True)
    for t, b in (p.logit_bias or {}).items():
        t = int(t)
        if 0 <= t < z.shape[0]:
            z[t] = z[t] + np.float32(b)
    return z


def penalize(logits_f32: np.ndarray, history, p: SamplingParams) -> np.ndarray:
    z = np.array(logits_f32, dtype=np.float32, copy=True)
    r = np.float32(p.repeat_penalty)
    fq = np.float32(p.frequency_penalty)
    pr = np.float32(p.presence_penalty)
    additive = fq != 0 or pr != 0
    n = int(p.repeat_last_n)
    hist = list(history)
    if (r == np.float32(1.0) and not additive) or n == 0 or not hist:
        return z
    window = [int(t) for t in (hist if n < 0 else hist[-n:])]
    for t in sorted(set(window)):
        if 0 <= t < z.shape[0]:
            z[t] = z[t] / r if z[t] > 0 else z[t] * r
            if additive:
                c = np.float32(window.count(t))
                z[t] = z[t] - (c * fq + pr)
    return z


def sample_row(logits_f32: np.ndarray, history, step: int, p: SamplingParams):
    """Returns (token, near_tie)."""
    z = penalize(bias_logits(logits_f32, p), history, p)
    v = z.shape[0]
    t = np.float32(p.temperature)
    if not (t > 0):
        return int(np.argmax(z)), False
    order = np.lexsort((np.arange(v), -z))       # z descending, then id ascending
    k = int(p.top_k)
    if 0 < k < v:
        order = order[:k]
    s = (z[order] / t).astype(np.float64)          # fp32 division, widened exactly
    e = np.exp(s - s[0])
    whole = len(order) > 1024
    tol = tie_tol(min(len(order), 1024)) + (whole_sum_tol(v) if whole else 0.0)
    near = False
    keep = len(order)
    if p.top_p < 1.0:
        cum = np.cumsum(e)
        target = float(np.float32(p.top_p)) * cum[-1]
        keep = int(np.searchsorted(cum, target, side="left")) + 1
        keep = max(1, min(keep, len(order)))
        # the cut moves if cum[keep-1] or cum[keep-2] sits at the target
        if np.any(np.abs(cum[max(0, keep - 2): keep] - target) <= tol * cum[-1]):
            near = True
    if p.min_p > 0.0:
        mp = float(np.float32(p.min_p))
        ok = e[:keep] >= mp
        n_ok = int(np.count_nonzero(ok))
        # the cut moves if the last kept or the first dropped e sits at min_p
        if np.any(np.abs(e[max(0, n_ok - 1): min(n_ok + 1, keep)] - mp) <= tol):
            near = True
        keep = max(1, n_ok)
    e = e[:keep]
    cum = np.cumsum(e)
    u = sampler_uniform(p.seed, step)
    target = u * cum[-1]
    idx = int(np.searchsorted(cum, target, side="right"))
    idx = min(idx, keep - 1)
    # the pick moves if cum[idx] or cum[idx-1] sits at the target
    if np.any(np.abs(cum[max(0, idx - 1): idx + 1] - target) <= tol * cum[-1]):
        near = True
    return int(order[idx]), near


def sample(logits_f32: np.ndarray, histories, steps, params):
    """logits [B][V] float32; per-row history lists, steps and params."""
    toks, ties = [], []
    for b in range(logits_f32.shape[0]):
        t, n = sample_row(logits_f32[b], histories[b], int(steps[b]), params[b])
        toks.append(t)
        ties.append(n)
    return np.array(toks, dtype=np.int32), np.array(ties, dtype=bool)
