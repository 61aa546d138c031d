"""The seeded sampler (test infrastructure only).

Follows Kinetic "Receipts", *Making a receipt*: a receipt records every sampler
setting -- temperature, top_k, top_p, min_p, typical-p, the repeat, presence
and frequency penalties, logit bias, repeat_last_n -- and the seed; a request without a seed gets a fresh one that is recorded.  The
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
4a. Typical-p (only if 0 < typical_p < 1; locally typical sampling, Meister et
   al. 2022): with p_i = e_i / sum(e) over the candidates and
   H = -sum p_i log p_i, order the candidates by |-log p_i - H| (then by
   candidate order) and keep the shortest such prefix whose p reaches
   typical_p (at least one).  The kept set keeps its candidate order and may
   leave out the most likely id.
5. Top-p (only if top_p < 1): over the kept candidates in candidate order,
   keep the shortest prefix whose sum of e reaches top_p * (their sum of e)
   (at least one candidate).
6. Min-p (only if min_p > 0): keep the candidates with p_i >= min_p * p_max,
   p_max the largest kept p, i.e. e_i >= min_p * e_first (e_first the first
   kept e; = 1 unless typical-p left out the first candidate).
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
    typical_p: float = 1.0


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
    n = len(order)
    kept = np.ones(n, dtype=bool)               # the set, in candidate order
    tp = float(np.float32(p.typical_p))
    if 0.0 < tp < 1.0:
        pr = e / e.sum()
        pos = pr > 0
        lp = np.log(np.where(pos, pr, 1.0))
        h = -float(np.sum(np.where(pos, pr * lp, 0.0)))
        eps = np.where(pos, np.abs(-lp - h), np.inf)
        torder = np.lexsort((np.arange(n), eps))  # typicality ascending, then candidate order
        cum_t = np.cumsum(pr[torder])
        m = max(1, min(int(np.searchsorted(cum_t, tp, side="left")) + 1, n))
        # the cut moves if the kept mass sits at typical_p, or if the last kept
        # and the first dropped candidate are equally typical within the error
        if np.any(np.abs(cum_t[max(0, m - 2): m] - tp) <= tol):
            near = True
        if m < n and abs(eps[torder[m]] - eps[torder[m - 1]]) <= 4 * tol * (1.0 + abs(h)):
            near = True
        kept[:] = False
        kept[torder[:m]] = True
    em = np.where(kept, e, 0.0)
    keep = n
    if p.top_p < 1.0:
        cum = np.cumsum(em)
        target = float(np.float32(p.top_p)) * cum[-1]
        keep = int(np.searchsorted(cum, target, side="left")) + 1
        keep = max(1, min(keep, n))
        # the cut moves if cum[keep-1] or cum[keep-2] sits at the target
        if np.any(np.abs(cum[max(0, keep - 2): keep] - target) <= tol * cum[-1]):
            near = True
    first = int(np.argmax(kept))                # the first kept candidate
    if p.min_p > 0.0:
        thr = float(np.float32(p.min_p)) * e[first]
        idx_k = [j for j in range(keep) if kept[j]]
        ok = [j for j in idx_k if e[j] >= thr]
        drop = [j for j in idx_k if not e[j] >= thr]
        # the cut moves if the last kept or the first dropped e sits at the threshold
        edge = ([ok[-1]] if ok else []) + ([drop[0]] if drop else [])
        if any(abs(e[j] - thr) <= tol for j in edge):
            near = True
        keep = drop[0] if drop else keep
        keep = max(keep, first + 1)
    em = em[:keep]
    cum = np.cumsum(em)
    u = sampler_uniform(p.seed, step)
    target = u * cum[-1]
    idx = int(np.searchsorted(cum, target, side="right"))
    if idx >= keep:                               # (u < 1 never gets here) the last kept one
        idx = max(j for j in range(keep) if kept[j])
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
