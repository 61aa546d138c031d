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
kernel forms every mass it compares (the total, the entropy, the mass at or
above a key, the kept mass) as a sum over the whole row: 4 terms in order per
lane of a 128-id block, a 32-lane butterfly, a butterfly over the 32 blocks of
a 4096-id group, then the groups in order, each term exp(s_i - s_0) with its
argument rounded once (|s_i - s_0| units in the last place, at most 60 for
any term of weight above 1e-26, plus exp's own 2); the margin there is
``whole_tol(V) = 4e-6 + whole_sum_tol(V)``.  Thousands of candidates then sit
near a deep top-p or min-p cut, each with a tiny weight, so a cut there is a
near tie only if it can move the token: the draw is made with the smallest and
the largest kept prefix the margins allow, and the row is a near tie if the
two picks differ or either draw falls within the margin of a boundary.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .philox import sampler_uniform


def tie_tol(k: int) -> float:
    return 1e-5 + k * 6e-8


def whole_sum_tol(v: int) -> float:
    """Relative error bound of an fp32 sum of v nonnegative terms taken as
    128-term blocks (4 in order per lane, then a 32-lane butterfly), 4096-term
    groups (a butterfly over 32 blocks) and the groups in order: one rounding
    per addition along the longest chain."""
    groups = (v + 4095) // 4096
    chain = 4 + 5 + 5 + groups
    return chain * 2.0 ** -24


def whole_tol(v: int) -> float:
    return 4e-6 + whole_sum_tol(v)


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


def sample_row(logits_f32: np.ndarray, history, step: int, p: SamplingParams, allowed=None):
    """Returns (token, near_tie).  Over the whole vocabulary, a set passed as
    `allowed` receives every token a draw within the margins can give (the
    kept prefixes the margins allow, each with its draw target moved by the
    margin either way); for a near tie the kernel's token must be one of
    them."""
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
    tol = whole_tol(v) if whole else tie_tol(len(order))
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
    cum_all = np.cumsum(em)
    u = sampler_uniform(p.seed, step)
    first = int(np.argmax(kept))                # the first kept candidate

    def top_p_keep(target):
        return max(1, min(int(np.searchsorted(cum_all, target, side="left")) + 1, n))

    def min_p_keep(keep, thr):
        """the first kept candidate before `keep` whose e is below thr, else keep"""
        below = np.nonzero(kept[:keep] & ~(e[:keep] >= thr))[0]
        return int(below[0]) if len(below) else keep

    def draw(keep):
        cum = cum_all[:keep]
        target = u * cum[-1]
        idx = int(np.searchsorted(cum, target, side="right"))
        if idx >= keep:                               # (u < 1 never gets here) the last kept one
            idx = max(j for j in range(keep) if kept[j])
        # the pick moves if cum[idx] or cum[idx-1] sits at the target
        at_edge = bool(np.any(np.abs(cum[max(0, idx - 1): idx + 1] - target) <= tol * cum[-1]))
        return idx, at_edge

    keep = n
    if p.top_p < 1.0:
        target = float(np.float32(p.top_p)) * cum_all[-1]
        keep = top_p_keep(target)
        # the cut moves if cum[keep-1] or cum[keep-2] sits at the target
        if not whole and np.any(np.abs(cum_all[max(0, keep - 2): keep] - target) <= tol * cum_all[-1]):
            near = True
    keep_tp = keep
    if p.min_p > 0.0:
        thr = float(np.float32(p.min_p)) * e[first]
        if not whole:
            idx_k = [j for j in range(keep) if kept[j]]
            ok = [j for j in idx_k if e[j] >= thr]
            drop = [j for j in idx_k if not e[j] >= thr]
            # the cut moves if the last kept or the first dropped e sits at the threshold
            edge = ([ok[-1]] if ok else []) + ([drop[0]] if drop else [])
            if any(abs(e[j] - thr) <= tol for j in edge):
                near = True
        keep = max(min_p_keep(keep, thr), first + 1)
    idx, at_edge = draw(keep)
    near = near or at_edge
    if whole and (p.top_p < 1.0 or p.min_p > 0.0):
        # the smallest and the largest kept prefix within the margins
        k_lo, k_hi = keep_tp, keep_tp
        if p.top_p < 1.0:
            target = float(np.float32(p.top_p)) * cum_all[-1]
            k_lo = top_p_keep(target - tol * cum_all[-1])
            k_hi = top_p_keep(target + tol * cum_all[-1])
        if p.min_p > 0.0:
            thr = float(np.float32(p.min_p)) * e[first]
            k_lo = max(min_p_keep(k_lo, thr * (1.0 + tol)), first + 1)
            k_hi = max(min_p_keep(k_hi, thr * (1.0 - tol)), first + 1)
        for kk in (k_lo, k_hi):
            j, edge = draw(kk)
            if j != idx or edge:
                near = True
    if whole and allowed is not None:
        ks = [keep]
        if p.top_p < 1.0 or p.min_p > 0.0:
            ks += [k_lo, k_hi]
        for kk in ks:
            cum = cum_all[:kk]
            m = tol * cum[-1]
            target = u * cum[-1]
            lo = int(np.searchsorted(cum, target - m, side="right"))
            hi = min(int(np.searchsorted(cum, target + m, side="right")), kk - 1)
            allowed.update(int(order[j]) for j in range(min(lo, kk - 1), hi + 1) if kept[j])
    return int(order[idx]), near


def sample(logits_f32: np.ndarray, histories, steps, params):
    """logits [B][V] float32; per-row history lists, steps and params."""
    toks, ties = [], []
    for b in range(logits_f32.shape[0]):
        t, n = sample_row(logits_f32[b], histories[b], int(steps[b]), params[b])
        toks.append(t)
        ties.append(n)
    return np.array(toks, dtype=np.int32), np.array(ties, dtype=bool)
