"""Pins for the attention oracle: special cases with closed forms, brute force
on tiny inputs, the split-and-merge identity, causality and GQA grouping."""
import math

import numpy as np

from oracle import attention, bf16


def _b(x):
    return bf16.from_f64(np.asarray(x, np.float64))


def _rand(shape, rng, s=1.0):
    return _b(rng.standard_normal(shape) * s)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    q = _rand((1, 4, 64), rng)
    k = _rand((1, 8, 2, 64), rng)
    v = _rand((1, 8, 2, 64), rng)
    out = attention.decode(q, k, v, [1])
    assert np.array_equal(out[0, :2], np.stack([v[0, 0, 0]] * 2))
    assert np.array_equal(out[0, 2:], np.stack([v[0, 0, 1]] * 2))


def test_equal_scores_give_mean_of_values_and_empty_gives_zero():
    rng = np.random.default_rng(1)
    v = _rand((1, 16, 1, 32), rng)
    k = _rand((1, 16, 1, 32), rng)
    q = _b(np.zeros((1, 2, 32)))          # q = 0: every score is 0
    out = bf16.to_f64(attention.decode(q, k, v, [10]))
    assert np.array_equal(out[0, 0], bf16.round_f64(bf16.to_f64(v)[0, :10, 0].mean(0)))
    assert np.all(bf16.to_f64(attention.decode(q, k, v, [0])) == 0)


def test_dominant_key_selects_its_value():
    d = 64
    k = np.zeros((1, 5, 1, d))
    k[0, 3, 0, 0] = 64.0              # score 64 / 8 * 8 = 64 above the rest
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 8.0
    rng = np.random.default_rng(2)
    v = _rand((1, 5, 1, d), rng)
    out = attention.decode(_b(q), _b(k), v, [5])
    assert np.array_equal(out[0, 0], v[0, 3, 0])


def test_brute_force_tiny_with_gqa_grouping():
    rng = np.random.default_rng(3)
    hq, hk, d, n = 4, 2, 8, 6
    q, k, v = _rand((1, hq, d), rng), _rand((1, n, hk, d), rng), _rand((1, n, hk, d), rng)
    qf, kf, vf = bf16.to_f64(q)[0], bf16.to_f64(k)[0], bf16.to_f64(v)[0]
    out = bf16.to_f64(attention.decode(q, k, v, [n]))[0]
    for h in range(hq):
        g = h // (hq // hk)               # heads 0,1 -> kv 0; heads 2,3 -> kv 1
        sc = [sum(qf[h, t] * kf[j, g, t] for t in range(d)) / math.sqrt(d) for j in range(n)]
        mx = max(sc)
        ex = [math.exp(s - mx) for s in sc]
        tot = sum(ex)
        ref = [sum(ex[j] / tot * vf[j, g, t] for j in range(n)) for t in range(d)]
        assert np.array_equal(out[h], bf16.round_f64(np.array(ref)))


def test_split_merge_identity_any_split():
    rng = np.random.default_rng(4)
    h, d, n = 3, 16, 1000
    q = rng.standard_normal((h, d)) * 2
    k = rng.standard_normal((n, h, d))
    v = rng.standard_normal((n, h, d))
    s = np.einsum("hd,lhd->hl", q, k) * 0.25
    p = np.exp(s - s.max(1, keepdims=True))
    ref = np.einsum("hl,lhd->hd", p / p.sum(1, keepdims=True), v)
    for split in (1, 7, 64, 256, 999, 1000, 4096):
        assert np.allclose(attention.split_merge(q, k, v, 0.25, split), ref, rtol=0, atol=1e-12)


def test_prefill_is_causal_and_row_equals_decode():
    rng = np.random.default_rng(5)
    hq, hk, d, t_len, p0 = 4, 2, 16, 5, 3
    kc, vc = _rand((12, hk, d), rng), _rand((12, hk, d), rng)
    q = _rand((t_len, hq, d), rng)
    out = attention.prefill(q, kc, vc, p0)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[p0 + 2:] = _rand((12 - p0 - 2, hk, d), rng)   # change keys after row 1's position
    vc2[p0 + 2:] = _rand((12 - p0 - 2, hk, d), rng)
    out2 = attention.prefill(q, kc2, vc2, p0)
    assert np.array_equal(out[:2], out2[:2]) and not np.array_equal(out[2:], out2[2:])
    for t in range(t_len):
        dec = attention.decode(q[t: t + 1], kc[None], vc[None], [p0 + t + 1])
        assert np.array_equal(out[t], dec[0])
