"""Pins for Philox4x32-10 and the sampler oracle."""
import ctypes
import math
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox
from oracle.sampler import SamplingParams, bias_logits, penalize, sample_row


def test_philox_two_restatements_agree():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 2 ** 32, (200, 4), dtype=np.uint64)
    k = rng.integers(0, 2 ** 32, (200, 2), dtype=np.uint64)
    vec = philox.philox4x32_10_np(c[:, 0], c[:, 1], c[:, 2], c[:, 3], k[:, 0], k[:, 1])
    for i in range(200):
        ref = philox.philox4x32_10(tuple(int(x) for x in c[i]), tuple(int(x) for x in k[i]))
        assert tuple(int(v[i]) for v in vec) == ref


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """cuRAND's host Philox4_32_10 generator (a library routine) seeded with s
    emits, at offset 0, block j = Philox(counter=(0, 0, j, 0), key=(s_lo, s_hi))."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0
    try:
        for seed in (0, 42, 0x0123456789ABCDEF, 2 ** 64 - 1):
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0
            buf = (ctypes.c_uint * 64)()
            assert lib.curandGenerate(gen, buf, ctypes.c_size_t(64)) == 0
            for j in range(16):
                mine = philox.philox4x32_10((0, 0, j, 0), (seed & 0xFFFFFFFF, seed >> 32))
                assert tuple(buf[4 * j: 4 * j + 4]) == mine
    finally:
        lib.curandDestroyGenerator(gen)


def test_philox_uniformity():
    w = philox.philox4x32_10_np(np.arange(1 << 15), 0, 0, 0, 42, 0)
    u = (w[0] >> 8).astype(np.float64) / 2 ** 24
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    counts = np.bincount((w[1] >> 28).astype(np.int64), minlength=16)
    assert stats.chisquare(counts).pvalue > 1e-3


def _greedy_params(**kw):
    p = SamplingParams(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0, repeat_penalty=1.0,
                       repeat_last_n=0, seed=7)
    for a, b in kw.items():
        setattr(p, a, b)
    return p


def test_greedy_and_degenerate_filters_give_argmax():
    rng = np.random.default_rng(1)
    z = rng.standard_normal(1000).astype(np.float32)
    am = int(np.argmax(z))
    for p in (_greedy_params(temperature=0.0), _greedy_params(top_k=1),
              _greedy_params(top_k=50, top_p=1e-6), _greedy_params(top_k=50, min_p=1.0)):
        for step in range(20):
            assert sample_row(z, [], step, p)[0] == am
    z2 = np.zeros(10, np.float32)
    z2[[3, 7]] = 5.0                     # tie: lowest id wins
    assert sample_row(z2, [], 0, _greedy_params(temperature=0.0))[0] == 3
    assert sample_row(z2, [], 0, _greedy_params(top_k=1))[0] == 3


def test_repeat_penalty_closed_form():
    z = np.array([2.0, -2.0, 1.0, 0.0, 3.0], np.float32)
    p = _greedy_params(repeat_penalty=2.0, repeat_last_n=3)
    got = penalize(z, [4, 0, 1, 1, 0], p)      # last 3 = {1, 0}; id 4 is outside the window
    assert np.array_equal(got, np.array([1.0, -4.0, 1.0, 0.0, 3.0], np.float32))
    assert np.array_equal(penalize(z, [0, 1], _greedy_params(repeat_penalty=2.0, repeat_last_n=-1)),
                          np.array([1.0, -4.0, 1.0, 0.0, 3.0], np.float32))
    assert np.array_equal(penalize(z, [0, 1], _greedy_params(repeat_penalty=2.0, repeat_last_n=0)), z)


def test_presence_and_frequency_penalties_closed_form():
    # window (last 4) = [1, 0, 1, 1]: id 1 three times, id 0 once; id 4 outside
    z = np.array([2.0, -2.0, 1.0, 0.0, 3.0], np.float32)
    p = _greedy_params(repeat_penalty=1.0, repeat_last_n=4, frequency_penalty=0.5, presence_penalty=0.25)
    got = penalize(z, [4, 1, 0, 1, 1], p)
    # id 0: 2 - (1 * 0.5 + 0.25) = 1.25; id 1: -2 - (3 * 0.5 + 0.25) = -3.75
    assert np.array_equal(got, np.array([1.25, -3.75, 1.0, 0.0, 3.0], np.float32))
    # after the repeat penalty: id 0: 2 / 2 - 0.75 = 0.25; id 1: -2 * 2 - 1.75 = -5.75
    p2 = _greedy_params(repeat_penalty=2.0, repeat_last_n=4, frequency_penalty=0.5, presence_penalty=0.25)
    assert np.array_equal(penalize(z, [4, 1, 0, 1, 1], p2),
                          np.array([0.25, -5.75, 1.0, 0.0, 3.0], np.float32))
    # presence alone subtracts once per distinct id, frequency alone scales with the count
    pp = _greedy_params(repeat_penalty=1.0, repeat_last_n=-1, presence_penalty=1.0)
    assert np.array_equal(penalize(z, [0, 0, 0, 2], pp), np.array([1.0, -2.0, 0.0, 0.0, 3.0], np.float32))
    fp = _greedy_params(repeat_penalty=1.0, repeat_last_n=-1, frequency_penalty=1.0)
    assert np.array_equal(penalize(z, [0, 0, 0, 2], fp), np.array([-1.0, -2.0, 0.0, 0.0, 3.0], np.float32))
    # both zero: the repeat penalty alone (the receipt's example settings)
    assert np.array_equal(penalize(z, [0, 1], _greedy_params(repeat_penalty=2.0, repeat_last_n=-1)),
                          penalize(z, [0, 1], _greedy_params(repeat_penalty=2.0, repeat_last_n=-1,
                                                              presence_penalty=0.0, frequency_penalty=0.0)))
    # a penalty can move the greedy pick: id 4 (3.0) outranks id 0 (2.0) until id 4 is
    # penalised by more than 1
    z2 = np.array([2.0, 0.0, 0.0, 0.0, 3.0], np.float32)
    assert sample_row(z2, [4, 4], 0, _greedy_params(temperature=0.0, repeat_penalty=1.0,
                                                      frequency_penalty=0.75, repeat_last_n=-1))[0] == 0
    assert sample_row(z2, [4, 4], 0, _greedy_params(temperature=0.0, repeat_penalty=1.0,
                                                      frequency_penalty=0.25, repeat_last_n=-1))[0] == 4


def test_logit_bias_closed_form():
    z = np.array([2.0, -2.0, 1.0, 0.0, 3.0], np.float32)
    p = _greedy_params(logit_bias={1: 1.5, 4: -np.inf, 9: 100.0})   # id 9 is outside V = 5
    assert np.array_equal(bias_logits(z, p), np.array([2.0, -0.5, 1.0, 0.0, -np.inf], np.float32))
    # a banned id is never drawn, greedy or sampled
    assert sample_row(z, [], 0, _greedy_params(temperature=0.0, logit_bias={4: -np.inf}))[0] == 0
    for step in range(50):
        assert sample_row(z, [], step, _greedy_params(logit_bias={4: -np.inf}))[0] != 4
    # a large bias forces an id
    assert sample_row(z, [], 3, _greedy_params(logit_bias={3: 50.0}))[0] == 3
    # the bias comes before the penalties: id 0 biased to 6, then halved by the repeat penalty
    pb = _greedy_params(repeat_penalty=2.0, repeat_last_n=-1, logit_bias={0: 4.0})
    assert np.array_equal(penalize(bias_logits(z, pb), [0], pb),
                          np.array([3.0, -2.0, 1.0, 0.0, 3.0], np.float32))
    # an empty or absent list changes nothing (bit for bit, -0.0 included)
    zn = np.array([-0.0, 1.0], np.float32)
    assert np.signbit(bias_logits(zn, _greedy_params(logit_bias={}))[0])
    assert np.signbit(bias_logits(zn, _greedy_params())[0])


def test_typical_p_closed_form():
    # p = (0.4, 0.3, 0.3): H = -(0.4 ln 0.4 + 0.6 ln 0.3) = 1.0889; |-ln p - H| =
    # (0.1726, 0.1151, 0.1151): the two 0.3 ids are the most typical, so
    # typical_p 0.5 keeps ids 1 and 2 (mass 0.6) and leaves out the most likely id
    z = np.log(np.array([0.4, 0.3, 0.3])).astype(np.float32)
    tp = _greedy_params(typical_p=0.5)
    toks = [sample_row(z, [], s, tp)[0] for s in range(400)]
    assert set(toks) == {1, 2}
    assert 140 < toks.count(1) < 260          # ids 1 and 2 equally likely
    # typical_p 0.25: the single most typical id (id 1: ties go by candidate order)
    assert {sample_row(z, [], s, _greedy_params(typical_p=0.25))[0] for s in range(50)} == {1}
    # typical_p 1: no filter (the same draws as without it)
    for s in range(50):
        assert sample_row(z, [], s, _greedy_params(typical_p=1.0))[0] == sample_row(z, [], s, _greedy_params())[0]
    # min-p is relative to the largest kept probability: with ids 1 and 2 kept
    # (e = 0.75 each), min_p 0.9 keeps both (it would keep neither, so only
    # one, against the dropped id 0)
    both = {sample_row(z, [], s, _greedy_params(typical_p=0.5, min_p=0.9))[0] for s in range(100)}
    assert both == {1, 2}
    # top-p over the kept set: p = (0.5, 0.3, 0.2), typical_p 0.5 keeps ids 0 and 1
    # (|-ln p - H| = 0.337, 0.174, 0.580); top_p 0.6 of their mass (e 1 + 0.6)
    # keeps id 0 alone, where 0.6 of all three (e 2.0) would keep ids 0 and 1
    z2 = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)
    assert {sample_row(z2, [], s, _greedy_params(typical_p=0.5))[0] for s in range(200)} == {0, 1}
    assert {sample_row(z2, [], s, _greedy_params(typical_p=0.5, top_p=0.6))[0] for s in range(50)} == {0}
    assert {sample_row(z2, [], s, _greedy_params(top_p=0.6))[0] for s in range(200)} == {0, 1}


def _freq(z, p, n, hist=()):
    toks = [sample_row(z, list(hist), s, p)[0] for s in range(n)]
    return np.bincount(toks, minlength=len(z))


def test_frequencies_match_softmax_chi2():
    z = np.array([0.5, -1.0, 2.0, 0.0, 1.0, -0.5, 0.25, 1.5], np.float32)
    n = 40000
    p = _greedy_params(temperature=1.0)
    f = _freq(z, p, n)
    pr = np.exp(z.astype(np.float64) - z.max())
    pr /= pr.sum()
    assert stats.chisquare(f, pr * n).pvalue > 1e-4
    # temperature 0.5 and top-k 3: softmax(2z) over the three largest
    p = _greedy_params(temperature=0.5, top_k=3)
    f = _freq(z, p, n)
    top = [2, 7, 4]
    assert f.sum() == f[top].sum()
    pr = np.exp(2 * (z[top].astype(np.float64) - z.max()))
    pr /= pr.sum()
    assert stats.chisquare(f[top], pr * n).pvalue > 1e-4


def test_top_p_and_min_p_hand_built():
    # probabilities 0.5, 0.3, 0.15, 0.05 (ids 1, 3, 0, 2)
    pr = np.array([0.15, 0.5, 0.05, 0.3])
    z = np.log(pr).astype(np.float32)
    n = 20000
    f = _freq(z, _greedy_params(top_p=0.75), n)      # keeps 0.5 and 0.3 (0.8 >= 0.75)
    assert f[0] == 0 and f[2] == 0
    assert stats.chisquare(f[[1, 3]], np.array([5, 3]) / 8 * n).pvalue > 1e-4
    f = _freq(z, _greedy_params(min_p=0.2), n)       # keeps p >= 0.1: ids 1, 3, 0
    assert f[2] == 0
    assert stats.chisquare(f[[1, 3, 0]], np.array([0.5, 0.3, 0.15]) / 0.95 * n).pvalue > 1e-4


def test_draw_uses_request_step_not_slot():
    z = np.random.default_rng(3).standard_normal(500).astype(np.float32)
    p = SamplingParams()
    a = [sample_row(z, [], s, p)[0] for s in range(50)]
    b = [sample_row(z, [], s, p)[0] for s in range(50)]
    assert a == b
    u = [philox.sampler_uniform(42, s) for s in range(3)]
    assert len(set(u)) == 3 and all(0 <= x < 1 for x in u)
