"""Pins for the decoder-layer oracle: reductions to identities, closed forms
of one-hot layers with distinct non-unit norm gains, and the agreement of
decode and prefill restatements."""
import math

import numpy as np

from invariant_deterministic_gb300 import synth
from oracle import bf16
from oracle.model import Shape, layer_step, prefill_chunk

TINY = Shape(d_model=256, n_q=4, n_kv=2, head_dim=64, ffn=512, eps=1e-6, rope_base=1e4)


def _weights(seed=0):
    w = synth.layer_weights(256, 4, 2, 64, 512, seed, qk_norm=False)
    return {k: synth.bits(v) for k, v in w.items()}


def test_zero_output_projections_leave_the_residual_stream():
    lw = _weights()
    lw["w_o"] = np.zeros_like(lw["w_o"])
    lw["w_down"] = np.zeros_like(lw["w_down"])
    x = synth.bits(synth.normal_bf16((3, 256), 1.0, 1))
    kc = np.zeros((3, 8, 2, 64), np.uint16)
    vc = np.zeros_like(kc)
    out = layer_step(x, lw, kc, vc, [(0, 0), (1, 3), (2, 7)], TINY)
    assert np.array_equal(out, x)
    assert np.any(kc[1, 3] != 0) and np.all(kc[1, :3] == 0)   # only the new position is written


def test_decode_sequence_matches_whole_prefill():
    lw = _weights(1)
    t_len = 9
    x = synth.bits(synth.normal_bf16((t_len, 256), 1.0, 2))
    kc1 = np.zeros((1, 16, 2, 64), np.uint16)
    vc1 = np.zeros_like(kc1)
    whole = prefill_chunk(x, lw, kc1, vc1, 0, 0, TINY)
    kc2 = np.zeros_like(kc1)
    vc2 = np.zeros_like(kc1)
    rows = [layer_step(x[t: t + 1], lw, kc2, vc2, [(0, t)], TINY)[0] for t in range(t_len)]
    got = bf16.to_f64(np.stack(rows))
    ref = bf16.to_f64(whole)
    # fp64 BLAS may sum a matrix product and a vector product in different
    # orders; after bf16 rounding the two agree to one bf16 step at most.
    assert np.allclose(got, ref, rtol=2 ** -7, atol=1e-6)
    assert np.mean(got == ref) > 0.99


QK = Shape(d_model=256, n_q=4, n_kv=2, head_dim=64, ffn=512, eps=1e-6, rope_base=1e4, qk_norm=True)


def _one_hot_layer(attn_gain, ffn_gain):
    """A layer whose weights are all zero but for the entries each test sets,
    with input-column-5 gains attn_gain (attention norm) and ffn_gain (FFN norm)
    and every other gain 1."""
    one = lambda n: np.full(n, 0x3F80, np.uint16)  # bf16 1.0
    lw = {"attn_norm": one(256), "ffn_norm": one(256), "q_norm": one(64), "k_norm": one(64),
          "w_qkv": np.zeros((512, 256), np.uint16), "w_o": np.zeros((256, 256), np.uint16),
          "w_gu": np.zeros((1024, 256), np.uint16), "w_down": np.zeros((256, 512), np.uint16)}
    lw["attn_norm"][5] = _b(attn_gain)
    lw["ffn_norm"][5] = _b(ffn_gain)
    return lw


def _b(v):
    """bf16 bits of a number (a scalar) or of an array."""
    a = np.asarray(v, dtype=np.float64)
    return bf16.from_f64(a.reshape(-1)).reshape(a.shape) if a.ndim else bf16.from_f64(a.reshape(1))[0]


def test_layer_attention_side_closed_form():
    """x = ones, so the attention norm gives h_5 = g_5 / sqrt(1 + eps).  W_qkv
    copies h_5 into element 0 of k head 0 (row 256) and of v head 0 (row 384).
    QK-norm of the one-hot k head (D = 64) gives 8 * k_norm[0] at element 0,
    then RoPE at position 3 rotates the pair (0, 32) by 3 radians.  The q gains
    differ (a swapped q/k norm shows), k_norm[32] differs from k_norm[0] (a
    rotation before the norm shows), the FFN gain differs (a swapped block
    norm shows)."""
    lw = _one_hot_layer(2.0, 0.25)
    lw["w_qkv"][256, 5] = _b(1.0)
    lw["w_qkv"][384, 5] = _b(1.0)
    lw["q_norm"][0] = _b(3.0)
    lw["k_norm"][0] = _b(2.0)
    lw["k_norm"][32] = _b(0.5)
    x = np.full((1, 256), 0x3F80, np.uint16)
    kc = np.zeros((1, 8, 2, 64), np.uint16)
    vc = np.zeros_like(kc)
    out = layer_step(x, lw, kc, vc, [(0, 3)], QK)
    eps = 1e-6
    h5 = 2.0 / math.sqrt(1.0 + eps)
    kn = h5 / math.sqrt(h5 * h5 / 64 + eps) * 2.0
    k_ref = np.zeros(64)
    k_ref[0], k_ref[32] = kn * math.cos(3.0), kn * math.sin(3.0)
    # values compared as numbers: a zero may carry either sign
    assert np.array_equal(bf16.to_f64(kc[0, 3, 0]), bf16.to_f64(_b(k_ref)))
    assert np.all(bf16.to_f64(kc[0, 3, 1]) == 0) and np.all(kc[0, :3] == 0)
    v_ref = np.zeros(64)
    v_ref[0] = h5
    assert np.array_equal(bf16.to_f64(vc[0, 3, 0]), bf16.to_f64(_b(v_ref)))
    # W_o = 0 and W_down = 0: the residual stream passes through
    assert np.array_equal(out, x)


def test_layer_ffn_side_closed_form():
    """W_qkv = W_o = 0, so x2 = x = ones and the FFN norm gives
    h_5 = g_5 / sqrt(1 + eps).  Gate row 7 and up row F + 7 read column 5
    (weights 1 and 0.5), so act_7 = bf16(silu(h_5) * h_5 / 2); W_down[11][7] = 1
    adds act_7 to x_11, the sum rounded once.  The attention norm's gain
    differs, so a swapped block norm shows, and the up weight differs from the
    gate weight, so swapped gate and up halves show."""
    lw = _one_hot_layer(0.25, 2.0)
    lw["w_gu"][7, 5] = _b(1.0)
    lw["w_gu"][512 + 7, 5] = _b(0.5)
    lw["w_down"][11, 7] = _b(1.0)
    x = np.full((2, 256), 0x3F80, np.uint16)
    kc = np.zeros((2, 8, 2, 64), np.uint16)
    vc = np.zeros_like(kc)
    out = layer_step(x, lw, kc, vc, [(0, 0), (1, 5)], QK)
    h = 2.0 / math.sqrt(1.0 + 1e-6)
    act = bf16.to_f64(_b(h / (1.0 + math.exp(-h)) * (0.5 * h)))
    ref = np.full((2, 256), 0x3F80, np.uint16)
    ref[:, 11] = _b(1.0 + act)
    assert np.array_equal(out, ref)


def test_fold_rounds_the_gained_weight_once_per_column():
    """fold(W, g) = bf16(W[n][k] * g[k]): a column gain, rounded to bf16.
    (1 + 2^-7)^2 = 1 + 2^-6 + 2^-14 lies below the midpoint to the next bf16
    value, so it rounds to 1 + 2^-6; powers of two scale exactly."""
    from oracle.model import fold
    w = np.array([[_b(1.0 + 2.0 ** -7), _b(3.0)], [_b(-0.5), _b(1.0)]], np.uint16)
    g = np.array([_b(1.0 + 2.0 ** -7), _b(0.25)], np.uint16)
    got = bf16.to_f64(fold(w, g))
    assert np.array_equal(got, [[1.0 + 2.0 ** -6, 0.75], [-0.5 * (1.0 + 2.0 ** -7), 0.25]])
