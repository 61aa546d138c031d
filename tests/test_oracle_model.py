"""Pins for the decoder-layer oracle: reductions to identities and the
agreement of decode and prefill restatements."""
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
