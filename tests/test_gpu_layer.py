"""The small decoder layer (d_model 256, 4 query / 2 kv heads of 64, SwiGLU
512, RMSNorm eps 1e-6, RoPE base 1e4, weights ~N(0, 0.02), hidden states and
KV cache ~N(0, 1)): decode one token for batch sizes 1-4 over KV lengths
1-64; every row matches the oracle and its bits do not depend on the batch
size or on its batch-mates."""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth
from oracle import bf16 as obf
from oracle.model import Shape, layer_step

pytestmark = gpu
LMAX = 64
N_REQ = 4


@pytest.fixture(scope="module")
def setup():
    ensure_lib()
    from invariant_deterministic_gb300 import model as M
    shape = M.TINY
    w = M.random_weights(shape, seed=0, device="cuda", with_head=False)
    dec = M.Decoder(shape, w, max_batch=N_REQ, max_len=LMAX)
    # request r: hidden state and a full cache of N(0,1) values
    xs = [synth.normal_bf16((shape.d_model,), 1.0, 100 + r) for r in range(N_REQ)]
    caches = [synth.normal_bf16((2, LMAX, shape.n_kv, shape.head_dim), 1.0, 200 + r) for r in range(N_REQ)]
    oshape = Shape(d_model=256, n_q=4, n_kv=2, head_dim=64, ffn=512, eps=1e-6, rope_base=1e4)
    ow = {k: synth.bits(v) for k, v in w["layers"][0].items()}
    return dec, xs, caches, oshape, ow


def _length(r, L):
    # batch-mates get other lengths; the attention of request r sees this many keys
    return ((L - 1 + 17 * r) % LMAX) + 1


def _run(dec, xs, caches, reqs, L):
    """Decode one token for the listed requests (slot i <- request reqs[i])."""
    bsz = len(reqs)
    for i, r in enumerate(reqs):
        dec.x[i].copy_(xs[r])
        dec.kv[0, :, i].copy_(caches[r])
    dec.set_positions([_length(r, L) - 1 for r in reqs])
    dec.decode_layers(bsz)
    out = dec.close_residual(bsz).clone()
    kv_new = torch.stack([dec.kv[0, :, i, _length(r, L) - 1].clone() for i, r in enumerate(reqs)])
    return out, kv_new


def test_tiny_layer_sweep(setup):
    dec, xs, caches, oshape, ow = setup
    for L in range(1, LMAX + 1):
        full, kv_full = _run(dec, xs, caches, list(range(N_REQ)), L)
        # oracle for every request at batch 4
        x_bits = np.stack([synth.bits(x) for x in xs])
        kc = np.stack([synth.bits(c[0]) for c in caches])
        vc = np.stack([synth.bits(c[1]) for c in caches])
        pos = [(r, _length(r, L) - 1) for r in range(N_REQ)]
        ref = layer_step(x_bits, ow, kc, vc, pos, oshape)
        assert_close(f64(full), obf.to_f64(ref), f"L={L}")
        for r in range(N_REQ):
            p = _length(r, L) - 1
            assert_close(f64(kv_full[r, 0]), obf.to_f64(kc[r, p]), f"L={L} appended k")
        # batch sizes 1..3 and other orders: identical row bits
        for reqs in ([0], [1], [0, 1], [2, 0, 1], [3, 2], [1, 3, 0]):
            got, kv_got = _run(dec, xs, caches, reqs, L)
            for i, r in enumerate(reqs):
                assert_same_bits(got[i], full[r], f"L={L} request {r} in {reqs}")
                assert_same_bits(kv_got[i], kv_full[r], f"L={L} request {r} kv in {reqs}")
