"""The pre-norm decoder layer and the decode / prefill step (test
infrastructure only).

The pages name the three batch-invariant kernels (RMSNorm, matmul, attention,
"Deterministic and bit-exact inference", *technical*) and the sampler settings
(Kinetic "Receipts", *Making a receipt*) but not the block they sit in.  The
plainest reading is the standard pre-norm decoder block of Llama/Qwen-style
models, which is what the workloads describe (RMSNorm eps 1e-6, RoPE, SwiGLU
FFN, grouped-query attention):

    h  = RMSNorm(x) ; [q k v] = h . Wqkv^T
    q, k = RoPE(QKnorm(q)), RoPE(QKnorm(k))   (QK-norm optional)
    cache[pos] <- k, v ; a = Attention(q, cache)
    x2 = x + a . Wo^T ; h2 = RMSNorm(x2)
    [g u] = h2 . Wgu^T ; x3 = x2 + (silu(g) * u) . Wdown^T

bf16 rounding happens at each stored tensor, the same boundaries as the GPU
path.  The GPU path stores neither g and u (the gate/up product and SwiGLU are
one step), nor the O and down products (each is added into the residual
stream x in the projection that forms it, so x2 = bf16(x + o) is rounded
once), nor the normalised rows h, h2 and the final one: each RMSNorm is
folded into the projection it feeds, (x / rms(x) * w) . W^T computed as
(x . (W * w)^T) / rms(x), so here those rows stay unrounded fp64 and the gain
sits in the stored weight bf16(W * w) (``fold``), rounded like every stored
tensor.  Weights are
bf16 bit arrays; the dictionaries below name them.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import attention, bf16, glue
from .gemm import gemm, matmul
from .rmsnorm import rmsnorm, rmsnorm_f64
from .rope import rope
from .sampler import sample


@dataclass
class Shape:
    d_model: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int = 0
    n_layers: int = 1
    eps: float = 1e-6
    rope_base: float = 1e4
    qk_norm: bool = False


def fold(w_bits, g_bits):
    """bf16(W[n][k] * g[k]): an RMSNorm gain moved into the input columns of
    the projection it feeds.  The folded weight is what the step stores and
    reads, so it is rounded to bf16 like every stored tensor."""
    if np.all(np.asarray(g_bits) == 0x3F80):  # every gain 1.0: W itself, exactly
        return w_bits
    return bf16.from_f64(bf16.to_f64(w_bits) * bf16.to_f64(g_bits)[None, :])


def _unit(d):
    return np.ones(d, dtype=np.float64)


def layer_step(x_bits, lw: dict, k_cache, v_cache, pos, shape: Shape):
    """One decoder layer for rows x [M][d].  Row m belongs to sequence seq[m]
    at absolute position pos[m]; ``k_cache``/``v_cache`` are
    [B][Lmax][Hkv][D] bf16 arrays updated in place.  ``pos`` is a list of
    (seq, position) pairs in row order; rows of one sequence must be in
    ascending position order, and attention for a row sees keys 0..position.
    """
    hq, hk, dh = shape.n_q, shape.n_kv, shape.head_dim
    m = x_bits.shape[0]
    d = x_bits.shape[1]
    h = rmsnorm_f64(bf16.to_f64(x_bits), _unit(d), shape.eps)
    qkv = matmul(h, fold(lw["w_qkv"], lw["attn_norm"])).reshape(m, hq + 2 * hk, dh)
    positions = np.array([p for _, p in pos], dtype=np.int64)
    qn = lw.get("q_norm") if shape.qk_norm else None
    kn = lw.get("k_norm") if shape.qk_norm else None
    q = rope(qkv[:, :hq], positions, shape.rope_base, qn, shape.eps)
    k = rope(qkv[:, hq: hq + hk], positions, shape.rope_base, kn, shape.eps)
    v = qkv[:, hq + hk:]
    for i, (b, p) in enumerate(pos):
        k_cache[b, p] = k[i]
        v_cache[b, p] = v[i]
    a = np.zeros_like(q)
    for i, (b, p) in enumerate(pos):
        a[i] = attention.decode(q[i: i + 1], k_cache[b: b + 1], v_cache[b: b + 1], [p + 1])[0]
    # the O and down projections add into the residual stream: their outputs
    # are not stored, so each sum is rounded once
    x2 = glue.add_f64(x_bits, gemm(a.reshape(m, hq * dh), lw["w_o"], out="f64"))
    h2 = rmsnorm_f64(bf16.to_f64(x2), _unit(d), shape.eps)
    # gate/up and SwiGLU form one GPU kernel: g and u are not rounded to bf16
    act = glue.swiglu_f64(matmul(h2, fold(lw["w_gu"], lw["ffn_norm"]), out="f64"))
    return glue.add_f64(x2, gemm(act, lw["w_down"], out="f64"))


def final_logits(x_bits, model: dict, shape: Shape):
    """The final RMSNorm (its gain folded into the LM head) and the LM head:
    fp32 logits [M][V] of the residual rows x."""
    h = rmsnorm_f64(bf16.to_f64(x_bits), _unit(x_bits.shape[1]), shape.eps)
    return matmul(h, fold(model["lm_head"], model["final_norm"]), out="f32")


def decode_step(tokens, model: dict, k_caches, v_caches, lengths, shape: Shape,
                histories=None, steps=None, params=None, sample_tokens=True):
    """Full model, one new token per sequence b at position lengths[b].
    Returns (logits f32 [B][V], sampled ids or None, near-tie flags or None)."""
    x = glue.embed(model["embed"], tokens)
    pos = [(b, int(lengths[b])) for b in range(len(tokens))]
    for li, lw in enumerate(model["layers"]):
        x = layer_step(x, lw, k_caches[li], v_caches[li], pos, shape)
    logits = final_logits(x, model, shape)
    if not sample_tokens:
        return logits, None, None
    toks, ties = sample(logits, histories, steps, params)
    return logits, toks, ties


def prefill_chunk(x_bits, lw: dict, k_cache, v_cache, seq: int, p0: int, shape: Shape):
    """One layer over a chunk of T tokens of sequence ``seq`` at p0..p0+T-1."""
    pos = [(seq, p0 + t) for t in range(x_bits.shape[0])]
    return layer_step(x_bits, lw, k_cache, v_cache, pos, shape)
