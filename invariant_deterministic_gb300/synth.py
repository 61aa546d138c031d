"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it only draws numbers.  Every
draw goes through a seeded ``torch.Generator`` so that the GPU path and the
oracle receive the same bits.  Distributions follow the workloads: weights
~N(0, 0.02) in bf16, activations and KV caches ~N(0, 1) in bf16, RMSNorm gains
equal to 1, KV lengths and prompt lengths uniform over stated integer ranges.

Seeds: weights 0, activations / caches 1, lengths and prompts 2, request seeds
1000 + request index (callers may pass others).
"""
from __future__ import annotations

import numpy as np
import torch

SEED_WEIGHTS = 0
SEED_ACT = 1
SEED_LEN = 2
SEED_REQ_BASE = 1000


def gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """~N(0, std) rounded to bf16 (drawn in fp32 on ``device``)."""
    g = gen(seed, device)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def int_bf16(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integers uniform in [lo, hi] as bf16 (exact for |v| <= 256)."""
    g = gen(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


def uniform_int(n: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """n integers uniform in [lo, hi] (int32)."""
    g = gen(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a copy on the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor on the host."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def layer_weights(d: int, n_q: int, n_kv: int, head_dim: int, ffn: int, seed: int,
                  qk_norm: bool, device="cpu") -> dict:
    """One decoder layer: projections ~N(0, 0.02); gains = 1.

    Layout: w_qkv [(n_q + 2 n_kv) head_dim][d] (q rows, then k, then v);
    w_o [d][n_q head_dim]; w_gu [2 ffn][d] (gate rows, then up rows);
    w_down [d][ffn]."""
    one = lambda n: torch.ones(n, dtype=torch.bfloat16, device=device)
    w = {
        "attn_norm": one(d),
        "w_qkv": normal_bf16(((n_q + 2 * n_kv) * head_dim, d), 0.02, seed * 16 + 1, device),
        "w_o": normal_bf16((d, n_q * head_dim), 0.02, seed * 16 + 2, device),
        "ffn_norm": one(d),
        "w_gu": normal_bf16((2 * ffn, d), 0.02, seed * 16 + 3, device),
        "w_down": normal_bf16((d, ffn), 0.02, seed * 16 + 4, device),
    }
    if qk_norm:
        w["q_norm"] = one(head_dim)
        w["k_norm"] = one(head_dim)
    return w


# kinv_sampling_params and kinv_logit_bias, field by field
SAMPLING_DTYPE = np.dtype([("temperature", "<f4"), ("top_p", "<f4"), ("min_p", "<f4"),
                           ("repeat_penalty", "<f4"), ("top_k", "<i4"), ("repeat_last_n", "<i4"),
                           ("seed", "<u8"), ("presence_penalty", "<f4"), ("frequency_penalty", "<f4"),
                           ("logit_bias", "<u8"), ("n_logit_bias", "<i4"), ("typical_p", "<f4")])
BIAS_DTYPE = np.dtype([("id", "<i4"), ("bias", "<f4")])


def bias_entries(params_list):
    """The rows' logit-bias lists back to back (kinv_logit_bias entries, in
    each dict's insertion order) and the index of each row's first entry."""
    rows, starts = [], []
    for p in params_list:
        starts.append(len(rows))
        rows.extend((int(t), float(v)) for t, v in (getattr(p, "logit_bias", None) or {}).items())
    return np.array(rows, dtype=BIAS_DTYPE), starts


def sampling_struct(params_list, bias_base: int = 0) -> np.ndarray:
    """Pack per-request sampler settings into the C struct layout
    (SAMPLING_DTYPE, 56 bytes).  bias_base: device address of the entries of
    bias_entries(params_list), which row i's logit_bias points into."""
    _, starts = bias_entries(params_list)
    a = np.zeros(len(params_list), dtype=SAMPLING_DTYPE)
    for i, p in enumerate(params_list):
        nb = len(getattr(p, "logit_bias", None) or {})
        if nb and not bias_base:
            raise ValueError("a logit-bias list needs bias_base (the entries' device address)")
        a[i] = (p.temperature, p.top_p, p.min_p, p.repeat_penalty, p.top_k, p.repeat_last_n, p.seed,
                getattr(p, "presence_penalty", 0.0), getattr(p, "frequency_penalty", 0.0),
                bias_base + BIAS_DTYPE.itemsize * starts[i] if nb else 0, nb,
                getattr(p, "typical_p", 1.0))
    return a
