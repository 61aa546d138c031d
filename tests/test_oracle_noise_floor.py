"""The rounding noise floor of a multi-layer comparison (CPU only).

The oracle computes every product in fp64 and rounds to bf16 where the GPU
path stores a tensor.  An implementation that accumulates in fp32 (as the
GPU's tensor cores do) rounds the same tensors, but a value that lies within
fp32 accumulation error of a bf16 rounding boundary rounds the other way;
the next layer takes the one-unit difference as input and it compounds.  This
test restates the oracle with fp32-accumulated matrix products (NumPy float32
matmul, everything else unchanged) and measures how far two 8B-shaped layers
drift from the fp64 oracle: some elements of the final residual rows leave
the per-element bound |g - r| <= 2e-2 + 1e-2 |r| although no kernel is
involved, while the norm-relative error stays far below 1e-2.  That spread is
why the two-layer GPU comparison checks shares and norms, and each kernel is
held to the per-element bound on its own inputs."""
import numpy as np
import pytest

from invariant_deterministic_gb300 import synth
from oracle import bf16, glue
import oracle.model as om


def _f32_gemm(a_bits, w_bits, out="bf16"):
    return _f32_matmul(bf16.to_f64(a_bits), w_bits, out)


def _f32_matmul(a, w_bits, out="bf16"):
    c = (np.asarray(a, np.float32) @ bf16.to_f64(w_bits).astype(np.float32).T).astype(np.float64)
    return {"bf16": bf16.from_f64, "f32": lambda v: v.astype(np.float32), "f64": lambda v: v}[out](c)


def _two_layers(lw_list, kv, x, lengths, shape):
    for li, lw in enumerate(lw_list):
        x = om.layer_step(x, lw, kv[li][0].copy(), kv[li][1].copy(),
                          [(b, lengths[b]) for b in range(len(lengths))], shape)
    return bf16.to_f64(x)


def test_fp32_accumulation_drifts_past_the_per_element_bound_over_two_layers(monkeypatch):
    shape = om.Shape(d_model=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, n_layers=2, eps=1e-6,
                     rope_base=1e6, qk_norm=True)
    lws = [{k: synth.bits(v) for k, v in synth.layer_weights(4096, 32, 8, 128, 12288, li, True).items()}
           for li in range(2)]
    lengths = [16, 300]
    kv = []
    for li in range(2):
        kc = np.zeros((2, 320, 8, 128), np.uint16)
        vc = np.zeros_like(kc)
        for r, n in enumerate(lengths):
            kc[r, :n] = synth.bits(synth.normal_bf16((n, 8, 128), 1.0, 7000 + 10 * li + r))
            vc[r, :n] = synth.bits(synth.normal_bf16((n, 8, 128), 1.0, 7100 + 10 * li + r))
        kv.append((kc, vc))
    x0 = synth.bits(synth.normal_bf16((2, 4096), 0.02, 7200))
    ref = _two_layers(lws, kv, x0, lengths, shape)
    monkeypatch.setattr(om, "gemm", _f32_gemm)
    monkeypatch.setattr(om, "matmul", _f32_matmul)
    got = _two_layers(lws, kv, x0, lengths, shape)
    outside = np.abs(got - ref) > 2e-2 + 1e-2 * np.abs(ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    print(f"fp32 restatement vs fp64 oracle, two layers: {outside.sum()} of {outside.size} elements "
          f"outside the per-element bound, norm-relative error {rel:.2e}")
    assert outside.any()          # the spread exists without any GPU kernel
    assert outside.mean() <= 0.03
    assert rel <= 1e-2
