"""Pins for the oracle's bf16 conversion, GEMM, RMSNorm, RoPE and glue.

Each check compares the oracle with something other than itself: exact integer
arithmetic, closed forms, library routines, invariants of the definition."""
import math

import numpy as np
import pytest
import torch

from oracle import bf16, glue
from oracle.gemm import gemm, matmul
from oracle.rmsnorm import rmsnorm
from oracle.rope import rope


def _bits_from_f32(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- bf16
def test_bf16_matches_torch_rne_on_fp32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-40, 40, 200000))).astype(np.float32)
    assert np.array_equal(bf16.from_f64(x.astype(np.float64)), _bits_from_f32(x))


def test_bf16_ties_to_even_and_specials():
    one = 1.0
    assert bf16.from_f64(one) == 0x3F80
    assert bf16.from_f64(one + 2.0 ** -8) == 0x3F80          # tie -> even (down)
    assert bf16.from_f64(one + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (up)
    assert bf16.from_f64(one + 2.0 ** -8 + 2.0 ** -40) == 0x3F81  # just above the tie
    assert bf16.from_f64(-2.0) == 0xC000
    assert bf16.from_f64(np.inf) == 0x7F80
    assert bf16.from_f64(1e39) == 0x7F80                      # overflow -> inf
    assert bf16.from_f64(np.nan) == 0x7FC0
    assert bf16.to_f64(np.uint16(0x3F80)) == 1.0
    assert bf16.to_f64(np.uint16(0x0001)) == 2.0 ** -133      # smallest subnormal
    assert bf16.from_f64(2.0 ** -133 * 1.5) == 0x0002         # subnormal tie -> even


# ---------------------------------------------------------------- GEMM
def test_gemm_integer_exact_against_python_ints():
    rng = np.random.default_rng(1)
    m, n, k = 5, 7, 64
    a = rng.integers(-8, 9, (m, k))
    w = rng.integers(-8, 9, (n, k))
    exact = [[sum(int(a[i, t]) * int(w[j, t]) for t in range(k)) for j in range(n)] for i in range(m)]
    got = gemm(_bits_from_f32(a), _bits_from_f32(w), out="f32")
    assert np.array_equal(got, np.array(exact, dtype=np.float32))
    got_bf = gemm(_bits_from_f32(a), _bits_from_f32(w), out="bf16")
    assert np.array_equal(got_bf, _bits_from_f32(np.array(exact, dtype=np.float32)))


def test_gemm_identity_and_orientation():
    rng = np.random.default_rng(2)
    a = _bits_from_f32(rng.standard_normal((3, 16)))
    eye = _bits_from_f32(np.eye(16))
    assert np.array_equal(gemm(a, eye), a)
    # C[i, j] must be row i of A against ROW j of W (W is [N][K])
    w = np.zeros((2, 16), np.float32)
    w[1, 3] = 1.0
    c = gemm(a, _bits_from_f32(w), out="f64")
    assert np.array_equal(c[:, 1], bf16.to_f64(a)[:, 3]) and np.all(c[:, 0] == 0)


def test_gemm_matches_numpy_matmul_float32_library():
    rng = np.random.default_rng(3)
    a = _bits_from_f32(rng.standard_normal((9, 128)))
    w = _bits_from_f32(rng.standard_normal((33, 128)) * 0.02)
    ref = torch.from_numpy(bf16.to_f64(a)) @ torch.from_numpy(bf16.to_f64(w)).T
    assert np.allclose(gemm(a, w, out="f64"), ref.numpy(), rtol=0, atol=1e-12)


def test_matmul_of_unrounded_rows():
    """An fp64 left operand is used as is: times W = I it comes back rounded
    once to bf16 (1/3 is not a bf16 value), and integer rows multiply exactly."""
    a = np.array([[1.0 / 3.0, -2.5, 1e-3, 7.0]])
    eye = _bits_from_f32(np.eye(4))
    assert np.array_equal(matmul(a, eye, out="f64"), a)
    assert np.array_equal(matmul(a, eye), bf16.from_f64(a))
    assert matmul(a, eye, out="f64")[0, 0] != bf16.to_f64(bf16.from_f64(a))[0, 0]
    rng = np.random.default_rng(4)
    ai = rng.integers(-8, 9, (3, 32)).astype(np.float64)
    w = rng.integers(-8, 9, (5, 32))
    exact = [[sum(int(ai[i, t]) * int(w[j, t]) for t in range(32)) for j in range(5)] for i in range(3)]
    assert np.array_equal(matmul(ai, _bits_from_f32(w), out="f64"), np.array(exact, dtype=np.float64))


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_forms():
    d, eps = 64, 1e-6
    w = _bits_from_f32(np.linspace(0.5, 1.5, d))
    wf = bf16.to_f64(w)
    c = 3.0
    y = bf16.to_f64(rmsnorm(_bits_from_f32(np.full((1, d), c)), w, eps))[0]
    assert np.array_equal(y, bf16.round_f64(c / math.sqrt(c * c + eps) * wf))
    x = np.zeros((1, d))
    x[0, 5] = c
    y = bf16.to_f64(rmsnorm(_bits_from_f32(x), w, eps))[0]
    expect = np.zeros(d)
    expect[5] = c / math.sqrt(c * c / d + eps) * wf[5]
    assert np.array_equal(y, bf16.round_f64(expect))
    assert np.all(bf16.to_f64(rmsnorm(_bits_from_f32(np.zeros((1, d))), w, eps)) == 0)


def test_rmsnorm_against_loop_and_scale_invariance():
    rng = np.random.default_rng(4)
    d = 96
    x = _bits_from_f32(rng.standard_normal((3, d)))
    w = _bits_from_f32(rng.uniform(0.5, 2, d))
    xf, wf = bf16.to_f64(x), bf16.to_f64(w)
    got = bf16.to_f64(rmsnorm(x, w, 1e-6))
    for r in range(3):
        ss = 0.0
        for v in xf[r]:
            ss += v * v
        inv = 1.0 / math.sqrt(ss / d + 1e-6)
        ref = [bf16.round_f64(xf[r, i] * inv * wf[i]) for i in range(d)]
        assert np.array_equal(got[r], np.array(ref).ravel())
    y2 = bf16.to_f64(rmsnorm(_bits_from_f32(xf * 4.0), w, 1e-6))   # power-of-two scale is exact
    assert np.allclose(y2, got, atol=0, rtol=2 ** -7)


def test_rmsnorm_residual_fusion():
    rng = np.random.default_rng(5)
    x = _bits_from_f32(rng.standard_normal((2, 32)))
    r = _bits_from_f32(rng.standard_normal((2, 32)))
    w = _bits_from_f32(np.ones(32))
    y, s = rmsnorm(x, w, 1e-6, residual_bits=r)
    assert np.array_equal(s, bf16.from_f64(bf16.to_f64(x) + bf16.to_f64(r)))
    assert np.array_equal(y, rmsnorm(s, w, 1e-6))


# ---------------------------------------------------------------- RoPE
def test_rope_closed_form_small():
    # D = 4, base 1e4: theta_0 = p, theta_1 = p / 100; pairs (0, 2) and (1, 3)
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    got = bf16.to_f64(rope(_bits_from_f32(x), [3], 1e4))[0, 0]
    assert np.array_equal(got, bf16.round_f64(np.array([math.cos(3), 0, math.sin(3), 0])))
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    got = bf16.to_f64(rope(_bits_from_f32(x), [3], 1e4))[0, 0]
    assert np.array_equal(got, bf16.round_f64(np.array([0, math.cos(0.03), 0, math.sin(0.03)])))
    x = np.array([[[0.0, 0.0, 1.0, 0.0]]])
    got = bf16.to_f64(rope(_bits_from_f32(x), [3], 1e4))[0, 0]
    assert np.array_equal(got, bf16.round_f64(np.array([-math.sin(3), 0, math.cos(3), 0])))


def test_rope_qk_norm_closed_form_norm_before_rotation():
    # QK-norm then RoPE, D = 4, base 1e4, position 3, gains g = (2, 3, 0.5, 5):
    # a one-hot head a.e0 has mean square a^2 / 4, so the normalised head is
    # 2 sign(a) e0 (up to eps), times g0; the pair (0, 2) then rotates by 3.
    # Rotating first would give g2 (not g0) on element 2.
    g = _bits_from_f32(np.array([2.0, 3.0, 0.5, 5.0]))
    eps = 1e-6
    for a in (1.5, -0.75):
        x = _bits_from_f32(np.array([[[a, 0.0, 0.0, 0.0]]]))
        got = bf16.to_f64(rope(x, [3], 1e4, norm_w_bits=g, eps=eps))[0, 0]
        n = a / math.sqrt(a * a / 4 + eps) * 2.0
        assert np.array_equal(got, bf16.round_f64(np.array([n * math.cos(3), 0.0, n * math.sin(3), 0.0])))
    # a constant head c.(1, 1, 1, 1) normalises to sign(c) (up to eps) before the gains
    x = _bits_from_f32(np.array([[[4.0, 4.0, 4.0, 4.0]]]))
    got = bf16.to_f64(rope(x, [3], 1e4, norm_w_bits=g, eps=eps))[0, 0]
    u = 4.0 / math.sqrt(16.0 + eps)
    t0, t1 = 3.0, 3.0 / 100.0
    ref = [u * 2.0 * math.cos(t0) - u * 0.5 * math.sin(t0), u * 3.0 * math.cos(t1) - u * 5.0 * math.sin(t1),
           u * 0.5 * math.cos(t0) + u * 2.0 * math.sin(t0), u * 5.0 * math.cos(t1) + u * 3.0 * math.sin(t1)]
    assert np.array_equal(got, bf16.round_f64(np.array(ref)))


def test_rope_identity_norm_and_relative_position():
    from oracle.rope import rope_f64
    rng = np.random.default_rng(6)
    x = _bits_from_f32(rng.standard_normal((1, 2, 64)))
    assert np.array_equal(rope(x, [0], 1e4), x)
    xf = bf16.to_f64(x)
    y = rope_f64(xf, np.array([777]), 1e4)
    pn = lambda v: v[..., :32] ** 2 + v[..., 32:] ** 2
    assert np.allclose(pn(y), pn(xf), rtol=1e-12)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    d1 = np.sum(rope_f64(q, np.array([50]), 1e4) * rope_f64(k, np.array([20]), 1e4))
    d2 = np.sum(rope_f64(q, np.array([1030]), 1e4) * rope_f64(k, np.array([1000]), 1e4))
    assert abs(d1 - d2) < 1e-9


# ---------------------------------------------------------------- glue
def test_swiglu_and_add_closed_forms():
    g = np.array([0.0, 1.0, -2.0, 10.0])
    u = np.array([5.0, 2.0, 1.0, -1.0])
    gu = _bits_from_f32(np.concatenate([g, u])[None, :])
    got = bf16.to_f64(glue.swiglu(gu))[0]
    ref = [0.0, 2.0 / (1 + math.exp(-1)), -2.0 / (1 + math.exp(2)), -10.0 / (1 + math.exp(-10))]
    assert np.array_equal(got, bf16.round_f64(np.array(ref)))
    a, b = _bits_from_f32([[1.0, 256.0]]), _bits_from_f32([[2.0 ** -8, 1.0]])
    # 1 + 2^-8 ties to 1 (even); 256 + 1 = 257 rounds to 256 (8 significant bits, tie to even)
    assert np.array_equal(bf16.to_f64(glue.add(a, b)), [[1.0, 256.0]])
    # an unrounded addend is rounded once with the sum: 1 + (2^-8 + 2^-20) lies
    # above the tie and rounds up, where rounding the addend first (to 2^-8)
    # would tie back to 1
    got = bf16.to_f64(glue.add_f64(_bits_from_f32([[1.0, 1.0]]), np.array([[2.0 ** -8 + 2.0 ** -20, -0.5]])))
    assert np.array_equal(got, [[1.0 + 2.0 ** -7, 0.5]])
    tab = _bits_from_f32(np.arange(12.0).reshape(4, 3))
    assert np.array_equal(glue.embed(tab, [2, 0]), tab[[2, 0]])
