"""kinv_gemm on the GPU: exactness, oracle parity and batch invariance."""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth
from oracle import bf16 as obf
from oracle import glue as oglue
from oracle.gemm import gemm as ogemm, gemm_f64_rows

pytestmark = gpu


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


def _int_bf16(shape, seed, lo=-8, hi=8):
    return synth.int_bf16(shape, lo, hi, seed).cuda()


@pytest.mark.parametrize("m,n,k", [(1, 64, 64), (7, 80, 256), (130, 128, 512), (300, 208, 1024),
                                   (5, 4096, 4096), (129, 6144, 4096), (3, 4096, 12288)])
def test_integer_inputs_are_exact(kinv, m, n, k):
    """Integer inputs in [-8, 8]: every partial sum is an integer below 2^24,
    so fp32 accumulation is exact in any order and the result must equal the
    exact product (fp32 out) or its bf16 rounding (bf16 out)."""
    a = _int_bf16((m, k), 1)
    w = _int_bf16((n, k), 2)
    exact = ogemm(synth.bits(a), synth.bits(w), out="f64")
    c32 = kinv.gemm(a, w, out_dtype=torch.float32)
    assert np.array_equal(f64(c32), exact)
    c16 = kinv.gemm(a, w)
    assert np.array_equal(synth.bits(c16), obf.from_f64(exact))
    assert kinv.last_device_status() == 0


def test_identity_weights_copy_rows(kinv):
    a = synth.normal_bf16((33, 256), 1.0, 3).cuda()
    eye = torch.eye(256, dtype=torch.bfloat16, device="cuda")
    assert_same_bits(kinv.gemm(a, eye), a, "A . I")


@pytest.mark.parametrize("m,n,k", [(1, 512, 256), (4, 256, 512), (37, 1024, 256), (200, 96, 640)])
def test_parity_random(kinv, m, n, k):
    a = synth.normal_bf16((m, k), 1.0, 4).cuda()
    w = synth.normal_bf16((n, k), 0.02, 5).cuda()
    got = kinv.gemm(a, w)
    ref = ogemm(synth.bits(a), synth.bits(w))
    assert_close(f64(got), obf.to_f64(ref), f"gemm {m}x{n}x{k}")
    got32 = kinv.gemm(a, w, out_dtype=torch.float32)
    assert_close(f64(got32), ogemm(synth.bits(a), synth.bits(w), out="f64"), "gemm f32 out")


# Qwen3-8B-shaped projections: (N, K)
SHAPES_8B = [(6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288)]
MS = [1, 7, 16, 64, 128, 256]


@pytest.mark.parametrize("n,k", SHAPES_8B)
def test_8b_shapes_row_bits_independent_of_m(kinv, n, k):
    """Row i's bits are the same for M in {1, 7, 16, 64, 128, 256, 512, 1024}
    (the cluster split-K schedule below a few hundred rows, the tile schedule
    above) and for any co-batched rows; every output of the M = 256 product
    matches the oracle."""
    w = synth.normal_bf16((n, k), 0.02, 6).cuda()
    a_big = synth.normal_bf16((1024, k), 1.0, 7).cuda()
    big = kinv.gemm(a_big, w)
    a = a_big[:256].contiguous()
    full = kinv.gemm(a, w)
    assert_same_bits(full, big[:256], f"N={n} K={k}: M=256 vs M=1024")
    for m in MS + [512]:
        part = kinv.gemm(a_big[:m].contiguous(), w)
        assert_same_bits(part, big[:m], f"N={n} K={k} M={m}")
    # the same rows among different batch-mates, at other positions
    other = synth.normal_bf16((256, k), 1.0, 8).cuda()
    perm = torch.randperm(256, generator=synth.gen(9))
    mixed = other.clone()
    mixed[perm[:64]] = a[:64]
    got = kinv.gemm(mixed, w)
    assert_same_bits(got[perm[:64]], full[:64], "rows among other batch-mates")
    # the oracle on every row and column of the M = 256 product
    ref = ogemm(synth.bits(a), synth.bits(w), out="f64")
    assert_close(f64(full), obf.round_f64(ref), f"oracle N={n} K={k}, all of M = 256")
    assert kinv.last_device_status() == 0


def test_lm_head_fp32_row_invariance(kinv):
    n, k = 151936, 4096
    w = synth.normal_bf16((n, k), 0.02, 11).cuda()
    a_big = synth.normal_bf16((300, k), 1.0, 12).cuda()
    big = kinv.gemm(a_big, w, out_dtype=torch.float32)   # the tile schedule
    a = a_big[:16].contiguous()
    full = kinv.gemm(a, w, out_dtype=torch.float32)      # the cluster schedule
    assert_same_bits(full, big[:16], "LM head: 16 rows vs 300 rows")
    one = kinv.gemm(a[3:4].contiguous(), w, out_dtype=torch.float32)
    assert_same_bits(one, full[3:4], "LM head row 3")
    cols = torch.randint(0, n, (128,), generator=synth.gen(13)).numpy()
    ref = gemm_f64_rows(synth.bits(a), synth.bits(w), [0, 3, 15], cols)
    assert_close(f64(full)[[0, 3, 15]][:, cols], ref, "LM head vs oracle", atol=1e-4, rtol=1e-4)


def test_prefill_sized_m(kinv):
    """M up to 4096 (prefill chunks) keeps the same row bits."""
    n, k = 4096, 4096
    w = synth.normal_bf16((n, k), 0.02, 14).cuda()
    a = synth.normal_bf16((4096, k), 1.0, 15).cuda()
    full = kinv.gemm(a, w)
    # (2000 rows: the tile schedule with two K blocks per stage and a ragged last tile)
    for m0, m in [(0, 1), (4095, 1), (512, 512), (1000, 64), (1000, 2000)]:
        part = kinv.gemm(a[m0: m0 + m].contiguous(), w)
        assert_same_bits(part, full[m0: m0 + m], f"rows {m0}..{m0 + m}")


def test_errors_before_launch(kinv):
    a = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kinv.KinvError) as e:
        kinv.gemm(a, w)
    assert e.value.status == kinv.ERR_UNSUPPORTED
    a = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(24, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kinv.KinvError):
        kinv.gemm(a, w)
    m0 = kinv.gemm(torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"),
                   torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda"))
    assert m0.shape == (0, 64)


# ---------------------------------------------------------------- fused gate/up + SwiGLU
def _swiglu_ref(a, w_gu):
    """bf16(silu(g) * u) from unrounded fp64 g = a . Wgate^T, u = a . Wup^T."""
    return oglue.swiglu_f64(ogemm(synth.bits(a), synth.bits(w_gu), out="f64"))


@pytest.mark.parametrize("m,f,k", [(1, 64, 64), (5, 192, 256), (130, 320, 512), (33, 1024, 1024)])
def test_gemm_swiglu_parity(kinv, m, f, k):
    a = synth.normal_bf16((m, k), 1.0, 21).cuda()
    w_gu = synth.normal_bf16((2 * f, k), 0.05, 22).cuda()
    got = kinv.gemm_swiglu(a, kinv.interleave_gate_up(w_gu))
    assert got.shape == (m, f)
    assert_close(f64(got), obf.to_f64(_swiglu_ref(a, w_gu)), f"gemm_swiglu {m}x{f}x{k}")
    assert kinv.last_device_status() == 0


def test_gemm_swiglu_interleave_layout(kinv):
    """Gate rows and up rows are told apart: swapping them changes the result
    to silu(u) * g, which the oracle computes from the swapped weights."""
    m, f, k = 9, 64, 128
    a = synth.normal_bf16((m, k), 1.0, 23).cuda()
    w_gu = synth.normal_bf16((2 * f, k), 0.1, 24).cuda()
    swapped = torch.cat([w_gu[f:], w_gu[:f]])
    got = kinv.gemm_swiglu(a, kinv.interleave_gate_up(swapped))
    assert_close(f64(got), obf.to_f64(_swiglu_ref(a, swapped)), "swapped gate/up")
    direct = kinv.gemm_swiglu(a, kinv.interleave_gate_up(w_gu))
    assert not torch.equal(got, direct)


def test_gemm_swiglu_8b_row_bits_independent_of_m(kinv):
    """Qwen3-8B FFN (F=12288, K=4096): row bits do not depend on M or on the
    batch-mates, and sampled features match the oracle."""
    f, k = 12288, 4096
    w_gu = synth.normal_bf16((2 * f, k), 0.02, 25).cuda()
    w_il = kinv.interleave_gate_up(w_gu)
    a = synth.normal_bf16((256, k), 1.0, 26).cuda()
    full = kinv.gemm_swiglu(a, w_il)
    for m in MS:
        assert_same_bits(kinv.gemm_swiglu(a[:m].contiguous(), w_il), full[:m], f"swiglu M={m}")
    other = synth.normal_bf16((256, k), 1.0, 27).cuda()
    perm = torch.randperm(256, generator=synth.gen(28))
    mixed = other.clone()
    mixed[perm[:32]] = a[:32]
    assert_same_bits(kinv.gemm_swiglu(mixed, w_il)[perm[:32]], full[:32], "swiglu batch-mates")
    rows = [0, 5, 15, 127, 255]
    cols = torch.randint(0, f, (48,), generator=synth.gen(29)).numpy()
    gu = gemm_f64_rows(synth.bits(a), synth.bits(w_gu), rows, np.concatenate([cols, cols + f]))
    ref = oglue.swiglu_f64(gu)
    assert_close(f64(full)[rows][:, cols], obf.to_f64(ref), "swiglu 8B vs oracle")
    assert kinv.last_device_status() == 0


def test_gemm_swiglu_rejects_bad_f(kinv):
    a = torch.zeros(2, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(2 * 96, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kinv.KinvError):
        kinv.gemm_swiglu(a, w)


# ---------------------------------------------------------------- folded RMSNorm epilogues
@pytest.mark.parametrize("m", [64, 256, 1024])
def test_fused_epilogues_match_the_oracle_on_whole_rows(kinv, m):
    """The epilogues of kinv_gemm_fused / kinv_gemm_swiglu at 64 and 256 rows
    (the owners of split-K rows pull the partials) and at 1024 rows (the tile
    schedule: one block folds every K range of a tile), against the oracle on
    every element: the row scale 1/rms from per-tile sums of squares (QKV,
    gate/up), the residual add with the new rows' sums of squares (O, down).
    The same rows computed in a 4-row call (partials pushed to their owners)
    have the same bits."""
    from oracle.gemm import matmul
    from oracle.rmsnorm import rmsnorm_f64
    d, f = 4096, 12288
    b = synth.bits
    w_qkv = synth.normal_bf16((6144, d), 0.02, 81).cuda()
    w_o = synth.normal_bf16((d, d), 0.02, 82).cuda()
    w_gu = synth.normal_bf16((2 * f, d), 0.02, 83).cuda()
    w_down = synth.normal_bf16((d, f), 0.02, 84).cuda()
    w_il = kinv.interleave_gate_up(w_gu)
    x = synth.normal_bf16((m, d), 1.0, 85).cuda()
    attn = synth.normal_bf16((m, d), 1.0, 86).cuda()
    ss = torch.empty(m, d // 128, dtype=torch.float32, device="cuda")
    kinv.row_sumsq(x, ss)

    def check_ss(xb, ss_t, what):
        v = obf.to_f64(xb)
        assert np.allclose(ss_t.cpu().numpy(), (v * v).reshape(m, -1, 128).sum(-1), rtol=1e-5, atol=0), what

    check_ss(b(x), ss, "sums of squares of x")
    normed = lambda xb: rmsnorm_f64(obf.to_f64(xb), np.ones(d), 1e-6)
    qkv = kinv.gemm_fused(x, w_qkv, kinv.norm_in(ss, d, 1e-6), out=torch.empty(m, 6144, dtype=torch.bfloat16, device="cuda"))
    assert_close(f64(qkv), obf.to_f64(matmul(normed(b(x)), b(w_qkv))), f"QKV with the row scale, M={m}")
    x1 = x.clone()
    ss1 = torch.empty_like(ss)
    kinv.gemm_fused(attn, w_o, kinv.residual_out(x1, ss1))
    ref_x1 = oglue.add_f64(b(x), ogemm(b(attn), b(w_o), out="f64"))
    assert_close(f64(x1), obf.to_f64(ref_x1), f"x + O, M={m}")
    check_ss(b(x1), ss1, "sums of squares after O")
    act = kinv.gemm_swiglu(x1, w_il, fusion=kinv.norm_in(ss1, d, 1e-6))
    ref_act = oglue.swiglu_f64(matmul(normed(b(x1)), b(w_gu), out="f64"))
    assert_close(f64(act), obf.to_f64(ref_act), f"gate/up + SwiGLU with the row scale, M={m}")
    x2 = x1.clone()
    ss2 = torch.empty_like(ss)
    kinv.gemm_fused(act, w_down, kinv.residual_out(x2, ss2))
    ref_x2 = oglue.add_f64(b(x1), ogemm(b(act), b(w_down), out="f64"))
    assert_close(f64(x2), obf.to_f64(ref_x2), f"x + down, M={m}")
    check_ss(b(x2), ss2, "sums of squares after down")
    # rows 0..3 alone (the push path) give the same bits
    x1s, ss1s = x[:4].clone(), torch.empty_like(ss[:4])
    kinv.gemm_fused(attn[:4].contiguous(), w_o, kinv.residual_out(x1s, ss1s))
    assert_same_bits(x1s, x1[:4], "x + O: 4 rows vs in the larger call")
    assert_same_bits(ss1s, ss1[:4], "sums of squares: 4 rows vs in the larger call")
    acts = kinv.gemm_swiglu(x1[:4].contiguous(), w_il, fusion=kinv.norm_in(ss1[:4].contiguous(), d, 1e-6))
    assert_same_bits(acts, act[:4], "gate/up: 4 rows vs in the larger call")
    assert kinv.last_device_status() == 0


def test_tile_schedule_partial_last_tile(kinv):
    """The tile schedule (400 rows, a K split) on widths that end in half a
    256-column tile: SwiGLU (F = 320, N = 640) and an fp32 output match the
    oracle, and their rows keep the bits of the same rows in a 4-row call
    (the cluster schedule)."""
    a = synth.normal_bf16((400, 512), 1.0, 95).cuda()
    w_gu = synth.normal_bf16((640, 512), 0.05, 96).cuda()
    w_il = kinv.interleave_gate_up(w_gu)
    act = kinv.gemm_swiglu(a, w_il)
    assert_close(f64(act), obf.to_f64(_swiglu_ref(a, w_gu)), "SwiGLU, 400 rows")
    assert_same_bits(kinv.gemm_swiglu(a[:4].contiguous(), w_il), act[:4], "SwiGLU: 4 rows vs 400")
    a2 = synth.normal_bf16((400, 256), 1.0, 97).cuda()
    w2 = synth.normal_bf16((1024, 256), 0.05, 98).cuda()
    c = kinv.gemm(a2, w2, out_dtype=torch.float32)
    assert_same_bits(kinv.gemm(a2[:4].contiguous(), w2, out_dtype=torch.float32), c[:4], "fp32: 4 rows vs 400")
    ref = ogemm(synth.bits(a2), synth.bits(w2), out="f64")
    assert np.allclose(c.double().cpu().numpy(), ref, rtol=1e-5, atol=1e-4)
    assert kinv.last_device_status() == 0
