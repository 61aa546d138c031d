"""kinv_rmsnorm and the element-wise glue on the GPU: oracle parity and row
invariance."""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth
from oracle import bf16 as obf, glue as oglue
from oracle.rmsnorm import rmsnorm as ormsnorm
from oracle.rope import rope as orope

pytestmark = gpu


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


@pytest.mark.parametrize("dim", [128, 256, 4096, 12288])
def test_rmsnorm_parity_and_invariance(kinv, dim):
    x = synth.normal_bf16((256, dim), 1.0, 1).cuda()
    w = synth.normal_bf16((dim,), 0.5, 2).cuda() + 1
    y = kinv.rmsnorm(x, w, 1e-6)
    ref = ormsnorm(synth.bits(x), synth.bits(w), 1e-6)
    assert_close(f64(y), obf.to_f64(ref), f"rmsnorm d={dim}")
    for m in (1, 3, 16, 255):
        assert_same_bits(kinv.rmsnorm(x[:m].contiguous(), w, 1e-6), y[:m], f"rows={m}")
    perm = torch.randperm(256, generator=synth.gen(3)).cuda()
    assert_same_bits(kinv.rmsnorm(x[perm].contiguous(), w, 1e-6), y[perm], "permuted rows")


def test_rmsnorm_residual_fusion(kinv):
    x = synth.normal_bf16((33, 4096), 1.0, 4).cuda()
    r = synth.normal_bf16((33, 4096), 1.0, 5).cuda()
    w = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    xs = x.clone()
    y = kinv.rmsnorm(xs, w, 1e-6, residual=r)
    ry, rs = ormsnorm(synth.bits(x), synth.bits(w), 1e-6, residual_bits=synth.bits(r))
    assert_close(f64(xs), obf.to_f64(rs), "residual stream")
    assert_close(f64(y), obf.to_f64(ry), "normed")
    assert np.array_equal(synth.bits(xs), oglue.add(synth.bits(x), synth.bits(r)))


def test_rmsnorm_edge_rows(kinv):
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(3, 256, dtype=torch.bfloat16, device="cuda")
    x[1] = 3.0
    x[2, 7] = -5.0
    y = kinv.rmsnorm(x, w, 1e-6)
    ref = ormsnorm(synth.bits(x), synth.bits(w), 1e-6)
    assert np.array_equal(synth.bits(y)[0], ref[0])          # zero row stays zero
    assert_close(f64(y), obf.to_f64(ref), "edge rows")


def test_swiglu_add_embed(kinv):
    gu = synth.normal_bf16((9, 2 * 512), 2.0, 6).cuda()
    a = kinv.swiglu(gu)
    assert_close(f64(a), obf.to_f64(oglue.swiglu(synth.bits(gu))), "swiglu")
    x = synth.normal_bf16((7, 64), 1.0, 7).cuda()
    y = synth.normal_bf16((7, 64), 1.0, 8).cuda()
    s = kinv.add(x, y)
    ref = oglue.add(synth.bits(x), synth.bits(y))
    assert_close(f64(s), obf.to_f64(ref), "add")
    tab = synth.normal_bf16((100, 256), 1.0, 9).cuda()
    ids = torch.tensor([5, 0, 99, 5, 200, -1], dtype=torch.int32, device="cuda")
    e = kinv.embed(tab, ids)
    assert_same_bits(e[:4], tab[[5, 0, 99, 5]], "embed")
    assert torch.all(e[4:] == 0)


@pytest.mark.parametrize("d,hq,hkv,base,qk", [(64, 4, 2, 1e4, False), (128, 32, 8, 1e6, True)])
def test_rope_append(kinv, d, hq, hkv, base, qk):
    rows, bsz, lmax = 6, 3, 40
    qkv = synth.normal_bf16((rows, (hq + 2 * hkv) * d), 1.0, 10).cuda()
    seq = torch.tensor([0, 2, 1, 2, 0, 1], dtype=torch.int32)
    pos = torch.tensor([0, 39, 5, 17, 1, 32], dtype=torch.int32)
    kc = torch.zeros(bsz, lmax, hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.empty(rows, hq, d, dtype=torch.bfloat16, device="cuda")
    qn = (synth.normal_bf16((d,), 0.3, 11) + 1).cuda() if qk else None
    kn = (synth.normal_bf16((d,), 0.3, 12) + 1).cuda() if qk else None
    kinv.rope_append(qkv, q, kc, vc, seq.cuda(), pos.cuda(), hq, hkv, d, base, qn, kn, 1e-6)
    qb = synth.bits(qkv).reshape(rows, hq + 2 * hkv, d)
    rq = orope(qb[:, :hq], pos.numpy(), base, synth.bits(qn) if qk else None)
    rk = orope(qb[:, hq: hq + hkv], pos.numpy(), base, synth.bits(kn) if qk else None)
    assert_close(f64(q), obf.to_f64(rq), "rope q")
    for i in range(rows):
        s, p = int(seq[i]), int(pos[i])
        assert_close(f64(kc[s, p]), obf.to_f64(rk[i]), f"rope k row {i}")
        assert np.array_equal(synth.bits(vc[s, p]), qb[i, hq + hkv:])
    # untouched slots stay zero
    assert torch.all(kc[0, 2] == 0) and torch.all(vc[1, 0] == 0)


def test_decode_advance(kinv):
    hist = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    hist[1] = torch.tensor([1, 2, 3, 4])
    hl = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    step = torch.tensor([0, 10], dtype=torch.int64, device="cuda")
    pos = torch.tensor([5, 6], dtype=torch.int32, device="cuda")
    kvl = torch.tensor([6, 7], dtype=torch.int32, device="cuda")
    tok = torch.tensor([9, 8], dtype=torch.int32, device="cuda")
    kinv.decode_advance(tok, hist, hl, step, pos=pos, kv_len=kvl)
    assert hist.cpu().tolist() == [[9, 0, 0, 0], [2, 3, 4, 8]]
    assert hl.cpu().tolist() == [1, 4] and step.cpu().tolist() == [1, 11]
    assert pos.cpu().tolist() == [6, 7] and kvl.cpu().tolist() == [7, 8]


@pytest.mark.parametrize("d,hq,hkv,base,qk,k,m", [(64, 4, 2, 1e4, False, 256, 5), (128, 32, 8, 1e6, True, 4096, 1),
                                                  (128, 32, 8, 1e6, True, 4096, 8),
                                                  (128, 32, 8, 1e6, True, 4096, 16),
                                                  (128, 32, 8, 1e6, True, 4096, 64),
                                                  (128, 32, 8, 1e6, True, 4096, 200)])
def test_gemm_qkv_rope_equals_gemm_then_rope_append(kinv, d, hq, hkv, base, qk, k, m):
    """The fused projection writes the same bits as kinv_gemm followed by
    kinv_rope_append: q, the new K/V cache slots, and nothing else."""
    n = (hq + 2 * hkv) * d
    a = synth.normal_bf16((m, k), 1.0, 30).cuda()
    w = synth.normal_bf16((n, k), 0.02, 31).cuda()
    bsz, lmax = 4, 300
    seq = torch.arange(m, dtype=torch.int32) % bsz  # distinct (seq, pos) slots per row
    pos = torch.arange(m, dtype=torch.int32) // bsz + 7
    qn = (synth.normal_bf16((d,), 0.3, 32) + 1).cuda() if qk else None
    kn = (synth.normal_bf16((d,), 0.3, 33) + 1).cuda() if qk else None
    outs = []
    for fused in (False, True):
        kc = torch.zeros(bsz, lmax, hkv, d, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        q = torch.zeros(m, hq, d, dtype=torch.bfloat16, device="cuda")
        if fused:
            kinv.gemm_qkv_rope(a, w, q, kc, vc, seq.cuda(), pos.cuda(), hq, hkv, d, base, qn, kn, 1e-6)
        else:
            qkv = kinv.gemm(a, w)
            kinv.rope_append(qkv, q, kc, vc, seq.cuda(), pos.cuda(), hq, hkv, d, base, qn, kn, 1e-6)
        outs.append((q, kc, vc))
    for x, y, name in zip(outs[0], outs[1], ("q", "k cache", "v cache")):
        assert_same_bits(y, x, f"fused {name}")
    assert kinv.last_device_status() == 0


def test_scale_columns_matches_the_oracle_product(kinv):
    """kinv_scale_columns: bf16(w * g) per element (the fp32 product of two
    bf16 values is exact, so one rounding), for a gain vector with values
    that are and are not powers of two."""
    n, k = 300, 512
    w = synth.normal_bf16((n, k), 0.02, 91).cuda()
    g = (0.5 + torch.rand(k, generator=synth.gen(92))).to(torch.bfloat16)
    g[:8] = torch.tensor([1, 2, 0.5, 4, 0.25, -1, 0, 3], dtype=torch.bfloat16)
    got = kinv.scale_columns(w, g.cuda())
    ref = obf.from_f64(obf.to_f64(synth.bits(w)) * obf.to_f64(synth.bits(g))[None, :])
    assert np.array_equal(synth.bits(got), ref)
    # in place
    w2 = w.clone()
    kinv.scale_columns(w2, g.cuda(), out=w2)
    assert_same_bits(w2, got, "in place")
