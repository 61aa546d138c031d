"""Split-KV attention on the GPU: oracle parity, batch invariance, chunk
invariance and decode == one-row prefill."""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth
from oracle import attention as oattn, bf16 as obf

pytestmark = gpu


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


def _cache(bsz, lmax, hkv, d, seed, device="cuda"):
    k = synth.normal_bf16((bsz, lmax, hkv, d), 1.0, seed, device)
    v = synth.normal_bf16((bsz, lmax, hkv, d), 1.0, seed + 1, device)
    return k, v


@pytest.mark.parametrize("hq,hkv,d,lens,lmax", [
    (4, 2, 64, [0, 1, 2, 63, 64], 64),
    (32, 8, 128, [1, 255, 256, 257, 1000, 4097], 4352),
    (8, 1, 128, [513, 3], 600),
    (2, 2, 64, [300, 17], 300),
])
def test_decode_parity(kinv, hq, hkv, d, lens, lmax):
    bsz = len(lens)
    k, v = _cache(bsz, lmax, hkv, d, 20)
    q = synth.normal_bf16((bsz, hq, d), 1.0, 22).cuda()
    kv_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = kinv.attn_decode(q, k, v, kv_len)
    ref = oattn.decode(synth.bits(q), synth.bits(k), synth.bits(v), lens)
    assert_close(f64(out), obf.to_f64(ref), f"decode Hq={hq} Hkv={hkv} D={d}")
    if 0 in lens:
        assert torch.all(out[lens.index(0)] == 0)
    assert kinv.last_device_status() == 0


def test_decode_config3_invariance_and_sampled_parity(kinv):
    """32 query / 8 kv heads, D 128, KV lengths U{1..32768}, split 256:
    a sequence's bits do not depend on its batch-mates or their lengths."""
    bsz, lmax, hq, hkv, d = 128, 32768, 32, 8, 128
    k, v = _cache(bsz, lmax, hkv, d, 30)
    q = synth.normal_bf16((bsz, hq, d), 1.0, 32, "cuda")
    lens = synth.uniform_int(bsz, 1, lmax, synth.SEED_LEN)
    kv_len = lens.cuda()
    out = kinv.attn_decode(q, k, v, kv_len)
    picks = [0, 1, 77, 127]
    for b in picks:
        one = kinv.attn_decode(q[b: b + 1].contiguous(), k[b: b + 1], v[b: b + 1], kv_len[b: b + 1])
        assert_same_bits(one, out[b: b + 1], f"seq {b} alone vs in batch 128")
    # other batch-mates with other lengths, the sequence at another slot
    perm = torch.randperm(bsz, generator=synth.gen(33))
    out_p = kinv.attn_decode(q[perm].contiguous(), k[perm], v[perm], kv_len[perm].contiguous())
    inv = torch.argsort(perm)
    assert_same_bits(out_p[inv], out, "permuted batch")
    lens2 = kv_len.clone()
    lens2[1:] = synth.uniform_int(bsz - 1, 1, lmax, 34).cuda()
    out2 = kinv.attn_decode(q, k, v, lens2)
    assert_same_bits(out2[0], out[0], "seq 0 with mates of other lengths")
    for b in picks[:3]:
        n = int(lens[b])
        ref = oattn.decode(synth.bits(q[b: b + 1]), synth.bits(k[b: b + 1, :n]),
                           synth.bits(v[b: b + 1, :n]), [n])
        assert_close(f64(out[b: b + 1]), obf.to_f64(ref), f"oracle seq {b} (L={n})")


# 2, 4, 8 and 1 query heads per kv head: 32, 16, 8 and 64 rows per prefill block
@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (32, 8, 128), (8, 1, 128), (2, 2, 64)])
def test_prefill_parity_chunk_invariance_and_decode_equality(kinv, hq, hkv, d):
    lmax, p0, t_len = 1100, 200, 700
    k, v = _cache(1, lmax, hkv, d, 40)
    q = synth.normal_bf16((t_len, hq, d), 1.0, 42).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")

    def run(rows0, n):
        return kinv.attn_prefill(q[rows0: rows0 + n].contiguous(), k, v,
                                 torch.tensor([p0 + rows0], **i32), torch.tensor([n], **i32),
                                 torch.zeros(1, **i32), n, p0 + rows0 + n)

    whole = run(0, t_len)
    ref = oattn.prefill(synth.bits(q), synth.bits(k[0]), synth.bits(v[0]), p0)
    assert_close(f64(whole), obf.to_f64(ref), "prefill vs oracle")
    for chunk in (1, 7, 64, 512):
        parts = [run(r0, min(chunk, t_len - r0)) for r0 in range(0, t_len, chunk)] if chunk > 1 else \
            [run(r0, 1) for r0 in (0, 55, 56, 311, 699)]
        if chunk > 1:
            assert_same_bits(torch.cat(parts), whole, f"chunk {chunk}")
        else:
            for r0, part in zip((0, 55, 56, 311, 699), parts):
                assert_same_bits(part, whole[r0: r0 + 1], f"row {r0} alone")
    for t in (0, 56, 699):
        dec = kinv.attn_decode(q[t: t + 1].contiguous(), k, v, torch.tensor([p0 + t + 1], **i32))
        assert_same_bits(dec, whole[t: t + 1], f"decode == prefill row {t}")


def test_prefill_many_sequences(kinv):
    """Several sequences in one call (varlen rows) equal one call each."""
    hq, hkv, d, lmax = 32, 8, 128, 700
    k, v = _cache(3, lmax, hkv, d, 50)
    lens = [5, 300, 1]
    starts = [0, 100, 650]
    offs = [0, 5, 305]
    rows = sum(lens)
    q = synth.normal_bf16((rows, hq, d), 1.0, 52).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    out = kinv.attn_prefill(q, k, v, torch.tensor(starts, **i32), torch.tensor(lens, **i32),
                            torch.tensor(offs, **i32), max(lens), max(s + n for s, n in zip(starts, lens)))
    for b in range(3):
        one = kinv.attn_prefill(q[offs[b]: offs[b] + lens[b]].contiguous(), k[b: b + 1], v[b: b + 1],
                                torch.tensor([starts[b]], **i32), torch.tensor([lens[b]], **i32),
                                torch.zeros(1, **i32), lens[b], starts[b] + lens[b])
        assert_same_bits(one, out[offs[b]: offs[b] + lens[b]], f"sequence {b}")
        ref = oattn.prefill(synth.bits(q[offs[b]: offs[b] + lens[b]]), synth.bits(k[b]),
                            synth.bits(v[b]), starts[b])
        assert_close(f64(one), obf.to_f64(ref), f"oracle sequence {b}")


def test_workspace_too_small_is_rejected(kinv):
    k, v = _cache(2, 512, 2, 64, 60)
    q = synth.normal_bf16((2, 4, 64), 1.0, 61).cuda()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kinv.KinvError) as e:
        kinv.attn_decode(q, k, v, torch.tensor([3, 4], dtype=torch.int32, device="cuda"), workspace=ws)
    assert e.value.status == kinv.ERR_WORKSPACE


def test_device_lengths_outside_bounds_are_left_out_and_reported(kinv):
    """kv_len is device data the host cannot check: a sequence whose length
    lies outside [0, Lmax] (decode) or whose rows or keys fall outside the
    stated bounds (prefill) is left out and the status word says so.  The
    workspace past what the call needs is filled with NaN bit patterns and the
    cache past Lmax with NaN too, so a read beyond either would show in the
    other sequences' outputs."""
    hq, hkv, d, lmax = 4, 2, 64, 512
    pad = 300
    i32 = dict(dtype=torch.int32, device="cuda")
    kfull, vfull = _cache(3, lmax + pad, hkv, d, 70)
    kfull[:, lmax:] = float("nan")
    vfull[:, lmax:] = float("nan")
    k, v = kfull[:, :lmax], vfull[:, :lmax]          # strides of the padded buffer
    q = synth.normal_bf16((3, hq, d), 1.0, 71).cuda()
    need = kinv.attn_decode_workspace(3, hq, d, lmax)
    ws = torch.full((need + (1 << 20),), 0xFF, dtype=torch.uint8, device="cuda")
    good = kinv.attn_decode(q, k, v, torch.tensor([100, 5, 7], **i32))
    assert kinv.last_device_status() == 0
    for bad_slot, bad_len in ((1, lmax + pad), (2, lmax + 1), (0, -3)):
        lens = [100, 5, 7]
        lens[bad_slot] = bad_len
        out = kinv.attn_decode(q, k, v, torch.tensor(lens, **i32), workspace=ws)
        assert kinv.last_device_status() == kinv.ERR_INVALID_ARG
        assert torch.all(out[bad_slot] == 0)
        for b in range(3):
            if b != bad_slot:
                assert_same_bits(out[b], good[b], f"sequence {b} beside a bad length at {bad_slot}")
    # prefill: sequence 1 claims keys past max_kv; sequence 0 is untouched by it
    rows = [5, 6]
    qp = synth.normal_bf16((11, hq, d), 1.0, 72).cuda()
    out = torch.full_like(qp, 7.0)
    starts, offs = [20, lmax - 3], [0, 5]
    kinv.attn_prefill(qp, k[:2], v[:2], torch.tensor(starts, **i32), torch.tensor(rows, **i32),
                      torch.tensor(offs, **i32), 6, lmax, out=out)
    assert kinv.last_device_status() == kinv.ERR_INVALID_ARG
    assert torch.all(out[5:] == 7.0)
    alone = kinv.attn_prefill(qp[:5].contiguous(), k[:1], v[:1], torch.tensor([20], **i32),
                              torch.tensor([5], **i32), torch.zeros(1, **i32), 5, 25)
    assert_same_bits(out[:5], alone, "valid sequence beside an out-of-bounds one")
    assert kinv.last_device_status() == 0
