"""kinv_sample on the GPU: token parity with the oracle, bit-exactness across
batch composition, ties, greedy and the unsupported-settings path."""
import json
import os

import numpy as np
import pytest
import torch

from helpers import ensure_lib, gpu, synth
from oracle.sampler import SamplingParams as OParams, sample_row

pytestmark = gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "receipt_sampling.json")


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


def _receipt_params():
    with open(GOLDEN) as fh:
        g = json.load(fh)
    return dict(temperature=g["temperature"], top_k=g["top_k"], top_p=g["top_p"],
                min_p=g["min_p"], repeat_penalty=g["repeat_penalty"],
                repeat_last_n=g["repeat_last_n"], seed=g["seed"])


def _run(kinv, logits, plist, hists, steps, hist_ld=64):
    bsz = logits.shape[0]
    pdev, _bias = kinv.sampling_params_device(plist)
    hist = torch.zeros(bsz, hist_ld, dtype=torch.int32)
    hl = torch.zeros(bsz, dtype=torch.int32)
    for b, h in enumerate(hists):
        h = list(h)[-hist_ld:]
        hist[b, : len(h)] = torch.tensor(h, dtype=torch.int32)
        hl[b] = len(h)
    st = torch.tensor(steps, dtype=torch.int64)
    return kinv.sample(logits, pdev, hist.cuda(), hl.cuda(), st.cuda()).cpu().numpy()


def _oracle(logits, plist, hists, steps):
    z = logits.cpu().numpy()
    toks, ties = [], []
    for b in range(z.shape[0]):
        p = OParams(**{k: getattr(plist[b], k) for k in OParams.__dataclass_fields__})
        t, n = sample_row(z[b], list(hists[b])[-64:], steps[b], p)
        toks.append(t)
        ties.append(n)
    return np.array(toks), np.array(ties)


@pytest.mark.parametrize("sigma", [1.3, 5.0])
def test_token_parity_receipt_settings(kinv, sigma):
    bsz, vocab = 64, 151936
    g = synth.gen(70)
    logits = (torch.randn(bsz, vocab, generator=g) * sigma).cuda()
    base = _receipt_params()
    plist = [kinv.SamplingParams(**{**base, "seed": 1000 + b}) for b in range(bsz)]
    hists = [torch.randint(0, vocab, (int(torch.randint(0, 100, (1,), generator=g)),), generator=g).tolist()
             for _ in range(bsz)]
    # make the penalty matter: put some history ids at the top
    for b in range(0, bsz, 4):
        top = torch.topk(logits[b], 3).indices.cpu().tolist()
        hists[b] = hists[b] + top
    steps = [int(s) for s in torch.randint(0, 10 ** 6, (bsz,), generator=g)]
    got = _run(kinv, logits, plist, hists, steps)
    ref, ties = _oracle(logits, plist, hists, steps)
    ok = ~ties
    assert ties.sum() <= max(2, bsz // 16), f"{ties.sum()} near ties"
    assert np.array_equal(got[ok], ref[ok]), np.nonzero(got != ref)
    assert kinv.last_device_status() == 0


def test_setting_variants(kinv):
    vocab = 151936
    g = synth.gen(71)
    variants = [
        dict(temperature=0.0, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.1, repeat_last_n=64),
        dict(temperature=1.0, top_k=1, top_p=1.0, min_p=0.0, repeat_penalty=1.0, repeat_last_n=0),
        dict(temperature=1.5, top_k=1024, top_p=1.0, min_p=0.0, repeat_penalty=1.3, repeat_last_n=-1),
        dict(temperature=0.7, top_k=200, top_p=0.5, min_p=0.0, repeat_penalty=1.0, repeat_last_n=64),
        dict(temperature=0.7, top_k=200, top_p=1.0, min_p=0.2, repeat_penalty=0.9, repeat_last_n=8),
        dict(temperature=2.0, top_k=vocab + 5, top_p=1.0, min_p=0.0, repeat_penalty=1.0, repeat_last_n=0),
    ]
    plist, hists, steps = [], [], []
    for i, v in enumerate(variants):
        for j in range(4):
            plist.append(kinv.SamplingParams(**v, seed=17 * i + j))
            hists.append(torch.randint(0, 500, (70,), generator=g).tolist())
            steps.append(i * 100 + j)
    logits = (torch.randn(len(plist), vocab, generator=g) * 2).cuda()
    logits[:, :500] += 3.0   # the history ids are among the top candidates
    # the last variant keeps the whole vocabulary only when V <= 1024: shrink it
    small = logits[-4:, :1000].contiguous()
    got = _run(kinv, logits[:-4].contiguous(), plist[:-4], hists[:-4], steps[:-4])
    ref, ties = _oracle(logits[:-4], plist[:-4], hists[:-4], steps[:-4])
    assert np.array_equal(got[~ties], ref[~ties])
    got2 = _run(kinv, small, plist[-4:], hists[-4:], steps[-4:])
    ref2, ties2 = _oracle(small, plist[-4:], hists[-4:], steps[-4:])
    assert np.array_equal(got2[~ties2], ref2[~ties2])


def test_presence_and_frequency_penalties(kinv):
    """Presence and frequency penalties on top of the repeat penalty, with the
    window counted from shared memory (<= 256 ids) and from the history row
    (400 ids); zero penalties give the bits of the repeat penalty alone."""
    vocab = 151936
    g = synth.gen(74)
    hist_ld = 512
    variants = [
        dict(temperature=0.0, top_k=50, top_p=1.0, min_p=0.0, repeat_penalty=1.1, repeat_last_n=64,
             presence_penalty=0.5, frequency_penalty=0.4),
        dict(temperature=0.8, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.0, repeat_last_n=64,
             presence_penalty=0.0, frequency_penalty=0.7),
        dict(temperature=1.0, top_k=200, top_p=1.0, min_p=0.0, repeat_penalty=1.2, repeat_last_n=-1,
             presence_penalty=1.5, frequency_penalty=0.0),
        dict(temperature=0.0, top_k=20, top_p=1.0, min_p=0.0, repeat_penalty=1.0, repeat_last_n=400,
             presence_penalty=-0.5, frequency_penalty=0.3),
    ]
    plist, hists, steps = [], [], []
    for i, v in enumerate(variants):
        for j in range(6):
            plist.append(kinv.SamplingParams(**v, seed=31 * i + j))
            # few distinct ids, many repeats: counts up to dozens
            hists.append(torch.randint(0, 40, (400,), generator=g).tolist())
            steps.append(7 * i + j)
    logits = (torch.randn(len(plist), vocab, generator=g) * 2).cuda()
    logits[:, :40] += 4.0   # the history ids are the top candidates
    got = _run(kinv, logits, plist, hists, steps, hist_ld=hist_ld)
    z = logits.cpu().numpy()
    for b, p in enumerate(plist):
        op = OParams(**{k: getattr(p, k) for k in OParams.__dataclass_fields__})
        t, tie = sample_row(z[b], hists[b][-hist_ld:], steps[b], op)
        if not tie:
            assert got[b] == t, (b, got[b], t)
    # zero presence and frequency: the bits of the repeat penalty alone
    zero = [kinv.SamplingParams(**{**variants[0], "presence_penalty": 0.0, "frequency_penalty": 0.0},
                                seed=3) for _ in range(4)]
    a = _run(kinv, logits[:4].contiguous(), zero, hists[:4], steps[:4], hist_ld=hist_ld)
    ref = [sample_row(z[b], hists[b][-hist_ld:], steps[b],
                      OParams(**{k: getattr(zero[b], k) for k in OParams.__dataclass_fields__}))[0]
           for b in range(4)]
    assert list(a) == ref
    assert kinv.last_device_status() == 0


def test_logit_bias(kinv):
    """Logit-bias lists (bans with -inf, forced ids, small biases on ids the
    penalties also touch) match the oracle token for token; a row's bias does
    not change its batch-mates' tokens."""
    vocab = 151936
    g = synth.gen(75)
    plist, hists, steps = [], [], []
    logits = (torch.randn(24, vocab, generator=g) * 2)
    logits[:, :40] += 4.0
    for b in range(24):
        kind = b % 4
        if kind == 0:     # ban the row's ten most likely ids
            top = torch.topk(logits[b], 10).indices.tolist()
            bias = {t: float("-inf") for t in top}
        elif kind == 1:   # force one id
            bias = {int(torch.randint(1000, vocab, (1,), generator=g)): 50.0}
        elif kind == 2:   # small biases on history ids, with penalties on
            bias = {t: float(torch.randn(1, generator=g)) for t in range(0, 40, 3)}
        else:             # no bias at all
            bias = None
        plist.append(kinv.SamplingParams(temperature=0.0 if b % 8 == 0 else 0.9, top_k=100, top_p=0.95,
                                         min_p=0.0, repeat_penalty=1.2, repeat_last_n=32,
                                         presence_penalty=0.3 if kind == 2 else 0.0,
                                         frequency_penalty=0.2 if kind == 2 else 0.0,
                                         logit_bias=bias, seed=900 + b))
        hists.append(torch.randint(0, 40, (50,), generator=g).tolist())
        steps.append(11 * b)
    logits = logits.cuda()
    got = _run(kinv, logits, plist, hists, steps)
    z = logits.cpu().numpy()
    for b, p in enumerate(plist):
        op = OParams(**{k: getattr(p, k) for k in OParams.__dataclass_fields__})
        t, tie = sample_row(z[b], hists[b][-64:], steps[b], op)
        if not tie:
            assert got[b] == t, (b, got[b], t)
        if b % 4 == 0:
            assert got[b] not in set(p.logit_bias), (b, got[b])
        if b % 4 == 1:
            assert got[b] == next(iter(p.logit_bias)), (b, got[b])
    # the rows without a bias draw the same tokens with biased rows beside them or alone
    for b in (3, 7):
        one = _run(kinv, logits[b: b + 1].contiguous(), plist[b: b + 1], hists[b: b + 1], steps[b: b + 1])
        assert one[0] == got[b]
    assert kinv.last_device_status() == 0


def test_typical_p(kinv):
    """Typical-p with top-k, top-p, min-p and temperature against the oracle,
    and over the whole vocabulary (no top-k)."""
    vocab = 151936
    g = synth.gen(76)
    variants = [
        dict(temperature=1.0, top_k=50, top_p=1.0, min_p=0.0, typical_p=0.5),
        dict(temperature=0.8, top_k=200, top_p=0.95, min_p=0.05, typical_p=0.9),
        dict(temperature=1.3, top_k=1024, top_p=1.0, min_p=0.1, typical_p=0.2),
        dict(temperature=0.7, top_k=20, top_p=0.8, min_p=0.0, typical_p=0.95),
    ]
    plist, steps = [], []
    for i, v in enumerate(variants):
        for j in range(8):
            plist.append(kinv.SamplingParams(**v, repeat_penalty=1.1, repeat_last_n=16, seed=77 * i + j))
            steps.append(5 * i + j)
    hists = [torch.randint(0, 50, (20,), generator=g).tolist() for _ in plist]
    logits = (torch.randn(len(plist), vocab, generator=g) * 2.5).cuda()
    got = _run(kinv, logits, plist, hists, steps)
    ref, ties = _oracle(logits, plist, hists, steps)
    assert ties.sum() <= 8, f"{ties.sum()} near ties"
    assert np.array_equal(got[~ties], ref[~ties]), np.nonzero(got != ref)
    # a typical-p pick can leave out the most likely id: seen in these rows
    z = logits.cpu().numpy()
    top1 = z.argmax(axis=1)
    assert np.any(got[:8] != top1[:8])
    assert kinv.last_device_status() == 0
    # the whole vocabulary: typical set, then top-p and min-p over it
    whole_v = [dict(temperature=1.0, top_k=0, top_p=0.9, min_p=0.0, typical_p=0.5),
               dict(temperature=0.8, top_k=0, top_p=1.0, min_p=0.05, typical_p=0.9),
               dict(temperature=1.2, top_k=-1, top_p=0.95, min_p=0.01, typical_p=0.3),
               dict(temperature=0.9, top_k=0, top_p=1.0, min_p=0.0, typical_p=0.95)]
    whole = [kinv.SamplingParams(**v, repeat_penalty=1.0, repeat_last_n=0, seed=31 + i)
             for i, v in enumerate(whole_v) for _ in range(2)]
    # rows with a few raised ids: the typical set's edge is not crowded
    wl = _peaked(len(whole), vocab, 78)
    wh, ws = [[] for _ in whole], list(range(len(whole)))
    out = _run(kinv, wl, whole, wh, ws)
    ref, ties = _oracle(wl, whole, wh, ws)
    assert (out >= 0).all()
    assert ties.sum() <= 2, f"{ties.sum()} near ties"
    assert np.array_equal(out[~ties], ref[~ties]), np.nonzero(out != ref)
    one = _run(kinv, wl[3:4].contiguous(), whole[3:4], wh[3:4], ws[3:4])
    assert one[0] == out[3]
    assert kinv.last_device_status() == 0


def test_exact_ties_take_lowest_ids(kinv):
    vocab = 151936
    logits = torch.zeros(3, vocab, device="cuda")
    logits[1, 7] = 1.0
    p = [kinv.SamplingParams(temperature=1.0, top_k=50, top_p=1.0, min_p=0.0, repeat_penalty=1.0,
                             repeat_last_n=0, seed=s) for s in range(3)]
    p[2].temperature = 0.0
    steps = [0, 1, 2]
    got = _run(kinv, logits, p, [[], [], []], steps)
    ref, ties = _oracle(logits, p, [[], [], []], steps)
    assert np.array_equal(got, ref)
    assert got[0] < 50 and got[2] == 0


def test_row_bits_independent_of_batch(kinv):
    vocab = 151936
    g = synth.gen(72)
    logits = (torch.randn(32, vocab, generator=g) * 1.3).cuda()
    base = _receipt_params()
    plist = [kinv.SamplingParams(**{**base, "seed": 5000 + b}) for b in range(32)]
    hists = [list(range(b, b + 40)) for b in range(32)]
    steps = list(range(100, 132))
    full = _run(kinv, logits, plist, hists, steps)
    for b in (0, 13, 31):
        one = _run(kinv, logits[b: b + 1].contiguous(), plist[b: b + 1], hists[b: b + 1], steps[b: b + 1])
        assert one[0] == full[b]
    perm = torch.randperm(32, generator=g).tolist()
    got = _run(kinv, logits[perm].contiguous(), [plist[i] for i in perm], [hists[i] for i in perm],
               [steps[i] for i in perm])
    assert np.array_equal(got, full[perm])


def test_unsupported_top_k_reports_status(kinv):
    logits = torch.randn(2, 5000, device="cuda")
    p = [kinv.SamplingParams(top_k=2000, seed=1), kinv.SamplingParams(top_k=10, seed=2)]
    got = _run(kinv, logits, p, [[], []], [0, 0])
    assert got[0] == -1 and got[1] >= 0
    assert kinv.last_device_status() == kinv.ERR_UNSUPPORTED
    assert kinv.last_device_status() == 0


def _peaked(rows, vocab, seed, boost=12.0, n_top=20):
    """N(0, 1.3) logits with n_top ids per row raised by `boost`: the top-p /
    min-p cut falls among those ids even over the whole vocabulary."""
    g = synth.gen(seed)
    logits = torch.randn(rows, vocab, generator=g) * 1.3
    for b in range(rows):
        ids = torch.randint(0, vocab, (n_top,), generator=g)
        logits[b, ids] += boost + torch.rand(n_top, generator=g) * 2.0
    return logits.cuda()


@pytest.mark.parametrize("top_k,top_p,min_p", [(0, 0.9, 0.0), (-1, 1.0, 0.05), (0, 0.95, 0.02)])
def test_whole_vocabulary_top_p_min_p(kinv, top_k, top_p, min_p):
    """top_k <= 0 samples over all 151936 ids (softmax total over the whole
    row); tokens match the oracle away from near ties, and a row's token does
    not depend on the batch (the number of blocks sharing a row follows it)."""
    vocab, bsz = 151936, 32
    logits = _peaked(bsz, vocab, 80)
    plist = [kinv.SamplingParams(temperature=0.8, top_k=top_k, top_p=top_p, min_p=min_p,
                                 repeat_penalty=1.1, repeat_last_n=64, seed=900 + b) for b in range(bsz)]
    hists = [list(range(10 * b, 10 * b + 30)) for b in range(bsz)]
    steps = list(range(bsz))
    got = _run(kinv, logits, plist, hists, steps)
    ref, ties = _oracle(logits, plist, hists, steps)
    assert (got >= 0).all()
    assert ties.sum() <= bsz // 4, f"{ties.sum()} near ties"
    assert np.array_equal(got[~ties], ref[~ties]), np.nonzero(got != ref)
    for b in (0, 17):
        one = _run(kinv, logits[b: b + 1].contiguous(), plist[b: b + 1], hists[b: b + 1], steps[b: b + 1])
        assert one[0] == got[b]
    assert kinv.last_device_status() == 0


@pytest.mark.parametrize("temperature,top_p,min_p", [(0.8, 0.95, 0.0), (1.0, 0.5, 0.0), (0.6, 0.99, 0.0),
                                                       (1.2, 1.0, 0.02), (0.9, 0.9, 0.001)])
def test_whole_vocabulary_flat_rows(kinv, temperature, top_p, min_p):
    """Un-peaked N(0, 1.3) logits over all 151936 ids: the top-p / min-p cut
    lies tens of thousands of ids deep and most ids weigh less than the
    oracle's margin, so many rows are near ties.  Away from near ties the token
    is the oracle's; at a near tie it is one the oracle reaches within the
    margins.  A row's token does not depend on the batch; an all-equal row
    (every id tied) gives a valid token."""
    vocab, bsz = 151936, 16
    g = synth.gen(85)
    logits = torch.randn(bsz, vocab, generator=g) * 1.3
    logits[bsz - 1] = 0.0
    logits = logits.cuda()
    plist = [kinv.SamplingParams(temperature=temperature, top_k=0, top_p=top_p, min_p=min_p,
                                 repeat_penalty=1.1, repeat_last_n=64, seed=700 + b) for b in range(bsz)]
    hists = [list(range(100 * b, 100 * b + 40)) for b in range(bsz)]
    steps = [3 * b for b in range(bsz)]
    got = _run(kinv, logits, plist, hists, steps)
    ref, ties = _oracle(logits, plist, hists, steps)
    assert (got >= 0).all() and (got < vocab).all()
    assert np.array_equal(got[~ties], ref[~ties]), np.nonzero(got != ref)
    assert (~ties[: bsz - 1]).sum() >= 3, f"only {(~ties).sum()} rows away from near ties"
    z = logits.cpu().numpy()
    for b in np.nonzero(ties[: bsz - 1])[0]:
        ok = set()
        p = OParams(**{k: getattr(plist[b], k) for k in OParams.__dataclass_fields__})
        sample_row(z[b], hists[b][-64:], steps[b], p, allowed=ok)
        assert int(got[b]) in ok, (b, int(got[b]), sorted(ok)[:10])
    for b in (0, 5, bsz - 1):
        one = _run(kinv, logits[b: b + 1].contiguous(), plist[b: b + 1], hists[b: b + 1], steps[b: b + 1])
        assert one[0] == got[b]
    assert kinv.last_device_status() == 0
