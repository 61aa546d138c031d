"""Qwen3-8B-shaped stacks on the GPU.

* Chunked prefill: a 4096-token prompt processed whole and in chunks of 512,
  64 and 1 gives bit-identical outputs and KV caches, and the decode that
  follows emits the same tokens.
* A tagged request emits identical tokens (and logits bits) alone and
  co-batched with other requests of other prompt lengths, at any slot.
* First-step logits of short prompts match the oracle.
Depth is reduced in the chunking and co-batching tests (full widths, full
vocabulary); the full 36-layer depth runs once alone vs co-batched."""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth
from oracle import bf16 as obf
from oracle.model import Shape
from oracle.sampler import SamplingParams as OParams

pytestmark = gpu


@pytest.fixture(scope="module")
def M():
    ensure_lib()
    from invariant_deterministic_gb300 import model
    return model


def _shape(M, layers):
    s = M.QWEN3_8B
    return M.ModelShape(**{**s.__dict__, "n_layers": layers})


def _params(M, n, base_seed=1000):
    return [M.kinv.SamplingParams(seed=base_seed + i) for i in range(n)]


def test_chunked_prefill_bit_identical_then_same_decode(M):
    shape = _shape(M, 2)
    w = M.random_weights(shape, device="cuda")
    T = 4096
    prompt = synth.uniform_int(T, 0, shape.vocab - 1, 80).cuda()
    results = {}
    for chunk in (4096, 512, 64, 1):
        dec = M.Decoder(shape, w, max_batch=1, max_len=T + 16, max_chunk=min(chunk, 4096))
        outs = []
        for p0 in range(0, T, chunk):
            n = min(chunk, T - p0)
            M.kinv.embed(w["embed"], prompt[p0: p0 + n], out=dec.x[:n])
            dec.prefill_chunk(0, p0, n)
            outs.append(dec.close_residual(n).clone())
        hidden = torch.cat(outs)
        # decode 8 tokens after the prompt
        dec.set_sampling(_params(M, 1))
        dec.set_history([prompt[-64:].cpu().tolist()])
        dec.set_positions([T])
        dec.tokens[0] = prompt[-1]
        toks = []
        for _ in range(8):
            dec.decode_step(1)
            toks.append(int(dec.tokens[0]))
        results[chunk] = (hidden, dec.kv[:, :, 0, :T].clone(), toks)
        del dec
    h0, kv0, t0 = results[4096]
    for chunk in (512, 64, 1):
        h, kv, t = results[chunk]
        assert_same_bits(h, h0, f"prefill outputs, chunk {chunk}")
        assert_same_bits(kv, kv0, f"KV cache, chunk {chunk}")
        assert t == t0, f"decode after chunk {chunk}: {t} vs {t0}"


def _fill_prompt_cache(dec, slot, req, length, shape):
    """Synthetic prompt state of request ``req``: KV ~N(0,1) for `length`
    positions (the same values whatever the slot)."""
    kv = synth.normal_bf16((shape.n_layers, 2, length, shape.n_kv, shape.head_dim), 1.0,
                           5000 + req, "cuda")
    dec.kv[:, :, slot, :length].copy_(kv)


def _decode_tokens(M, shape, w, reqs, lengths, steps, lmax):
    bsz = len(reqs)
    dec = M.Decoder(shape, w, max_batch=bsz, max_len=lmax)
    for i, r in enumerate(reqs):
        _fill_prompt_cache(dec, i, r, lengths[r], shape)
    dec.set_sampling([M.kinv.SamplingParams(seed=1000 + r) for r in reqs])
    hist = [synth.uniform_int(64, 0, shape.vocab - 1, 6000 + r).tolist() for r in reqs]
    dec.set_history(hist)
    dec.set_positions([lengths[r] for r in reqs])
    dec.tokens[:bsz] = torch.tensor([h[-1] for h in hist], dtype=torch.int32, device="cuda")
    toks, logits = [], []
    for _ in range(steps):
        dec.decode_step(bsz)
        toks.append(dec.tokens[:bsz].cpu().clone())
        logits.append(dec.logits[:bsz].clone())
    return torch.stack(toks, 1), torch.stack(logits, 1)


def test_tagged_request_alone_vs_cobatched(M):
    shape = _shape(M, 4)
    w = M.random_weights(shape, device="cuda")
    n_req = 40
    lengths = synth.uniform_int(n_req, 16, 4096, synth.SEED_LEN).tolist()
    lmax = max(lengths) + 16
    alone_t, alone_l = _decode_tokens(M, shape, w, [0], lengths, 12, lmax)
    for reqs in ([0] + list(range(1, 8)), list(range(39, 7, -1)) + [0], [5, 9, 0, 2]):
        t, l = _decode_tokens(M, shape, w, reqs, lengths, 12, lmax)
        slot = reqs.index(0)
        assert torch.equal(t[slot], alone_t[0]), f"tokens differ in batch {len(reqs)}"
        assert_same_bits(l[slot], alone_l[0], f"logits, batch of {len(reqs)}")


def _decode_tagged(M, shape, w, reqs, lengths, steps, lmax, tag=0):
    """Decode `steps` tokens for requests `reqs` (slot i holds request
    reqs[i]); returns every slot's tokens [bsz][steps] and the tagged
    request's logits at the first and last step."""
    bsz = len(reqs)
    dec = M.Decoder(shape, w, max_batch=bsz, max_len=lmax)
    for i, r in enumerate(reqs):
        _fill_prompt_cache(dec, i, r, lengths[r], shape)
    dec.set_sampling([M.kinv.SamplingParams(seed=1000 + r) for r in reqs])
    hist = [synth.uniform_int(64, 0, shape.vocab - 1, 6000 + r).tolist() for r in reqs]
    dec.set_history(hist)
    dec.set_positions([lengths[r] for r in reqs])
    dec.tokens[:bsz] = torch.tensor([h[-1] for h in hist], dtype=torch.int32, device="cuda")
    slot = reqs.index(tag)
    toks = torch.empty(bsz, steps, dtype=torch.int32, device="cuda")
    logits = []
    for s_ in range(steps):
        dec.decode_step(bsz)
        toks[:, s_] = dec.tokens[:bsz]
        if s_ in (0, steps - 1):
            logits.append(dec.logits[slot].clone())
    assert M.kinv.last_device_status() == 0
    out = toks.cpu(), torch.stack(logits)
    del dec
    torch.cuda.empty_cache()
    return out


def test_tagged_request_alone_vs_batches_of_128_and_256_over_256_tokens(M):
    """The busy-server check at the full batch range: request 0 decodes 256
    tokens alone, then among 127 and 255 other requests (prompt lengths
    U{16..4096}, each with its own seed) at a middle and at the last slot; its
    tokens and its logits bits are the same every time.  Two layers, full
    widths and vocabulary."""
    shape = _shape(M, 2)
    w = M.random_weights(shape, device="cuda")
    n_req = 256
    lengths = synth.uniform_int(n_req, 16, 4096, synth.SEED_LEN).tolist()
    steps = 256
    lmax = max(lengths) + steps + 8
    alone_t, alone_l = _decode_tagged(M, shape, w, [0], lengths, steps, lmax)
    perm = torch.randperm(n_req - 1, generator=synth.gen(44)).add(1).tolist()
    for reqs in (perm[:64] + [0] + perm[64:127], perm[:255] + [0]):
        t, l = _decode_tagged(M, shape, w, reqs, lengths, steps, lmax)
        slot = reqs.index(0)
        assert torch.equal(t[slot], alone_t[0]), f"tokens differ in a batch of {len(reqs)}"
        assert_same_bits(l, alone_l, f"logits, batch of {len(reqs)}")


def test_full_depth_alone_vs_cobatched(M):
    shape = M.QWEN3_8B
    w = M.random_weights(shape, device="cuda")
    lengths = [700, 33, 4000, 16, 1500, 2048, 257, 999]
    lmax = 4096 + 16
    alone_t, alone_l = _decode_tokens(M, shape, w, [0], lengths, 4, lmax)
    t, l = _decode_tokens(M, shape, w, [3, 1, 0, 7, 2, 6, 4, 5], lengths, 4, lmax)
    assert torch.equal(t[2], alone_t[0])
    assert_same_bits(l[2], alone_l[0], "logits at full depth")


@pytest.mark.parametrize("gains", [False, True], ids=["unit_gains", "random_gains"])
def test_every_stage_of_the_step_matches_the_oracle(M, gains):
    """Each kernel of a 2-layer 8B-shaped decode step, fed the GPU's own
    inputs for that stage, matches the oracle within the tolerance.  The
    RMSNorms are folded into the projections: the O and down projections add
    their output to the residual stream and leave per-tile sums of squares;
    the QKV and gate/up projections and the LM head scale their rows by
    1/rms (the oracle: the unrounded fp64 normalised row times W)."""
    from oracle import attention as oattn, glue as oglue
    from oracle.gemm import gemm as og, matmul as omm
    from oracle.rmsnorm import rmsnorm_f64
    from oracle.rope import rope as orope
    kinv = M.kinv
    shape = _shape(M, 2)
    w = M.random_weights(shape, device="cuda")
    if gains:
        _random_gains(w)
    B, L = 3, [16, 300, 1]
    dec = M.Decoder(shape, w, max_batch=B, max_len=512)
    for r in range(B):
        dec.kv[:, :, r, : L[r]].copy_(synth.normal_bf16((2, 2, L[r], 8, 128), 1.0, 5000 + r, "cuda"))
    dec.set_positions(L)
    dec.tokens[:B] = torch.tensor([5, 77, 151935], dtype=torch.int32, device="cuda")
    b = synth.bits

    from oracle.model import fold

    def normed(x_bits):
        return rmsnorm_f64(obf.to_f64(x_bits), np.ones(x_bits.shape[1]), 1e-6)

    def check_ss(x_bits, name):
        x = obf.to_f64(x_bits)
        ref = (x * x).reshape(B, -1, 128).sum(-1)
        assert np.allclose(dec.ss[:B].cpu().numpy(), ref, rtol=1e-5, atol=0), name

    x, ss = dec.x[:B], dec.ss[:B]
    kinv.embed(w["embed"], dec.tokens[:B], out=x)
    assert np.array_equal(b(x), oglue.embed(b(w["embed"]), [5, 77, 151935]))
    kinv.row_sumsq(x, ss)
    check_ss(b(x), "sums of squares of the embedding rows")
    for li in range(2):
        lw = w["layers"][li]
        x0 = b(x)
        kinv.gemm_fused(x, dec.w_qkv_f[li], kinv.norm_in(ss, 4096, 1e-6), out=dec.qkv[:B])
        assert_close(f64(dec.qkv[:B]), obf.to_f64(omm(normed(x0), fold(b(lw["w_qkv"]), b(lw["attn_norm"])))),
                     "qkv with the attention norm folded in")
        qkv = b(dec.qkv[:B]).reshape(B, 48, 128)
        kc, vc = dec.kv[li, 0], dec.kv[li, 1]
        kinv.rope_append(dec.qkv[:B], dec.q[:B], kc, vc, dec.seq[:B], dec.pos[:B], 32, 8, 128, 1e6,
                         lw["q_norm"], lw["k_norm"], 1e-6)
        pos = np.array(L)
        assert_close(f64(dec.q[:B]), obf.to_f64(orope(qkv[:, :32], pos, 1e6, b(lw["q_norm"]))), "rope q")
        rk = orope(qkv[:, 32:40], pos, 1e6, b(lw["k_norm"]))
        for r in range(B):
            assert_close(f64(kc[r, L[r]]), obf.to_f64(rk[r]), "rope k")
            assert np.array_equal(b(vc[r, L[r]]), qkv[r, 40:])
        kinv.attn_decode(dec.q[:B], kc[:B], vc[:B], dec.kv_len[:B], out=dec.attn[:B], workspace=dec.ws)
        ref = oattn.decode(b(dec.q[:B]), b(kc[:B]), b(vc[:B]), [n + 1 for n in L])
        assert_close(f64(dec.attn[:B]), obf.to_f64(ref), "attention")
        x1 = b(x)
        kinv.gemm_fused(dec.attn[:B].view(B, -1), lw["w_o"], kinv.residual_out(x, ss))
        o_ref = og(b(dec.attn[:B]).reshape(B, -1), b(lw["w_o"]), out="f64")
        assert_close(f64(x), obf.to_f64(oglue.add_f64(x1, o_ref)), "x + o")
        check_ss(b(x), "sums of squares after the O projection")
        x2 = b(x)
        kinv.gemm_swiglu(x, dec.w_gu_il[li], out=dec.act[:B], fusion=kinv.norm_in(ss, 4096, 1e-6))
        gu = omm(normed(x2), fold(b(lw["w_gu"]), b(lw["ffn_norm"])), out="f64")
        assert_close(f64(dec.act[:B]), obf.to_f64(oglue.swiglu_f64(gu)), "gate/up + swiglu, norm folded in")
        kinv.gemm_fused(dec.act[:B], lw["w_down"], kinv.residual_out(x, ss))
        d_ref = og(b(dec.act[:B]), b(lw["w_down"]), out="f64")
        assert_close(f64(x), obf.to_f64(oglue.add_f64(x2, d_ref)), "x + down")
        check_ss(b(x), "sums of squares after the down projection")
    xf = b(x)
    kinv.gemm_fused(x, dec.lm_head_f, kinv.norm_in(ss, 4096, 1e-6), out=dec.logits[:B])
    assert_close(f64(dec.logits[:B]), omm(normed(xf), fold(b(w["lm_head"]), b(w["final_norm"])), out="f64"),
                 "logits with the final norm folded in", atol=1e-4, rtol=1e-4)
    assert kinv.last_device_status() == 0


def _random_gains(w, seed=4242):
    """Replace every norm gain with bf16 values drawn from U(0.5, 1.5)."""
    g = synth.gen(seed)
    draw = lambda t: (0.5 + torch.rand(t.shape, generator=g)).to(torch.bfloat16).to(t.device)
    for lw in w["layers"]:
        for key in ("attn_norm", "ffn_norm", "q_norm", "k_norm"):
            if key in lw:
                lw[key] = draw(lw[key])
    w["final_norm"] = draw(w["final_norm"])


def _first_step(M, layers, lengths, gains=False):
    """One decode step of an 8B-shaped stack (full widths and vocabulary) for
    requests with synthetic prompt caches; returns the GPU's logits and final
    residual rows, the oracle's (its own end-to-end computation from the same
    weights, caches, tokens and settings), the GPU's sampled tokens, the
    histories, the settings and the oracle's near-tie flags."""
    from oracle import glue as oglue
    from oracle.gemm import matmul
    from oracle.model import fold, layer_step
    from oracle.rmsnorm import rmsnorm_f64
    from oracle.sampler import sample as osample
    shape = _shape(M, layers)
    w = M.random_weights(shape, device="cuda")
    if gains:
        _random_gains(w)
    bsz = len(lengths)
    lmax = max(lengths) + 16
    dec = M.Decoder(shape, w, max_batch=bsz, max_len=lmax)
    for r in range(bsz):
        dec.kv[:, :, r, : lengths[r]].copy_(
            synth.normal_bf16((layers, 2, lengths[r], 8, 128), 1.0, 5000 + r, "cuda"))
    hist = [synth.uniform_int(64, 0, shape.vocab - 1, 6000 + r).tolist() for r in range(bsz)]
    dec.set_sampling([M.kinv.SamplingParams(seed=1000 + r) for r in range(bsz)])
    dec.set_history(hist)
    dec.set_positions(lengths)
    dec.tokens[:bsz] = torch.tensor([h[-1] for h in hist], dtype=torch.int32, device="cuda")
    kv = synth.bits(dec.kv[:, :, :bsz])
    dec.decode_step(bsz)
    g_logits = f64(dec.logits[:bsz])
    g_hidden = f64(dec.x[:bsz])
    toks = dec.tokens[:bsz].cpu().tolist()
    assert M.kinv.last_device_status() == 0
    oshape = Shape(d_model=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, vocab=shape.vocab,
                   n_layers=layers, eps=1e-6, rope_base=1e6, qk_norm=True)
    x = oglue.embed(synth.bits(w["embed"]), [h[-1] for h in hist])
    for li in range(layers):
        lw = {k: synth.bits(v) for k, v in w["layers"][li].items()}
        x = layer_step(x, lw, kv[li, 0].copy(), kv[li, 1].copy(), [(b, lengths[b]) for b in range(bsz)], oshape)
    h = rmsnorm_f64(obf.to_f64(x), np.ones(x.shape[1]), 1e-6)
    o_logits = matmul(h, fold(synth.bits(w["lm_head"]), synth.bits(w["final_norm"])), out="f32").astype(np.float64)
    params = [OParams(seed=1000 + r) for r in range(bsz)]
    _, ties = osample(o_logits.astype(np.float32), hist, [0] * bsz, params)
    return g_logits, g_hidden, o_logits, obf.to_f64(x), toks, hist, params, ties


def test_first_step_one_layer_end_to_end_matches_oracle(M):
    """Embedding, one 8B-shaped layer, final norm, LM head and sampler, end to
    end against the oracle's own computation: every element of the final
    residual rows (bf16) and of all 2 x 151936 logits within the per-element
    tolerance, and the sampled token equal to the oracle sampler's on the
    GPU's logits."""
    from oracle.sampler import sample_row
    g_l, g_h, o_l, o_h, toks, hist, params, ties = _first_step(M, 1, [16, 300])
    assert_close(g_h, o_h, "final residual rows, one layer")
    assert_close(g_l, o_l, "logits, one layer")
    for r in range(2):
        t, near = sample_row(g_l[r].astype(np.float32), hist[r], 0, params[r])
        if not near:
            assert t == toks[r]


def test_first_step_one_layer_with_non_unit_gains(M):
    """The same end-to-end check with every norm gain drawn from U(0.5, 1.5):
    the attention, FFN and final gains are folded into the weights they feed
    (kinv_scale_columns, one bf16 rounding of W * g), the QK-norm gains are
    applied per head; the oracle applies every gain to the unrounded
    normalised rows."""
    g_l, g_h, o_l, o_h, toks, hist, params, ties = _first_step(M, 1, [16, 300], gains=True)
    assert_close(g_h, o_h, "final residual rows, non-unit gains")
    assert_close(g_l, o_l, "logits, non-unit gains")


def test_first_step_two_layers_within_the_rounding_noise(M):
    """Over two layers the GPU and the oracle round to bf16 at the same
    tensors, but a value that lies within fp32 accumulation error of a bf16
    rounding boundary rounds one way on each side; the one-unit differences
    feed the next layer and compound (an fp32-accumulating restatement of the
    oracle on the CPU, tests/test_oracle_noise_floor.py, shows the same spread).
    Each kernel is held to the per-element tolerance on its own inputs in
    test_every_stage_of_the_step_matches_the_oracle; end to end over two layers
    the check is the norm-relative error (<= 1e-2 per tensor) and the share of
    elements within the per-element bound: >= 99.9 % of the logits, >= 97 % of
    the final residual rows."""
    g_l, g_h, o_l, o_h, toks, hist, params, ties = _first_step(M, 2, [16, 300])
    for name, g, r, share in (("logits", g_l, o_l, 0.999), ("final residual rows", g_h, o_h, 0.97)):
        assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-2, name
        within = np.mean(np.abs(g - r) <= 2e-2 + 1e-2 * np.abs(r))
        assert within >= share, f"{name}: {within:.5f} of elements within the per-element bound"


def test_prefix_cache_reuse_gives_the_same_bits(M):
    """A request whose prompt starts with a cached prefix copies that prefix's
    keys and values and prefills only the rest: its KV cache and last hidden
    row equal those of prefilling the whole prompt at once (so everything
    decoded from them is the same too)."""
    shape = _shape(M, 2)
    w = M.random_weights(shape, device="cuda")
    prompt = synth.uniform_int(1000, 0, shape.vocab - 1, 90).cuda()
    n_pre = 700
    dec = M.Decoder(shape, w, max_batch=3, max_len=1100, max_chunk=1000)
    whole = dec.prefill(0, prompt)                       # slot 0: the whole prompt at once
    cache = M.PrefixCache(dec)
    dec.prefill(1, prompt[:n_pre], chunk=256)           # slot 1: the shared prefix, in chunks
    cache.insert(prompt[:n_pre].tolist(), 1)
    reused, last = cache.prefill(2, prompt, chunk=128)  # slot 2: prefix from the cache
    assert reused == n_pre
    assert_same_bits(last, whole, "last hidden row")
    assert_same_bits(dec.kv[:, :, 2, :1000], dec.kv[:, :, 0, :1000], "KV cache")
