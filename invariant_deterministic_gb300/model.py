"""Decoder drivers over the kinv C ABI: a pre-norm decoder (RMSNorm, QKV GEMM,
RoPE + KV append, split-KV attention, O GEMM, residual RMSNorm, gate/up GEMM,
SwiGLU, down GEMM), an untied LM head and the seeded sampler.

Every arithmetic step is a kinv kernel; this module only owns buffers and
issues the calls in order on the current CUDA stream, so a whole decode step
can be captured into a CUDA graph.  Kernels per layer: the QKV projection
(with RoPE and the KV append for 2..64 rows), split-KV attention (split and
merge), the O projection, the gate/up projection with SwiGLU, the down
projection.  The RMSNorms are folded into the projections (kinv_gemm_fusion):
the O and down projections add their output to the residual stream x and
leave per-tile sums of squares of the new rows; the QKV and gate/up
projections and the LM head scale their rows by 1/rms, with the norm gains
folded into their weight columns once.

Layouts (all bf16 unless noted):
  embed, lm_head [V][d]; per layer w_qkv [(Hq + 2 Hkv) D][d], w_o [d][Hq D],
  w_gu [2F][d] (gate rows then up rows; the decoder keeps a copy interleaved
  in blocks of 64 for the fused gate/up + SwiGLU GEMM), w_down [d][F], norm
  gains [d] / [D];
  KV cache [layers][2][B][Lmax][Hkv][D] (k then v), token-major per sequence.
"""
from __future__ import annotations

import contextlib
from dataclasses import dataclass

import numpy as np
import torch

from . import kinv, synth


@dataclass
class ModelShape:
    d_model: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    n_layers: int
    eps: float = 1e-6
    rope_base: float = 1e4
    qk_norm: bool = False

    @property
    def qkv_dim(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim


TINY = ModelShape(d_model=256, n_q=4, n_kv=2, head_dim=64, ffn=512, vocab=512, n_layers=1,
                  rope_base=1e4, qk_norm=False)
# Qwen3-8B-shaped: 36 layers, d 4096, 32 query / 8 kv heads of 128, FFN 12288,
# vocab 151936; QK-norm on; RoPE base 1e6.
QWEN3_8B = ModelShape(d_model=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, vocab=151936,
                      n_layers=36, rope_base=1e6, qk_norm=True)


def random_weights(shape: ModelShape, seed: int = synth.SEED_WEIGHTS, device="cuda",
                   with_head: bool = True) -> dict:
    """Projections ~N(0, 0.02) bf16, gains 1 (drawn with seeded generators on
    ``device``)."""
    w = {"layers": [synth.layer_weights(shape.d_model, shape.n_q, shape.n_kv, shape.head_dim,
                                        shape.ffn, seed * 1000 + li, shape.qk_norm, device)
                    for li in range(shape.n_layers)]}
    if with_head:
        w["embed"] = synth.normal_bf16((shape.vocab, shape.d_model), 0.02, seed * 1000 + 997, device)
        w["lm_head"] = synth.normal_bf16((shape.vocab, shape.d_model), 0.02, seed * 1000 + 998, device)
        w["final_norm"] = torch.ones(shape.d_model, dtype=torch.bfloat16, device=device)
    return w


def fold_gain(w: torch.Tensor, g: torch.Tensor) -> torch.Tensor:
    """bf16(W * g) over the input columns (kinv_scale_columns), the RMSNorm
    gain moved into the projection it feeds; W itself when every gain is 1
    (the product would return W's bits)."""
    if bool(torch.all(g == 1)):
        return w
    return kinv.scale_columns(w, g)


# From 2 to this many rows the QKV projection runs with RoPE and the KV append
# in its epilogue (kinv_gemm_qkv_rope); otherwise kinv_gemm then
# kinv_rope_append (measured faster at one row and at many).  Both give the
# same bits, so the choice never changes a result.
FUSED_ROPE_MIN_ROWS = 2
FUSED_ROPE_MAX_ROWS = 64


class Decoder:
    """Owns weights, the KV cache and every activation buffer for up to
    ``max_batch`` sequences of up to ``max_len`` tokens (and prefill chunks of
    up to ``max_chunk`` rows)."""

    def __init__(self, shape: ModelShape, weights: dict, max_batch: int, max_len: int,
                 max_chunk: int = 0, device="cuda"):
        self.s = shape
        self.w = weights
        self.B = max_batch
        self.Lmax = max_len
        self.dev = torch.device(device)
        s = shape
        rows = max(max_batch, max_chunk)
        self.max_rows = rows
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        self.kv = torch.zeros(s.n_layers, 2, max_batch, max_len, s.n_kv, s.head_dim, **bf)
        self.x = torch.zeros(rows, s.d_model, **bf)
        self.qkv = torch.zeros(rows, s.qkv_dim, **bf)
        self.q = torch.zeros(rows, s.n_q, s.head_dim, **bf)
        self.attn = torch.zeros(rows, s.n_q, s.head_dim, **bf)
        # norm gains folded into the projections they feed; gate/up weights in
        # the interleaved layout of kinv_gemm_swiglu
        self.w_qkv_f = [fold_gain(lw["w_qkv"], lw["attn_norm"]) for lw in weights["layers"]]
        self.w_gu_il = [kinv.interleave_gate_up(fold_gain(lw["w_gu"], lw["ffn_norm"]))
                        for lw in weights["layers"]]
        if "lm_head" in weights:
            self.lm_head_f = fold_gain(weights["lm_head"], weights["final_norm"])
        self.act = torch.zeros(rows, s.ffn, **bf)
        # per-row sums of squares of the residual stream over 128-column tiles
        self.ss = torch.zeros(rows, s.d_model // 128, dtype=torch.float32, device=self.dev)
        ws = kinv.attn_decode_workspace(max_batch, s.n_q, s.head_dim, max_len)
        if max_chunk:
            ws = max(ws, kinv.attn_prefill_workspace(max_chunk, s.n_q, s.head_dim, max_len))
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.dev)
        i32 = dict(dtype=torch.int32, device=self.dev)
        # decode state: row b is sequence b at position pos[b]; attention sees pos[b] + 1 keys
        self.seq = torch.arange(max_batch, **i32)
        self.pos = torch.zeros(max_batch, **i32)
        self.kv_len = torch.ones(max_batch, **i32)
        if "lm_head" in weights:
            self.logits = torch.zeros(max_batch, s.vocab, dtype=torch.float32, device=self.dev)
        self.tokens = torch.zeros(max_batch, **i32)
        self.hist_ld = 64
        self.history = torch.zeros(max_batch, self.hist_ld, **i32)
        self.hist_len = torch.zeros(max_batch, **i32)
        self.step = torch.zeros(max_batch, dtype=torch.int64, device=self.dev)
        self.params = torch.zeros(max_batch * synth.SAMPLING_DTYPE.itemsize, dtype=torch.uint8,
                                  device=self.dev)
        # optional per-call timing: name -> list of (start, end) CUDA events
        self.timer = None

    def _t(self, name: str):
        """Brackets one kernel call with CUDA events on the current stream
        when a timer dict is installed (used by the benchmark only)."""
        if self.timer is None:
            return contextlib.nullcontext()
        return _EventPair(self.timer, name)

    # ------------------------------------------------------------ state setup
    def set_sampling(self, params_list) -> None:
        entries, _ = synth.bias_entries(params_list)
        # the logit-bias entries the packed settings point to (kept while in use)
        self.bias = (torch.from_numpy(entries.view(np.uint8).copy()).to(self.dev)
                     if len(entries) else None)
        packed = synth.sampling_struct(params_list, self.bias.data_ptr() if self.bias is not None else 0)
        self.params[: packed.nbytes].copy_(torch.from_numpy(packed.view(np.uint8)))

    def set_positions(self, pos) -> None:
        """pos[b]: index of the token to decode next (= tokens already cached)."""
        p = torch.as_tensor(pos, dtype=torch.int32)
        self.pos[: len(p)].copy_(p)
        self.kv_len[: len(p)].copy_(p + 1)

    def set_history(self, hist_rows) -> None:
        """hist_rows[b]: the request's tokens so far (prompt and output)."""
        for b, row in enumerate(hist_rows):
            tail = list(row)[-self.hist_ld:]
            self.history[b, : len(tail)] = torch.tensor(tail, dtype=torch.int32)
            self.hist_len[b] = len(tail)

    # --------------------------------------------------------------- a layer
    def layer(self, li: int, rows: int, seq, pos, attention) -> None:
        """One decoder layer on rows [0, rows): ``x`` holds the residual stream
        and ``ss`` its per-tile sums of squares; row r is sequence seq[r] at
        position pos[r].  Leaves the updated stream and sums in place."""
        s, lw = self.s, self.w["layers"][li]
        x = self.x[:rows]
        norm_in = kinv.norm_in(self.ss[:rows], s.d_model, s.eps)
        kc, vc = self.kv[li, 0], self.kv[li, 1]
        qn = lw.get("q_norm") if s.qk_norm else None
        kn = lw.get("k_norm") if s.qk_norm else None
        if FUSED_ROPE_MIN_ROWS <= rows <= FUSED_ROPE_MAX_ROWS:
            # the QKV projection with RoPE and the KV append in its epilogue
            with self._t("gemm_qkv"):
                kinv.gemm_qkv_rope(x, self.w_qkv_f[li], self.q[:rows], kc, vc, seq, pos, s.n_q, s.n_kv,
                                   s.head_dim, s.rope_base, qn, kn, s.eps, fusion=norm_in)
        else:
            # the same bits in two kernels (faster when many rows share a tile)
            with self._t("gemm_qkv"):
                kinv.gemm_fused(x, self.w_qkv_f[li], norm_in, out=self.qkv[:rows])
            with self._t("rope_append"):
                kinv.rope_append(self.qkv[:rows], self.q[:rows], kc, vc, seq, pos, s.n_q, s.n_kv,
                                 s.head_dim, s.rope_base, qn, kn, s.eps)
        attention(li, rows, kc, vc)
        with self._t("gemm_o"):
            kinv.gemm_fused(self.attn[:rows].view(rows, -1), lw["w_o"],
                            kinv.residual_out(x, self.ss[:rows]))
        with self._t("gemm_gate_up"):
            kinv.gemm_swiglu(x, self.w_gu_il[li], out=self.act[:rows], fusion=norm_in)
        with self._t("gemm_down"):
            kinv.gemm_fused(self.act[:rows], lw["w_down"], kinv.residual_out(x, self.ss[:rows]))

    # ---------------------------------------------------------------- decode
    def decode_layers(self, bsz: int) -> None:
        """All layers for one new token of sequences 0..bsz-1 (rows = bsz);
        the token's hidden state must be in x; leaves the final residual
        pieces in x and delta."""
        def attention(li, rows, kc, vc):
            with self._t("attn_decode"):
                kinv.attn_decode(self.q[:rows], kc[:rows], vc[:rows], self.kv_len[:rows],
                                 out=self.attn[:rows], workspace=self.ws)
        with self._t("row_sumsq"):
            kinv.row_sumsq(self.x[:bsz], self.ss[:bsz])
        for li in range(self.s.n_layers):
            self.layer(li, bsz, self.seq[:bsz], self.pos[:bsz], attention)

    def decode_step(self, bsz: int, sample: bool = True) -> None:
        """Embed tokens[:bsz], run every layer, the final norm, the LM head
        and (optionally) the sampler, then advance positions and histories.
        The sampled ids land in ``tokens`` (they are the next step's input)."""
        s = self.s
        with self._t("embed"):
            kinv.embed(self.w["embed"], self.tokens[:bsz], out=self.x[:bsz])
        self.decode_layers(bsz)
        with self._t("gemm_lm_head"):  # with the final RMSNorm folded in
            kinv.gemm_fused(self.x[:bsz], self.lm_head_f, kinv.norm_in(self.ss[:bsz], s.d_model, s.eps),
                            out=self.logits[:bsz])
        if sample:
            with self._t("sample"):
                kinv.sample(self.logits[:bsz], self.params, self.history[:bsz],
                            self.hist_len[:bsz], self.step[:bsz], out=self.tokens[:bsz])
            with self._t("decode_advance"):
                kinv.decode_advance(self.tokens[:bsz], self.history[:bsz], self.hist_len[:bsz],
                                    self.step[:bsz], pos=self.pos[:bsz], kv_len=self.kv_len[:bsz])

    # --------------------------------------------------------------- prefill
    def prefill_chunk(self, seq: int, p0: int, rows: int) -> None:
        """All layers for rows [0, rows) of x, which hold tokens p0..p0+rows-1
        of sequence ``seq``; their keys and values go into the cache."""
        i32 = dict(dtype=torch.int32, device=self.dev)
        seq_t = torch.full((rows,), seq, **i32)
        pos_t = torch.arange(p0, p0 + rows, **i32)
        q_start = torch.tensor([p0], **i32)
        q_len = torch.tensor([rows], **i32)
        q_off = torch.zeros(1, **i32)

        def attention(li, n, kc, vc):
            # a one-sequence view of the cache keeps the sequence index at 0
            with self._t("attn_prefill"):
                kinv.attn_prefill(self.q[:n], kc[seq: seq + 1], vc[seq: seq + 1], q_start, q_len,
                                  q_off, n, p0 + n, out=self.attn[:n], workspace=self.ws)
        kinv.row_sumsq(self.x[:rows], self.ss[:rows])
        for li in range(self.s.n_layers):
            self.layer(li, rows, seq_t, pos_t, attention)

    def prefill(self, seq: int, tokens: torch.Tensor, p0: int = 0, chunk: int = 0) -> torch.Tensor:
        """Prefill ``tokens`` (int32, device) as positions p0.. of sequence
        ``seq`` in chunks of ``chunk`` rows (0: as large as the buffers allow);
        returns the last row's final residual stream (a copy).  Any chunking
        gives the same bits (the kernels' per-row arithmetic does not depend
        on the rows beside it)."""
        n = int(tokens.shape[0])
        chunk = chunk or self.max_rows
        for c0 in range(0, n, chunk):
            rows = min(chunk, n - c0)
            kinv.embed(self.w["embed"], tokens[c0: c0 + rows], out=self.x[:rows])
            self.prefill_chunk(seq, p0 + c0, rows)
        return self.x[rows - 1].clone()

    def copy_prefix(self, src: int, dst: int, n: int) -> None:
        """Sequence dst takes sequence src's cached keys and values for
        positions 0..n-1 (every layer): a cached prompt prefix, reused."""
        self.kv[:, :, dst, :n].copy_(self.kv[:, :, src, :n])

    def close_residual(self, rows: int) -> torch.Tensor:
        """The last layer's output for rows [0, rows) (the residual stream;
        every layer already added its projections to it)."""
        return self.x[:rows]


def run_requests(dec: Decoder, prompts, params, steps: int, chunk: int = 0):
    """Serve requests together: request i takes slot i; its prompt, all but
    the last token, is prefilled into the slot (chunks of `chunk` rows, 0 =
    as large as the buffers allow), then every request decodes `steps` tokens
    in one batch, starting from its last prompt token, with its own sampler
    settings (repeat window over its prompt and output so far; Philox counter
    = its own output index).  Returns each request's output ids.  A
    request's tokens do not depend on the other requests, the slot or the
    chunking, so a rerun alone reproduces them."""
    bsz = len(prompts)
    if bsz > dec.B:
        raise ValueError("more requests than the decoder's slots")
    for i, p in enumerate(prompts):
        if len(p) < 1 or len(p) + steps > dec.Lmax:
            raise ValueError("prompt empty or too long for the decoder's cache")
        if len(p) > 1:
            dec.prefill(i, torch.tensor(list(p[:-1]), dtype=torch.int32, device=dec.dev), chunk=chunk)
    dec.set_sampling(params)
    dec.set_history([list(p) for p in prompts])
    dec.set_positions([len(p) - 1 for p in prompts])
    dec.step[:bsz] = 0
    dec.tokens[:bsz] = torch.tensor([int(p[-1]) for p in prompts], dtype=torch.int32, device=dec.dev)
    out = torch.empty(bsz, steps, dtype=torch.int32, device=dec.dev)
    for k in range(steps):
        dec.decode_step(bsz)
        out[:, k] = dec.tokens[:bsz]
    return out.cpu().tolist()


class _EventPair:
    def __init__(self, timer: dict, name: str):
        self.timer, self.name = timer, name

    def __enter__(self):
        self.a = torch.cuda.Event(enable_timing=True)
        self.b = torch.cuda.Event(enable_timing=True)
        self.a.record()
        return self

    def __exit__(self, *exc):
        self.b.record()
        self.timer.setdefault(self.name, []).append((self.a, self.b))
        return False


class PrefixCache:
    """Host-side index of prompt prefixes whose keys and values sit in a
    Decoder's cache.  The cached rows of a prefix are a function of its tokens
    alone (batch- and chunk-invariant kernels, causal attention), so a new
    request sharing the prefix can copy them instead of recomputing them and
    gets the same bits."""

    def __init__(self, dec: Decoder):
        self.dec = dec
        self.entries = {}  # tuple(tokens) -> slot

    def insert(self, tokens, slot: int) -> None:
        self.entries[tuple(int(t) for t in tokens)] = slot

    def longest(self, tokens):
        """(slot, n): the longest registered prefix of ``tokens``, or (None, 0)."""
        toks = tuple(int(t) for t in tokens)
        best = (None, 0)
        for key, slot in self.entries.items():
            n = len(key)
            if best[1] < n <= len(toks) and toks[:n] == key:
                best = (slot, n)
        return best

    def prefill(self, slot: int, tokens: torch.Tensor, chunk: int = 0) -> tuple[int, torch.Tensor]:
        """Prefill ``tokens`` into ``slot``, starting from the longest cached
        prefix; returns (reused positions, last row's final residual)."""
        src, n = self.longest(tokens.tolist())
        if src is not None and n == tokens.shape[0]:
            n -= 1  # recompute the last token: its hidden state is the output
        if src is not None and n > 0 and src != slot:
            self.dec.copy_prefix(src, slot, n)
        return n, self.dec.prefill(slot, tokens[n:], p0=n, chunk=chunk)
