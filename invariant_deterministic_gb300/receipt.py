"""Run records ("receipts") for the batch-invariant decode path.

A Kinetic receipt (Kinetic "Receipts", *Making a receipt*) records what makes
the output bits reproducible: the build that pins the kernels, the device
class, the settings that change bits, the exact prompt tokens, every sampler
setting and the seed, and the output tokens; token lists are hashed with
BLAKE3 over the ids as little-endian 32-bit integers.  *Verifying* reruns the
recorded prompt tokens the plainest way (one request, alone) and reports
"identical" or the first output token that differs.

This module holds the record: ``token_hash`` (BLAKE3 of LE int32 ids),
``make_receipt``, ``compare`` and ``verify``, which rebuilds the model from
the identity the record holds (shape and weight seed of the random-init
model), prefills the recorded prompt ids in one slot alone, decodes as many
tokens as were recorded with the recorded settings and seed, and compares.
Signing and model-file hashing are not part of it.

BLAKE3 is restated here from its published specification (O'Connor, Aumasson,
Neves, Wilcox-O'Hearn, "BLAKE3: one function, fast everywhere", 2020): a
Merkle tree of 1024-byte chunks, each chunk compressed in 64-byte blocks by a
7-round compression function on a 16-word state (the BLAKE2s G function and
the SHA-256 initial values), parents joining two chaining values.
"""
from __future__ import annotations

import json
import struct

_IV = (0x6A09E667, 0xBB67AE85, 0x3C6EF372, 0xA54FF53A,
       0x510E527F, 0x9B05688C, 0x1F83D9AB, 0x5BE0CD19)
_PERM = (2, 6, 3, 10, 7, 0, 4, 13, 1, 11, 12, 5, 9, 14, 15, 8)
_CHUNK_START, _CHUNK_END, _PARENT, _ROOT = 1, 2, 4, 8
_M = 0xFFFFFFFF
_BLOCK = 64
_CHUNK = 1024


def _rotr(x: int, n: int) -> int:
    return ((x >> n) | (x << (32 - n))) & _M


def _g(s, a, b, c, d, mx, my):
    s[a] = (s[a] + s[b] + mx) & _M
    s[d] = _rotr(s[d] ^ s[a], 16)
    s[c] = (s[c] + s[d]) & _M
    s[b] = _rotr(s[b] ^ s[c], 12)
    s[a] = (s[a] + s[b] + my) & _M
    s[d] = _rotr(s[d] ^ s[a], 8)
    s[c] = (s[c] + s[d]) & _M
    s[b] = _rotr(s[b] ^ s[c], 7)


def _compress(cv, block_words, counter: int, block_len: int, flags: int):
    s = list(cv) + list(_IV[:4]) + [counter & _M, (counter >> 32) & _M, block_len, flags]
    m = list(block_words)
    for r in range(7):
        _g(s, 0, 4, 8, 12, m[0], m[1])
        _g(s, 1, 5, 9, 13, m[2], m[3])
        _g(s, 2, 6, 10, 14, m[4], m[5])
        _g(s, 3, 7, 11, 15, m[6], m[7])
        _g(s, 0, 5, 10, 15, m[8], m[9])
        _g(s, 1, 6, 11, 12, m[10], m[11])
        _g(s, 2, 7, 8, 13, m[12], m[13])
        _g(s, 3, 4, 9, 14, m[14], m[15])
        if r < 6:
            m = [m[i] for i in _PERM]
    for i in range(8):
        s[i] ^= s[i + 8]
        s[i + 8] ^= cv[i]
    return s


def _words(block: bytes):
    return struct.unpack("<16I", block.ljust(_BLOCK, b"\0"))


class _Output:
    """The last compression of a node, held back so the root can be told."""

    def __init__(self, cv, words, counter, block_len, flags):
        self.cv, self.words, self.counter, self.block_len, self.flags = cv, words, counter, block_len, flags

    def chaining_value(self):
        return _compress(self.cv, self.words, self.counter, self.block_len, self.flags)[:8]

    def root_bytes(self, n: int = 32) -> bytes:
        out = b""
        i = 0
        while len(out) < n:
            s = _compress(self.cv, self.words, i, self.block_len, self.flags | _ROOT)
            out += struct.pack("<16I", *s)
            i += 1
        return out[:n]


def _chunk_output(data: bytes, chunk_index: int) -> _Output:
    cv = list(_IV)
    blocks = [data[i: i + _BLOCK] for i in range(0, len(data), _BLOCK)] or [b""]
    for j, blk in enumerate(blocks):
        flags = (_CHUNK_START if j == 0 else 0) | (_CHUNK_END if j == len(blocks) - 1 else 0)
        if j == len(blocks) - 1:
            return _Output(cv, _words(blk), chunk_index, len(blk), flags)
        cv = _compress(cv, _words(blk), chunk_index, _BLOCK, flags)[:8]
    raise AssertionError("unreachable")


def _parent_output(left_cv, right_cv) -> _Output:
    return _Output(list(_IV), list(left_cv) + list(right_cv), 0, _BLOCK, _PARENT)


def blake3(data: bytes, n: int = 32) -> bytes:
    """BLAKE3 hash (default mode, no key) of ``data``."""
    chunks = [data[i: i + _CHUNK] for i in range(0, len(data), _CHUNK)] or [b""]
    # chunk chaining values, merged pairwise the way the spec's incremental
    # hasher does: a stack of subtree CVs, joined when the count allows
    stack = []
    for idx, ch in enumerate(chunks[:-1]):
        cv = _chunk_output(ch, idx).chaining_value()
        total = idx + 1
        while total & 1 == 0:
            cv = _parent_output(stack.pop(), cv).chaining_value()
            total >>= 1
        stack.append(cv)
    out = _chunk_output(chunks[-1], len(chunks) - 1)
    while stack:
        out = _parent_output(stack.pop(), out.chaining_value())
    return out.root_bytes(n)


def token_hash(ids) -> str:
    """BLAKE3 over the ids as little-endian 32-bit integers, hex."""
    data = struct.pack(f"<{len(ids)}i", *[int(i) for i in ids])
    return blake3(data).hex()


def make_receipt(*, build_id: str, device_class: str, settings: dict, prompt_ids, sampling: dict,
                 output_ids, finish: str = "length", model: dict | None = None) -> dict:
    """A run record in the spirit of a Kinetic receipt (unsigned, no model
    file hash): enough to rerun the request and compare the tokens.  `model`
    names the weights (here: the shape and seed of the random-init model)."""
    return {
        "receipt": 1,
        "kinv": {"build": build_id},
        "model": dict(model) if model else None,
        "device": {"class": device_class, "settings": dict(settings)},
        "prompt": {"count": len(prompt_ids), "blake3": token_hash(prompt_ids),
                   "ids": [int(i) for i in prompt_ids]},
        "sampling": dict(sampling),
        "output": {"finish": finish, "tokens": {"count": len(output_ids),
                                                "blake3": token_hash(output_ids),
                                                "ids": [int(i) for i in output_ids]}},
    }


def check_hashes(receipt: dict) -> bool:
    """The recorded hashes match the recorded ids."""
    return (token_hash(receipt["prompt"]["ids"]) == receipt["prompt"]["blake3"]
            and token_hash(receipt["output"]["tokens"]["ids"]) == receipt["output"]["tokens"]["blake3"])


def compare(receipt: dict, rerun_ids, build_id: str, device_class: str) -> str:
    """'identical', or where the rerun first differs (and whether the build or
    device class differ, in which case a difference is expected)."""
    want = receipt["output"]["tokens"]["ids"]
    note = ""
    if receipt["kinv"]["build"] != build_id or receipt["device"]["class"] != device_class:
        note = " (build or device class differs from the receipt's: bits are promised only within one)"
    for i, (a, b) in enumerate(zip(want, rerun_ids)):
        if int(a) != int(b):
            return f"differs at output token {i}: receipt {a}, rerun {b}{note}"
    if len(want) != len(rerun_ids):
        return f"differs in length: receipt {len(want)}, rerun {len(rerun_ids)}{note}"
    return f"identical, {len(want)} of {len(want)} output tokens{note}"


def model_identity(shape, weight_seed: int) -> dict:
    """The model fields of a record: every ModelShape field and the seed the
    random-init weights are drawn with."""
    return {"shape": dict(shape.__dict__), "weight_seed": int(weight_seed),
            "init": "projections ~N(0, 0.02) bf16, norm gains 1"}


def settings_of(shape) -> dict:
    """The settings that change bits: the KV split length, the RoPE base,
    QK-norm, the RMSNorm eps and the prefill rule (all but the last prompt
    token prefilled, the last one decoded)."""
    from . import kinv
    return {"split_len": kinv.SPLIT_LEN, "rope_base": shape.rope_base, "qk_norm": shape.qk_norm,
            "eps": shape.eps, "prefill": "prompt[:-1], then decode from prompt[-1]"}


def verify(record: dict, device="cuda", chunk: int = 0) -> str:
    """Kinetic "Receipts", *Verifying*: rerun the recorded request the
    plainest way -- one slot, alone, prefill chunk `chunk` (0: whole) -- and
    report "identical" or the first differing output token.  Refuses a record
    whose hashes do not match its ids, or whose settings are not this
    library's."""
    if not check_hashes(record):
        return "refused: the recorded hashes do not match the recorded ids"
    if not record.get("model"):
        return "refused: the record does not identify the model"
    from . import kinv, model as M
    shape = M.ModelShape(**record["model"]["shape"])
    if dict(record["device"]["settings"]) != settings_of(shape):
        return "refused: the recorded settings are not this library's"
    w = M.random_weights(shape, seed=record["model"]["weight_seed"], device=device)
    prompt = record["prompt"]["ids"]
    n_out = record["output"]["tokens"]["count"]
    dec = M.Decoder(shape, w, max_batch=1, max_len=len(prompt) + n_out + 8,
                    max_chunk=chunk or max(len(prompt) - 1, 1), device=device)
    s = dict(record["sampling"])
    if s.get("logit_bias"):
        s["logit_bias"] = {int(k): float(v) for k, v in s["logit_bias"].items()}
    out = M.run_requests(dec, [prompt], [kinv.SamplingParams(**s)], n_out, chunk=chunk)
    return compare(record, out[0], kinv.build_id(), kinv.device_class())


def dumps(receipt: dict) -> str:
    return json.dumps(receipt, separators=(",", ":"), sort_keys=False)
