"""Run records: BLAKE3 token hashes pinned to the values a Kinetic receipt
prints, and the record / compare logic."""
import json
import os

from invariant_deterministic_gb300 import receipt

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "receipt_tokens.json")


def test_token_hashes_match_the_printed_receipt():
    g = json.load(open(GOLDEN))
    assert receipt.token_hash(g["prompt_ids"]) == g["prompt_blake3"]
    assert receipt.token_hash(g["output_ids"]) == g["output_blake3"]
    # little-endian int32 matters: another byte order gives another hash
    import struct
    be = struct.pack(f">{len(g['prompt_ids'])}i", *g["prompt_ids"])
    assert receipt.blake3(be).hex() != g["prompt_blake3"]


def test_blake3_tree_is_consistent_across_chunk_boundaries():
    # the tree path (more than one 1024-byte chunk) is exercised for
    # determinism and sensitivity; no published vector is available here
    data = bytes(range(256)) * 20
    h = receipt.blake3(data)
    assert h == receipt.blake3(bytes(data))
    assert len({receipt.blake3(data[:n]) for n in (1023, 1024, 1025, 2048, 2049, 4096, 5120)}) == 7
    assert receipt.blake3(data[:3072]) != receipt.blake3(data[:3071] + b"\x01")


def test_make_and_compare():
    g = json.load(open(GOLDEN))
    r = receipt.make_receipt(build_id="abc", device_class="cuda-sm103a",
                             settings={"split_len": 256}, prompt_ids=g["prompt_ids"],
                             sampling={"temperature": 0.8, "seed": 42}, output_ids=g["output_ids"])
    assert r["prompt"]["blake3"] == g["prompt_blake3"]
    assert receipt.check_hashes(r)
    assert receipt.compare(r, g["output_ids"], "abc", "cuda-sm103a").startswith("identical, 18 of 18")
    bad = list(g["output_ids"])
    bad[5] += 1
    assert receipt.compare(r, bad, "abc", "cuda-sm103a").startswith("differs at output token 5")
    assert "build or device class differs" in receipt.compare(r, g["output_ids"], "xyz", "cuda-sm103a")
    r2 = json.loads(receipt.dumps(r))
    r2["output"]["tokens"]["ids"][0] = 1
    assert not receipt.check_hashes(r2)


def _blake3_recursive(data: bytes) -> bytes:
    """A second BLAKE3 (default hash mode, 32-byte output), written from the
    published specification in another shape than the package's: the tree is
    built top-down (the left subtree holds the largest power-of-two number of
    1 KiB chunks that leaves at least one for the right), not with the
    incremental stack of chaining values."""
    mask = 0xFFFFFFFF
    iv = (0x6A09E667, 0xBB67AE85, 0x3C6EF372, 0xA54FF53A, 0x510E527F, 0x9B05688C, 0x1F83D9AB, 0x5BE0CD19)
    perm = (2, 6, 3, 10, 7, 0, 4, 13, 1, 11, 12, 5, 9, 14, 15, 8)
    start, end, parent, root = 1, 2, 4, 8

    def rot(x, n):
        return ((x >> n) | (x << (32 - n))) & mask

    def mix(v, a, b, c, d, x, y):
        v[a] = (v[a] + v[b] + x) & mask
        v[d] = rot(v[d] ^ v[a], 16)
        v[c] = (v[c] + v[d]) & mask
        v[b] = rot(v[b] ^ v[c], 12)
        v[a] = (v[a] + v[b] + y) & mask
        v[d] = rot(v[d] ^ v[a], 8)
        v[c] = (v[c] + v[d]) & mask
        v[b] = rot(v[b] ^ v[c], 7)

    def compress(cv, block: bytes, counter: int, flags: int):
        n = len(block)
        m = list(int.from_bytes(block.ljust(64, b"\0")[4 * i: 4 * i + 4], "little") for i in range(16))
        v = list(cv) + list(iv[:4]) + [counter & mask, counter >> 32, n, flags]
        for r in range(7):
            if r:
                m = [m[p] for p in perm]
            for i, (a, b, c, d) in enumerate(((0, 4, 8, 12), (1, 5, 9, 13), (2, 6, 10, 14), (3, 7, 11, 15),
                                              (0, 5, 10, 15), (1, 6, 11, 12), (2, 7, 8, 13), (3, 4, 9, 14))):
                mix(v, a, b, c, d, m[2 * i], m[2 * i + 1])
        return [v[i] ^ v[i + 8] for i in range(8)]

    def chunk_cv(chunk: bytes, index: int, is_root: bool):
        blocks = [chunk[i: i + 64] for i in range(0, len(chunk), 64)] or [b""]
        cv = iv
        for j, blk in enumerate(blocks):
            f = (start if j == 0 else 0) | (end if j == len(blocks) - 1 else 0)
            if is_root and j == len(blocks) - 1:
                f |= root
            cv = compress(cv, blk, index, f)
        return cv

    def subtree(chunks, first: int, is_root: bool):
        if len(chunks) == 1:
            return chunk_cv(chunks[0], first, is_root)
        left = 1
        while left * 2 < len(chunks):
            left *= 2
        lcv = subtree(chunks[:left], first, False)
        rcv = subtree(chunks[left:], first + left, False)
        block = b"".join(w.to_bytes(4, "little") for w in lcv + rcv)
        return compress(iv, block, 0, parent | (root if is_root else 0))

    chunks = [data[i: i + 1024] for i in range(0, len(data), 1024)] or [b""]
    return b"".join(w.to_bytes(4, "little") for w in subtree(chunks, 0, True))


def test_blake3_agrees_with_an_independent_tree_implementation():
    """The package's incremental BLAKE3 against the top-down one above, over
    every tree shape up to 17 chunks (inputs that end inside, at and just
    after chunk and block boundaries) and token-id inputs of the lengths the
    run records hash (prompts of up to 4,096 ids are 16 KiB)."""
    import random
    rng = random.Random(7)
    data = bytes(rng.randrange(256) for _ in range(17 * 1024 + 100))
    lengths = {0, 1, 63, 64, 65, 1023, 1024, 1025, 17 * 1024 + 100}
    for c in range(1, 18):
        lengths |= {c * 1024 - 1, c * 1024, c * 1024 + 1, c * 1024 + 64, c * 1024 + 700}
    for n in sorted(lengths):
        assert receipt.blake3(data[:n]) == _blake3_recursive(data[:n]), n
    g = json.load(open(GOLDEN))
    assert _blake3_recursive(bytes.fromhex("")).hex() == receipt.blake3(b"").hex()
    # the printed single-chunk receipt hashes pin this implementation too
    import struct
    assert _blake3_recursive(struct.pack(f"<{len(g['prompt_ids'])}i", *g["prompt_ids"])).hex() == g["prompt_blake3"]
    ids = [rng.randrange(151936) for _ in range(4096)]
    for n in (256, 257, 1000, 4096):
        assert receipt.token_hash(ids[:n]) == _blake3_recursive(struct.pack(f"<{n}i", *ids[:n])).hex()
