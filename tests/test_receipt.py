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
