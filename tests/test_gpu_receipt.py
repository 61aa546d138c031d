"""Receipt round trip (Kinetic "Receipts", *Verifying*): a tagged request's
receipt made while it shares a busy batch verifies as identical when the
request is rerun alone, the plainest way."""
import pytest
import torch

from helpers import ensure_lib, gpu, synth
from invariant_deterministic_gb300 import receipt

pytestmark = gpu


@pytest.fixture(scope="module")
def M():
    ensure_lib()
    from invariant_deterministic_gb300 import model
    return model


def test_receipt_from_busy_batch_verifies_alone(M):
    from test_gpu_model import _decode_tokens
    shape = M.ModelShape(**{**M.QWEN3_8B.__dict__, "n_layers": 4})
    w = M.random_weights(shape, device="cuda")
    lengths = synth.uniform_int(24, 16, 4096, synth.SEED_LEN + 5).tolist()
    lmax = max(lengths) + 40
    busy = [11, 3, 0, 17, 5, 23, 8, 1, 14, 20, 2, 9]
    toks, _ = _decode_tokens(M, shape, w, busy, lengths, 32, lmax)
    tag = busy.index(0)
    kinv = M.kinv
    prompt_ids = synth.uniform_int(64, 0, shape.vocab - 1, 6000).tolist()   # request 0's recorded tail
    p = kinv.SamplingParams(seed=1000)
    r = receipt.make_receipt(build_id=kinv.build_id(), device_class=kinv.device_class(),
                             settings={"split_len": 256, "rope_base": shape.rope_base,
                                       "qk_norm": shape.qk_norm, "layers": shape.n_layers},
                             prompt_ids=prompt_ids, sampling=p.__dict__,
                             output_ids=toks[tag].tolist())
    assert receipt.check_hashes(r)
    alone, _ = _decode_tokens(M, shape, w, [0], lengths, 32, lmax)
    verdict = receipt.compare(r, alone[0].tolist(), kinv.build_id(), kinv.device_class())
    assert verdict.startswith("identical, 32 of 32"), verdict
