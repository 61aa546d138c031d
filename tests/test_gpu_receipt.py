"""Receipt round trip (Kinetic "Receipts", *Verifying*): a request served in a
busy batch of 64, from a real prompt prefill, gets a receipt that names the
model (shape and weight seed), the settings, the prompt ids, the sampler
settings and seed and the output ids; verify() rebuilds the model from the
record and reruns the request alone, the plainest way, and finds it
identical -- with any prefill chunking.  A record with a changed seed is
reported at the first differing token, one with a wrong hash is refused."""
import json

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
    kinv = M.kinv
    shape = M.ModelShape(**{**M.QWEN3_8B.__dict__, "n_layers": 4})
    seed = 0
    w = M.random_weights(shape, seed=seed, device="cuda")
    n_req, steps = 64, 24
    lens = synth.uniform_int(n_req, 16, 600, synth.SEED_LEN + 11).tolist()
    prompts = [synth.uniform_int(n, 0, shape.vocab - 1, 7000 + i).tolist() for i, n in enumerate(lens)]
    params = [kinv.SamplingParams(seed=1000 + i) for i in range(n_req)]
    dec = M.Decoder(shape, w, max_batch=n_req, max_len=max(lens) + steps + 8, max_chunk=256)
    outs = M.run_requests(dec, prompts, params, steps, chunk=256)
    assert kinv.last_device_status() == 0
    del dec, w
    torch.cuda.empty_cache()
    tag = 37
    r = receipt.make_receipt(build_id=kinv.build_id(), device_class=kinv.device_class(),
                             settings=receipt.settings_of(shape), prompt_ids=prompts[tag],
                             sampling=params[tag].__dict__, output_ids=outs[tag],
                             model=receipt.model_identity(shape, seed))
    r = json.loads(receipt.dumps(r))      # the record as stored
    assert receipt.check_hashes(r)
    assert receipt.verify(r).startswith(f"identical, {steps} of {steps}")
    assert receipt.verify(r, chunk=7).startswith(f"identical, {steps} of {steps}")
    # another seed draws other tokens: reported at the first difference
    r2 = json.loads(json.dumps(r))
    r2["sampling"]["seed"] += 1
    assert receipt.verify(r2).startswith("differs at output token")
    # a record whose ids do not match its hashes is refused
    r3 = json.loads(json.dumps(r))
    r3["prompt"]["ids"][0] ^= 1
    assert receipt.verify(r3).startswith("refused")
