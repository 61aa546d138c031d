"""Failure detection on the device without a fault: every device-side wait
in the kernels is bounded, gives up, records KINV_ERR_TIMEOUT in the status
word and lets its block exit.  kinv_test_bounded_wait runs that wait against
a barrier nothing completes, with a short limit; the context must stay usable
and the status must come back through kinv_last_device_status."""
import time

import pytest
import torch

from helpers import ensure_lib, gpu, synth

pytestmark = gpu


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


def test_bounded_wait_gives_up_and_reports_timeout(kinv):
    assert kinv.last_device_status() == 0
    t0 = time.perf_counter()
    kinv.test_bounded_wait(1_000_000)  # 1 ms
    assert kinv.last_device_status() == kinv.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the status word was cleared by the read, and the context still works
    assert kinv.last_device_status() == 0
    a = synth.normal_bf16((4, 256), 1.0, 3, "cuda")
    w = synth.normal_bf16((128, 256), 0.02, 4, "cuda")
    c = kinv.gemm(a, w)
    ref = (a.float() @ w.float().T)
    assert torch.allclose(c.float(), ref, atol=2e-2, rtol=1e-2)
    assert kinv.last_device_status() == 0


def test_bounded_wait_limit_is_checked_on_the_host(kinv):
    for bad in (0, 999, 100_000_001, -5):
        with pytest.raises(kinv.KinvError) as e:
            kinv.test_bounded_wait(bad)
        assert e.value.status == kinv.ERR_INVALID_ARG
