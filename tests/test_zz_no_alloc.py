"""kinv_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory (a plug-in whose host owns all device memory through its own
pool, a real-time loop that must not take the allocator's implicit device
synchronisation, a binding without a device allocator).  Its partials live in a
scratch array compiled into the library instead of a caller workspace.

Checked here through the C ABI against kinv_attn_decode (caller workspace) on
two calls in a row, within the tests' tolerance and bit for bit, and for the
size limit.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import pytest
import torch

from helpers import assert_close, assert_same_bits, ensure_lib, f64, gpu, synth

pytestmark = gpu


@pytest.fixture(scope="module")
def kinv():
    return ensure_lib()


def _call_noalloc(kinv, q, k, v, kv_len, out):
    """Straight through the C entry point (ctypes), no Python wrapper."""
    bsz, hq, d = q.shape
    lmax, hkv = k.shape[1], k.shape[2]
    fn = kinv.lib().kinv_attn_decode_noalloc
    return fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
              k.stride(0), k.stride(1), ctypes.c_void_p(kv_len.data_ptr()), ctypes.c_void_p(out.data_ptr()),
              bsz, hq, hkv, d, lmax, 256, 0.0,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_path_twice(kinv):
    hq, hkv, d, lmax = 32, 8, 128, 4352
    for call, (bsz, seed) in enumerate([(8, 90), (5, 91)]):
        k = synth.normal_bf16((bsz, lmax, hkv, d), 1.0, seed, "cuda")
        v = synth.normal_bf16((bsz, lmax, hkv, d), 1.0, seed + 10, "cuda")
        q = synth.normal_bf16((bsz, hq, d), 1.0, seed + 20, "cuda")
        kv_len = synth.uniform_int(bsz, 0, lmax, seed + 30).cuda()
        ref = kinv.attn_decode(q, k, v, kv_len)
        got = torch.full_like(q, float("nan"))
        assert _call_noalloc(kinv, q, k, v, kv_len, got) == kinv.OK
        torch.cuda.synchronize()
        assert_close(f64(got), f64(ref), f"no-alloc call {call + 1}")
        assert_same_bits(got, ref, f"no-alloc call {call + 1}")
        # the Python wrapper reaches the same entry point with the same bits
        wrapped = torch.full_like(q, float("nan"))
        kinv.attn_decode_noalloc(q, k, v, kv_len, wrapped)
        assert_same_bits(wrapped, got, f"wrapper, call {call + 1}")
    assert kinv.last_device_status() == 0
    with pytest.raises(TypeError):
        kinv.attn_decode_noalloc(q, k, v, kv_len, torch.empty(q.shape, dtype=torch.float32, device="cuda"))


def test_noalloc_rejects_sizes_beyond_its_scratch(kinv):
    bsz, hq, hkv, d, lmax = 64, 32, 8, 128, 32768
    need = kinv.attn_decode_workspace(bsz, hq, d, lmax)
    assert need > kinv.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(bsz, hq, d, dtype=torch.bfloat16, device="cuda")
    # one sequence's worth of cache seen by every sequence (sequence stride 0):
    # valid strides, and every access would stay inside the buffer
    one = torch.zeros(lmax * hkv * d, dtype=torch.bfloat16, device="cuda")
    kv = one.as_strided((bsz, lmax, hkv, d), (0, hkv * d, d, 1))
    kv_len = torch.ones(bsz, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert _call_noalloc(kinv, q, kv, kv, kv_len, out) == kinv.ERR_WORKSPACE
    # argument errors come first, in kinv_attn_decode's order: a misaligned
    # output is reported as such even when the size is also too large
    bad_out = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + q.numel()].view(q.shape)
    assert _call_noalloc(kinv, q, kv, kv, kv_len, bad_out) == kinv.ERR_ALIGNMENT
