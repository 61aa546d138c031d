"""The C-ABI library builds, loads without a GPU and exports every entry
point the public header declares; host-side validation rejects bad arguments
before any CUDA call (these calls never reach the device)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kinv.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from invariant_deterministic_gb300 import build, kinv
    build.build()
    return kinv


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kinv_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "kinv_gemm" in names and "kinv_sample" in names and len(names) >= 17
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) <= set(lib.SIGNATURES), set(names) - set(lib.SIGNATURES)


def test_identity_strings(lib):
    assert lib.device_class() == "cuda-sm103a"
    bid = lib.build_id()
    assert re.fullmatch(r"[0-9a-f]{16}", bid)
    from invariant_deterministic_gb300 import build
    assert bid == build.build_id()
    assert lib.status_string(0) == "KINV_OK"
    assert lib.status_string(-6) == "KINV_ERR_TIMEOUT"
    assert lib.status_string(123) == "KINV_ERR_UNKNOWN"


def test_host_validation_without_gpu(lib):
    L = lib.lib()
    fake = 0x10000  # never dereferenced: every call below fails validation first
    # GEMM: K not a multiple of 64, N not a multiple of 16, bad dtype, misaligned
    assert L.kinv_gemm(fake, 100, fake, 100, fake, 64, 0, 4, 64, 100, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_gemm(fake, 64, fake, 64, fake, 24, 0, 4, 24, 64, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_gemm(fake, 64, fake, 64, fake, 64, 7, 4, 64, 64, None) == lib.ERR_INVALID_ARG
    assert L.kinv_gemm(fake + 2, 64, fake, 64, fake, 64, 0, 4, 64, 64, None) == lib.ERR_ALIGNMENT
    assert L.kinv_gemm(None, 64, fake, 64, fake, 64, 0, 4, 64, 64, None) == lib.ERR_INVALID_ARG
    assert L.kinv_gemm(fake, 64, fake, 64, fake, 64, 0, 0, 64, 64, None) == lib.OK  # M = 0
    # folded RMSNorm options: residual output needs N % 128 and sums; row scale needs its shape
    import ctypes
    resid = lib.GemmFusion(resid=fake, ld_resid=192, ss_out=fake)
    assert L.kinv_gemm_fused(fake, 64, fake, 64, None, 0, 0, 4, 192, 64, ctypes.byref(resid),
                             None) == lib.ERR_UNSUPPORTED
    no_ss = lib.GemmFusion(resid=fake, ld_resid=256, ss_out=None)
    assert L.kinv_gemm_fused(fake, 64, fake, 64, None, 0, 0, 4, 256, 64, ctypes.byref(no_ss),
                             None) == lib.ERR_INVALID_ARG
    bad_norm = lib.GemmFusion(row_ss=fake, row_ss_tiles=0, norm_dim=256, eps=1e-6)
    assert L.kinv_gemm_fused(fake, 64, fake, 64, fake, 256, 0, 4, 256, 64, ctypes.byref(bad_norm),
                             None) == lib.ERR_INVALID_ARG
    assert L.kinv_gemm_swiglu(fake, 64, fake, 64, fake, 64, 4, 96, 64, None, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_gemm_swiglu(fake, 64, fake, 64, fake, 64, 4, 128, 64, ctypes.byref(resid),
                              None) == lib.ERR_INVALID_ARG
    assert L.kinv_gemm_qkv_rope(fake, 64, fake, 64, fake, fake, fake, 0, 96, fake, fake, None, None,
                                1e-6, 4, 2, 1, 96, 64, 1e4, None, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_row_sumsq(fake, 100, 4, 100, fake, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_row_sumsq(fake, 64, 4, 128, fake, None) == lib.ERR_INVALID_ARG  # ldx < dim
    # RMSNorm
    assert L.kinv_rmsnorm(fake, 100, None, fake, fake, 100, 2, 100, 1e-6, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_rmsnorm(fake, 64, None, fake, fake, 64, 2, 64, -1.0, None) == lib.ERR_INVALID_ARG
    # attention: head dim, GQA ratio, split length, workspace
    args = lambda D=128, hq=32, hkv=8, split=256, ws=fake, wsb=1 << 30: (
        fake, fake, fake, 8 * 128 * 64, 8 * 128, fake, fake, 2, hq, hkv, D, 64, split, 0.0, ws, wsb, None)
    assert L.kinv_attn_decode(*args(D=96)) == lib.ERR_UNSUPPORTED
    assert L.kinv_attn_decode(*args(hq=30)) == lib.ERR_INVALID_ARG
    assert L.kinv_attn_decode(*args(hq=48, hkv=3)) == lib.ERR_UNSUPPORTED
    assert L.kinv_attn_decode(*args(split=128)) == lib.ERR_UNSUPPORTED
    assert L.kinv_attn_decode(*args(wsb=16)) == lib.ERR_WORKSPACE
    assert L.kinv_attn_decode(*args(ws=None)) == lib.ERR_INVALID_ARG
    need = L.kinv_attn_decode_workspace(2, 32, 128, 64, 256)
    assert need >= 2 * 32 * 128 * 4
    # sampler / glue
    assert L.kinv_sample(fake, 10, 2, 20, fake, None, 0, None, fake, fake, None, 0, None) == lib.ERR_INVALID_ARG
    # history rows longer than 1024 ids (the penalty window) are not supported
    assert L.kinv_sample(fake, 20, 2, 20, fake, fake, 2000, fake, fake, fake, None, 0, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_swiglu(fake, 20, fake, 10, 2, 10, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_rope_append(fake, 512, fake, fake, fake, 0, 128, fake, fake, None, None, 1e-6,
                              1, 2, 1, 96, 1e4, None) == lib.ERR_UNSUPPORTED
    assert L.kinv_add(fake, fake, fake, 12, None) == lib.ERR_UNSUPPORTED
    # the bounded-wait self-test checks its limit before any CUDA call
    assert L.kinv_test_bounded_wait(10, None) == lib.ERR_INVALID_ARG
    assert L.kinv_test_bounded_wait(10**9, None) == lib.ERR_INVALID_ARG
