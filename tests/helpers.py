"""Shared test helpers: device checks, tolerance, bitwise comparison."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from invariant_deterministic_gb300 import synth  # noqa: E402

# Tolerance on bf16 outputs (allclose form): |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL = 2e-2
RTOL = 1e-2


def ensure_lib():
    from invariant_deterministic_gb300 import build
    build.build()
    from invariant_deterministic_gb300 import kinv
    return kinv


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp32 tensor -> fp64 numpy (exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu_vals, ref_vals, what="", atol=ATOL, rtol=RTOL):
    g = np.asarray(gpu_vals, dtype=np.float64)
    r = np.asarray(ref_vals, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = np.abs(g - r)
    bad = err > atol + rtol * np.abs(r)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(r))), g.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {g.size} outside tolerance; worst at {i}: "
                             f"gpu {g[i]!r} oracle {r[i]!r}")
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= 1e-2, f"{what}: norm-relative error {rel}"


def assert_same_bits(a: torch.Tensor, b: torch.Tensor, what=""):
    """Byte equality (NaN-safe); reports the first differing element."""
    ab = a.detach().contiguous().view(torch.uint8).cpu().numpy()
    bb = b.detach().contiguous().view(torch.uint8).cpu().numpy()
    assert ab.shape == bb.shape, (ab.shape, bb.shape)
    if not np.array_equal(ab, bb):
        diff = np.nonzero(ab.reshape(-1) != bb.reshape(-1))[0]
        esz = a.element_size()
        raise AssertionError(f"{what}: {len(diff)} differing bytes; first element index "
                             f"{diff[0] // esz} of {a.numel()}")


gpu = pytest.mark.gpu
