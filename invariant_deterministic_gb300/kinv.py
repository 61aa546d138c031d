"""Thin ctypes binding over libkinv.so (the C ABI in ``include/kinv.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors are PyTorch CUDA tensors (PyTorch supplies
device memory and the current stream); each wrapper checks dtypes and
contiguity, passes raw pointers, sizes and the current stream, and raises
``KinvError`` if the library returns a non-zero status.  There is no fallback:
if the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkinv.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = (
    0, -1, -2, -3, -4, -5, -6)
BF16, F32 = 0, 1
SPLIT_LEN = 256

_lib = None

_c_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/kinv.h
SIGNATURES = {
    "kinv_status_string": (ctypes.c_char_p, [_i32]),
    "kinv_device_class": (ctypes.c_char_p, []),
    "kinv_build_id": (ctypes.c_char_p, []),
    "kinv_last_device_status": (_i32, [_c_p]),
    "kinv_test_bounded_wait": (_i32, [_i64, _c_p]),
    "kinv_gemm": (_i32, [_c_p, _i64, _c_p, _i64, _c_p, _i64, _i32, _i32, _i32, _i32, _c_p]),
    "kinv_gemm_fused": (_i32, [_c_p, _i64, _c_p, _i64, _c_p, _i64, _i32, _i32, _i32, _i32, _c_p, _c_p]),
    "kinv_row_sumsq": (_i32, [_c_p, _i64, _i32, _i32, _c_p, _c_p]),
    "kinv_gemm_swiglu": (_i32, [_c_p, _i64, _c_p, _i64, _c_p, _i64, _i32, _i32, _i32, _c_p, _c_p]),
    "kinv_gemm_qkv_rope": (_i32, [_c_p, _i64, _c_p, _i64, _c_p, _c_p, _c_p, _i64, _i64, _c_p, _c_p,
                                  _c_p, _c_p, _f32, _i32, _i32, _i32, _i32, _i32, _f32, _c_p, _c_p]),
    "kinv_rmsnorm": (_i32, [_c_p, _i64, _c_p, _c_p, _c_p, _i64, _i32, _i32, _f32, _c_p]),
    "kinv_attn_decode_workspace": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "kinv_attn_decode": (_i32, [_c_p, _c_p, _c_p, _i64, _i64, _c_p, _c_p, _i32, _i32, _i32, _i32,
                                _i32, _i32, _f32, _c_p, _sz, _c_p]),
    "kinv_attn_decode_noalloc": (_i32, [_c_p, _c_p, _c_p, _i64, _i64, _c_p, _c_p, _i32, _i32, _i32,
                                        _i32, _i32, _i32, _f32, _c_p]),
    "kinv_attn_prefill_workspace": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "kinv_attn_prefill": (_i32, [_c_p, _c_p, _c_p, _i64, _i64, _c_p, _c_p, _c_p, _c_p, _i32, _i32,
                                 _i32, _i32, _i32, _i32, _i32, _i32, _f32, _c_p, _sz, _c_p]),
    "kinv_sample_workspace": (_sz, [_i32, _i32]),
    "kinv_sample": (_i32, [_c_p, _i64, _i32, _i32, _c_p, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _sz,
                           _c_p]),
    "kinv_embed": (_i32, [_c_p, _i32, _i32, _c_p, _c_p, _i32, _c_p]),
    "kinv_add": (_i32, [_c_p, _c_p, _c_p, _i64, _c_p]),
    "kinv_scale_columns": (_i32, [_c_p, _i64, _c_p, _c_p, _i64, _i32, _i32, _c_p]),
    "kinv_swiglu": (_i32, [_c_p, _i64, _c_p, _i64, _i32, _i32, _c_p]),
    "kinv_rope_append": (_i32, [_c_p, _i64, _c_p, _c_p, _c_p, _i64, _i64, _c_p, _c_p, _c_p, _c_p,
                                _f32, _i32, _i32, _i32, _i32, _f32, _c_p]),
    "kinv_decode_advance": (_i32, [_c_p, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _i32, _c_p]),
}


class KinvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libkinv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkinv.so is not built ({LIB_PATH}); run "
                               "invariant_deterministic_gb300.build.build() first")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().kinv_status_string(int(status)).decode()


def device_class() -> str:
    return lib().kinv_device_class().decode()


def build_id() -> str:
    return lib().kinv_build_id().decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise KinvError(status, where)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")


def last_device_status(stream=None) -> int:
    return lib().kinv_last_device_status(_stream(stream))


def test_bounded_wait(limit_ns: int, stream=None) -> None:
    """kinv_test_bounded_wait: one block waits on a barrier nothing
    completes, gives up after limit_ns and records KINV_ERR_TIMEOUT."""
    _check(lib().kinv_test_bounded_wait(int(limit_ns), _stream(stream)), "kinv_test_bounded_wait")


# --------------------------------------------------------------------- GEMM
def gemm(a: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
         out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """out[M][N] = a[M][K] . w[N][K]^T (bf16 in, fp32 accumulate)."""
    _need(a, torch.bfloat16, "a")
    _need(w, torch.bfloat16, "w")
    m, k = a.shape
    n = w.shape[0]
    if w.shape[1] != k or a.stride(1) != 1 or w.stride(1) != 1:
        raise ValueError("gemm: shapes or layouts do not match")
    if out is None:
        out = torch.empty(m, n, dtype=out_dtype, device=a.device)
    if out.stride(1) != 1 or tuple(out.shape) != (m, n):
        raise ValueError("gemm: bad output")
    dt = F32 if out.dtype == torch.float32 else BF16
    _check(lib().kinv_gemm(_ptr(a), a.stride(0), _ptr(w), w.stride(0), _ptr(out), out.stride(0),
                           dt, m, n, k, _stream(stream)), "kinv_gemm")
    return out


class GemmFusion(ctypes.Structure):
    """kinv_gemm_fusion: the RMSNorm folded into the projections around it."""
    _fields_ = [("row_ss", _c_p), ("row_ss_tiles", _i32), ("norm_dim", _i32), ("eps", _f32),
                ("resid", _c_p), ("ld_resid", _i64), ("ss_out", _c_p)]


def norm_in(row_ss: torch.Tensor, norm_dim: int, eps: float) -> GemmFusion:
    """Consuming side: scale output row m by 1/rms from row_ss [M][tiles]."""
    _need(row_ss, torch.float32, "row_ss")
    return GemmFusion(row_ss=_ptr(row_ss), row_ss_tiles=row_ss.shape[1], norm_dim=norm_dim, eps=float(eps))


def residual_out(resid: torch.Tensor, ss_out: torch.Tensor) -> GemmFusion:
    """Producing side: resid <- bf16(resid + out), out the fp32 product
    (rounded once); ss_out [M][N/128]."""
    _need(resid, torch.bfloat16, "resid")
    _need(ss_out, torch.float32, "ss_out")
    return GemmFusion(resid=_ptr(resid), ld_resid=resid.stride(0), ss_out=_ptr(ss_out))


def _fusion_ptr(f):
    return ctypes.byref(f) if f is not None else None


def gemm_fused(a, w, fusion: GemmFusion, out=None, n=None, stream=None):
    """kinv_gemm_fused.  With a residual fusion there is no other output
    (out may be None); otherwise out is written as by gemm()."""
    _need(a, torch.bfloat16, "a")
    _need(w, torch.bfloat16, "w")
    m, k = a.shape
    n = w.shape[0] if n is None else n
    dt = F32 if (out is not None and out.dtype == torch.float32) else BF16
    _check(lib().kinv_gemm_fused(_ptr(a), a.stride(0), _ptr(w), w.stride(0), _ptr(out),
                                 out.stride(0) if out is not None else n, dt, m, n, k,
                                 _fusion_ptr(fusion), _stream(stream)), "kinv_gemm_fused")
    return out


def row_sumsq(x, ss_out, stream=None):
    """ss_out[r][t] = sum of x[r][128t .. 128t+127]^2 (fp32)."""
    _need(x, torch.bfloat16, "x")
    _need(ss_out, torch.float32, "ss_out")
    rows, dim = x.shape
    _check(lib().kinv_row_sumsq(_ptr(x), x.stride(0), rows, dim, _ptr(ss_out), _stream(stream)),
           "kinv_row_sumsq")
    return ss_out


def interleave_gate_up(w_gu: torch.Tensor) -> torch.Tensor:
    """[gate rows; up rows] ([2F][K]) -> the block-of-64 interleaved layout
    kinv_gemm_swiglu reads (a one-time weight layout change, a copy)."""
    two_f, k = w_gu.shape
    f = two_f // 2
    return w_gu.view(2, f // 64, 64, k).permute(1, 0, 2, 3).reshape(two_f, k).contiguous()


def gemm_swiglu(a: torch.Tensor, w_gu_il: torch.Tensor, out: torch.Tensor | None = None,
                fusion: GemmFusion | None = None, stream=None) -> torch.Tensor:
    """act[M][F] = bf16(silu(a . Wgate^T) * (a . Wup^T)), W in the interleaved
    layout of ``interleave_gate_up``."""
    _need(a, torch.bfloat16, "a")
    _need(w_gu_il, torch.bfloat16, "w_gu")
    m, k = a.shape
    f = w_gu_il.shape[0] // 2
    if out is None:
        out = torch.empty(m, f, dtype=torch.bfloat16, device=a.device)
    _check(lib().kinv_gemm_swiglu(_ptr(a), a.stride(0), _ptr(w_gu_il), w_gu_il.stride(0), _ptr(out),
                                  out.stride(0), m, f, k, _fusion_ptr(fusion), _stream(stream)),
           "kinv_gemm_swiglu")
    return out


def gemm_qkv_rope(a, w_qkv, q_out, k_cache, v_cache, seq, pos, n_q, n_kv, head_dim, rope_base,
                  q_norm=None, k_norm=None, eps=1e-6, fusion=None, stream=None):
    """kinv_gemm followed by kinv_rope_append in one kernel: q heads of
    a . w_qkv^T -> q_out [M][Hq][D]; k and v heads into the caches
    [B][Lmax][Hkv][D] at [seq][pos]."""
    _need(a, torch.bfloat16, "a")
    _need(w_qkv, torch.bfloat16, "w_qkv")
    m, k = a.shape
    _check(lib().kinv_gemm_qkv_rope(_ptr(a), a.stride(0), _ptr(w_qkv), w_qkv.stride(0), _ptr(q_out),
                                    _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), k_cache.stride(1),
                                    _ptr(seq), _ptr(pos), _ptr(q_norm), _ptr(k_norm),
                                    float(eps), m, n_q, n_kv, head_dim, k, float(rope_base),
                                    _fusion_ptr(fusion), _stream(stream)),
           "kinv_gemm_qkv_rope")
    return q_out


# ------------------------------------------------------------------ RMSNorm
def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, residual=None, out=None,
            stream=None) -> torch.Tensor:
    """y = RMSNorm(x) * w; with ``residual``, x <- bf16(x + residual) first
    (in place) and y = RMSNorm(x)."""
    _need(x, torch.bfloat16, "x")
    rows, dim = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(lib().kinv_rmsnorm(_ptr(x), x.stride(0), _ptr(residual), _ptr(w), _ptr(out),
                              out.stride(0), rows, dim, float(eps), _stream(stream)),
           "kinv_rmsnorm")
    return out


# ---------------------------------------------------------------- attention
def attn_decode_workspace(batch: int, n_q: int, head_dim: int, max_len: int,
                          split_len: int = SPLIT_LEN) -> int:
    return int(lib().kinv_attn_decode_workspace(batch, n_q, head_dim, max_len, split_len))


def attn_decode(q, k_cache, v_cache, kv_len, out=None, workspace=None, split_len=SPLIT_LEN,
                scale: float = 0.0, stream=None):
    """q [B][Hq][D]; caches [B][Lmax][Hkv][D] (or any layout with the same
    last two dims and strides along B and L); kv_len int32 [B]."""
    _need(q, torch.bfloat16, "q")
    _need(kv_len, torch.int32, "kv_len")
    bsz, hq, d = q.shape
    lmax, hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    need = attn_decode_workspace(bsz, hq, d, lmax, split_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().kinv_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.stride(0),
                                  k_cache.stride(1), _ptr(kv_len), _ptr(out), bsz, hq, hkv, d, lmax,
                                  split_len, float(scale), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "kinv_attn_decode")
    return out


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def attn_decode_noalloc(q, k_cache, v_cache, kv_len, out, split_len=SPLIT_LEN, scale: float = 0.0,
                        stream=None):
    """Decode attention for callers that cannot allocate device memory: the
    library's own scratch array holds the partials (up to
    NOALLOC_SCRATCH_BYTES; calls sharing a device must not overlap on the GPU).
    ``out`` must be given, since this path allocates nothing."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(kv_len, torch.int32, "kv_len")
    _need(out, torch.bfloat16, "out")
    if tuple(out.shape) != tuple(q.shape) or not out.is_contiguous() or not q.is_contiguous():
        raise ValueError("attn_decode_noalloc: q and out must be contiguous [B][Hq][D] of one shape")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or v_cache.stride() != k_cache.stride():
        raise ValueError("attn_decode_noalloc: the caches must share shape and strides")
    bsz, hq, d = q.shape
    lmax, hkv = k_cache.shape[1], k_cache.shape[2]
    _check(lib().kinv_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.stride(0),
                                          k_cache.stride(1), _ptr(kv_len), _ptr(out), bsz, hq, hkv,
                                          d, lmax, split_len, float(scale), _stream(stream)),
           "kinv_attn_decode_noalloc")
    return out


def attn_prefill_workspace(total_rows: int, n_q: int, head_dim: int, max_kv: int,
                           split_len: int = SPLIT_LEN) -> int:
    return int(lib().kinv_attn_prefill_workspace(total_rows, n_q, head_dim, max_kv, split_len))


def attn_prefill(q, k_cache, v_cache, q_start, q_len, q_offset, max_q_len: int, max_kv: int,
                 out=None, workspace=None, split_len=SPLIT_LEN, scale: float = 0.0, stream=None):
    """q [rows][Hq][D]; per-sequence int32 q_start, q_len, q_offset [B]."""
    _need(q, torch.bfloat16, "q")
    rows, hq, d = q.shape
    hkv = k_cache.shape[2]
    bsz = q_start.shape[0]
    if out is None:
        out = torch.empty_like(q)
    need = attn_prefill_workspace(rows, hq, d, max_kv, split_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().kinv_attn_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.stride(0),
                                   k_cache.stride(1), _ptr(q_start), _ptr(q_len), _ptr(q_offset),
                                   _ptr(out), bsz, rows, max_q_len, max_kv, hq, hkv, d, split_len,
                                   float(scale), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "kinv_attn_prefill")
    return out


# ------------------------------------------------------------------ sampler
@dataclass
class SamplingParams:
    """Per-request sampler settings (the fields a Kinetic receipt records)."""
    temperature: float = 0.8
    top_k: int = 50
    top_p: float = 0.95
    min_p: float = 0.05
    repeat_penalty: float = 1.1
    repeat_last_n: int = 64
    seed: int = 42
    presence_penalty: float = 0.0
    frequency_penalty: float = 0.0
    logit_bias: dict = None   # {id: bias}, applied in insertion order
    typical_p: float = 1.0    # on when 0 < typical_p < 1


def sampling_params_device(params_list, device="cuda"):
    """kinv_sampling_params [B] packed on the device, and the device buffer
    of logit-bias entries they point to (None without any); keep both alive
    while sampling with them."""
    from . import synth
    entries, _ = synth.bias_entries(params_list)
    bias = torch.from_numpy(entries.view(np.uint8).copy()).to(device) if len(entries) else None
    packed = synth.sampling_struct(params_list, bias.data_ptr() if bias is not None else 0)
    return torch.from_numpy(packed.view(np.uint8).copy()).to(device), bias


def sample(logits, params_dev, history, hist_len, step, out=None, stream=None):
    """logits fp32 [B][V]; params_dev uint8 tensor holding B packed
    kinv_sampling_params; history int32 [B][H]; hist_len int32 [B];
    step int64 [B] -> int32 [B]."""
    _need(logits, torch.float32, "logits")
    bsz, v = logits.shape
    if out is None:
        out = torch.empty(bsz, dtype=torch.int32, device=logits.device)
    _check(lib().kinv_sample(_ptr(logits), logits.stride(0), bsz, v, _ptr(params_dev),
                             _ptr(history), history.shape[1] if history is not None else 0,
                             _ptr(hist_len), _ptr(step), _ptr(out), None, 0, _stream(stream)),
           "kinv_sample")
    return out


# --------------------------------------------------------------------- glue
def embed(table, ids, out=None, stream=None):
    vocab, dim = table.shape
    rows = ids.shape[0]
    if out is None:
        out = torch.empty(rows, dim, dtype=table.dtype, device=table.device)
    _check(lib().kinv_embed(_ptr(table), vocab, dim, _ptr(ids), _ptr(out), rows, _stream(stream)),
           "kinv_embed")
    return out


def add(x, y, out=None, stream=None):
    if out is None:
        out = torch.empty_like(x)
    _check(lib().kinv_add(_ptr(x), _ptr(y), _ptr(out), x.numel(), _stream(stream)), "kinv_add")
    return out


def scale_columns(w, g, out=None, stream=None):
    """out[n][k] = bf16(w[n][k] * g[k]): a norm gain folded into a weight."""
    _need(w, torch.bfloat16, "w")
    _need(g, torch.bfloat16, "g")
    n, k = w.shape
    if out is None:
        out = torch.empty_like(w)
    _check(lib().kinv_scale_columns(_ptr(w), w.stride(0), _ptr(g), _ptr(out), out.stride(0), n, k,
                                    _stream(stream)), "kinv_scale_columns")
    return out


def swiglu(gu, out=None, stream=None):
    rows, two_f = gu.shape
    f = two_f // 2
    if out is None:
        out = torch.empty(rows, f, dtype=gu.dtype, device=gu.device)
    _check(lib().kinv_swiglu(_ptr(gu), gu.stride(0), _ptr(out), out.stride(0), rows, f,
                             _stream(stream)), "kinv_swiglu")
    return out


def rope_append(qkv, q_out, k_cache, v_cache, seq, pos, n_q, n_kv, head_dim, rope_base,
                q_norm=None, k_norm=None, eps=1e-6, stream=None):
    rows = qkv.shape[0]
    _check(lib().kinv_rope_append(_ptr(qkv), qkv.stride(0), _ptr(q_out), _ptr(k_cache),
                                  _ptr(v_cache), k_cache.stride(0), k_cache.stride(1), _ptr(seq),
                                  _ptr(pos), _ptr(q_norm), _ptr(k_norm), float(eps), rows, n_q,
                                  n_kv, head_dim, float(rope_base), _stream(stream)),
           "kinv_rope_append")
    return q_out


def decode_advance(tokens, history, hist_len, step, pos=None, kv_len=None, stream=None):
    bsz = tokens.shape[0]
    _check(lib().kinv_decode_advance(_ptr(tokens), _ptr(history), history.shape[1],
                                     _ptr(hist_len), _ptr(step), _ptr(pos), _ptr(kv_len), bsz,
                                     _stream(stream)), "kinv_decode_advance")


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
