"""Thin ctypes binding of libfattn (include/fattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfattn.so.  torch supplies device memory and the current stream.
There is no CPU path: if the library is missing or no GPU is present, calls
raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn.so")

FA_F32, FA_BF16 = 0, 1
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT = range(6)

# Every symbol include/fattn.h declares, with its ctypes signature.
_c_int, _c_long, _c_float, _vp = ctypes.c_int, ctypes.c_long, ctypes.c_float, ctypes.c_void_p
SIGNATURES = {
    "fa_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                             _c_int, _c_int, _vp]),
    "fa_attn_fwd_strided": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                     _vp, _c_float, _c_int, _c_int, _c_int, _vp]),
    "fa_attn_fwd_splitkv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                     _c_int, _c_int, _vp, _c_long, _c_int, _c_int, _vp]),
    "fa_attn_fwd_splitkv_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                             _c_float, _c_int, _c_int, _c_int, _c_int, _vp]),
    "fa_attn_splitkv_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "fa_attn_splitkv_workspace_bytes": (_c_long, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "fa_softmax_rows": (_c_int, [_vp, _vp, _vp, _c_long, _c_long, _c_int, _c_int, _vp]),
    "fa_logsumexp_rows": (_c_int, [_vp, _vp, _c_long, _c_long, _c_int, _vp]),
    "fa_log_softmax_rows": (_c_int, [_vp, _vp, _vp, _c_long, _c_long, _c_int, _c_int, _vp]),
    "fa_cross_entropy_rows": (_c_int, [_vp, _vp, _vp, _vp, _c_long, _c_long, _c_int, _vp]),
    "fa_device_status": (_c_int, [_vp, _c_int]),
    "fa_selftest_wait_timeout": (_c_int, [_c_int, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_c_int]),
    "fa_last_cuda_error": (ctypes.c_char_p, []),
    "fa_version": (_c_int, []),
}

_lock = threading.Lock()
_lib = None


class FattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = f": {lib().fa_last_cuda_error().decode()}" if status == FA_ERR_CUDA else ""
        super().__init__(f"{what} failed: {status_string(status)} ({status}){detail}")


def lib():
    """Load libfattn.so (built in-tree by online_softmax_10_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libfattn.so is not built ({LIB_PATH}); run online_softmax_10_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def version() -> int:
    return lib().fa_version()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return FA_F32
    if dt == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {dt}")


def _check_cuda(*ts):
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("libfattn works on CUDA tensors only (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def causal_code(causal) -> int:
    """False/0: no mask; True/1/'top_left': key j kept iff j <= i;
    2/'bottom_right': iff j <= i + (M - N)."""
    if causal in (2, "bottom_right"):
        return 2
    if causal in ("top_left",):
        return 1
    return int(bool(causal))


def attn_fwd(q, k, v, scale: float | None = None, causal: bool = False, out_dtype=None, out=None, lse=None,
             want_lse: bool = True, stream=None):
    """O = softmax(scale * q k^T [+ causal]) v and LSE, through fa_attn_fwd.

    q [B,H,N,d], k/v [B,H,M,d] contiguous CUDA tensors (bf16 or fp32).
    Returns (o, lse); lse is None when want_lse is False and lse is None.
    """
    _check_cuda(q, k, v)
    B, H, N, d = q.shape
    M = k.shape[2]
    if k.shape != (B, H, M, d) or v.shape != (B, H, M, d) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes/dtypes do not match")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_cuda(out, *([lse] if lse is not None else []))
    rc = lib().fa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, M, d, float(scale),
                           causal_code(causal), _dtype_code(q.dtype), _dtype_code(out.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_attn_fwd")
    return out, lse


def attn_fwd_strided(q, k, v, scale: float | None = None, causal=False, out=None, lse=None, want_lse: bool = True,
                     layout: str = "bshd", stream=None):
    """fa_attn_fwd_strided on views with any batch/head/row strides.

    With layout="bshd", q is [B, N, H, d], k/v [B, M, H, d] and ``out`` (made
    here if not given) is [B, N, H, d]; with layout="bhsd" the usual
    [B, H, N, d].  Strides are taken from the tensors themselves (d must be
    the contiguous dimension).  LSE is [B, H, N]."""
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.stride(-1) != 1:
            raise ValueError("CUDA tensors with a contiguous last dimension are required")
    if layout == "bshd":
        B, N, H, d = q.shape
        M = k.shape[1]
        pick = lambda t: (t.stride(0), t.stride(2), t.stride(1))  # (batch, head, row)
        oshape = (B, N, H, d)
    elif layout == "bhsd":
        B, H, N, d = q.shape
        M = k.shape[2]
        pick = lambda t: (t.stride(0), t.stride(1), t.stride(2))
        oshape = (B, H, N, d)
    else:
        raise ValueError(layout)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    arr = lambda t: (ctypes.c_longlong * 3)(*pick(t))
    qs, ks, vs, os_ = arr(q), arr(k), arr(v), arr(out)
    rc = lib().fa_attn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, M, d, qs, ks, vs, os_,
                                   float(scale), causal_code(causal), _dtype_code(q.dtype), _dtype_code(out.dtype),
                                   _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_attn_fwd_strided")
    return out, lse


def splitkv_num_splits(B: int, H: int, N: int, M: int, d: int, causal: bool) -> int:
    return lib().fa_attn_splitkv_num_splits(B, H, N, M, d, causal_code(causal))


def splitkv_workspace_bytes(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    return lib().fa_attn_splitkv_workspace_bytes(B, H, N, d, num_splits)


def attn_fwd_splitkv(q, k, v, scale: float | None = None, causal: bool = False, num_splits: int = 0,
                     workspace=None, out_dtype=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """fa_attn_fwd_splitkv: the key range of each query block split over
    ``num_splits`` CTAs (0 = automatic), partials merged by a second kernel.
    ``workspace`` is a caller-owned CUDA byte tensor; allocated here (by torch)
    when not given."""
    _check_cuda(q, k, v)
    B, H, N, d = q.shape
    M = k.shape[2]
    if k.shape != (B, H, M, d) or v.shape != (B, H, M, d) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes/dtypes do not match")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    S = num_splits if num_splits > 0 else splitkv_num_splits(B, H, N, M, d, causal_code(causal))
    need = splitkv_workspace_bytes(B, H, N, d, S)
    if need < 0:
        raise ValueError("invalid split count")
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().fa_attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, M, d, float(scale),
                                   causal_code(causal), S, _ptr(workspace), wbytes, _dtype_code(q.dtype),
                                   _dtype_code(out.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_attn_fwd_splitkv")
    return out, lse


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # FA_NOALLOC_SCRATCH_BYTES


def attn_fwd_splitkv_noalloc(q, k, v, scale: float | None = None, causal: bool = False, num_splits: int = 0,
                             out=None, lse=None, stream=None):
    """fa_attn_fwd_splitkv_noalloc: split-KV attention whose partials go to the
    library's fixed 32 MiB scratch instead of a caller workspace.  ``out`` and
    ``lse`` must be given (this call allocates nothing; torch is not asked
    for memory either)."""
    if out is None or lse is None:
        raise ValueError("attn_fwd_splitkv_noalloc allocates nothing: pass both out and lse")
    _check_cuda(q, k, v, out, lse)
    B, H, N, d = q.shape
    M = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = lib().fa_attn_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, M, d,
                                           float(scale), causal_code(causal), int(num_splits), _dtype_code(q.dtype),
                                           _dtype_code(out.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_attn_fwd_splitkv_noalloc")
    return out, lse


def softmax_rows(x, out_dtype=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Row-wise softmax of a 2-D CUDA tensor through fa_softmax_rows. Returns (p, lse)."""
    _check_cuda(x)
    rows, cols = x.shape
    out_dtype = out_dtype or x.dtype
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype, device=x.device)
    if lse is None and want_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = lib().fa_softmax_rows(_ptr(x), _ptr(out), _ptr(lse), rows, cols, _dtype_code(x.dtype),
                               _dtype_code(out.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_softmax_rows")
    return out, lse


def log_softmax_rows(x, out_dtype=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Row-wise log-softmax of a 2-D CUDA tensor through fa_log_softmax_rows. Returns (logp, lse)."""
    _check_cuda(x)
    rows, cols = x.shape
    out_dtype = out_dtype or x.dtype
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype, device=x.device)
    if lse is None and want_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = lib().fa_log_softmax_rows(_ptr(x), _ptr(out), _ptr(lse), rows, cols, _dtype_code(x.dtype),
                                   _dtype_code(out.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_log_softmax_rows")
    return out, lse


def cross_entropy_rows(x, labels, loss=None, lse=None, want_lse: bool = False, stream=None):
    """Per-row cross-entropy LSE(x_r) - x_r[label_r] through fa_cross_entropy_rows
    (int64 labels; labels outside [0, cols) give 0).  Returns (loss, lse)."""
    _check_cuda(x, labels)
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    rows, cols = x.shape
    if loss is None:
        loss = torch.empty((rows,), dtype=torch.float32, device=x.device)
    if lse is None and want_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = lib().fa_cross_entropy_rows(_ptr(x), _ptr(labels), _ptr(loss), _ptr(lse), rows, cols,
                                     _dtype_code(x.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_cross_entropy_rows")
    return loss, lse


def logsumexp_rows(x, out=None, stream=None):
    """Row-wise log-sum-exp of a 2-D CUDA tensor through fa_logsumexp_rows."""
    _check_cuda(x)
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = lib().fa_logsumexp_rows(_ptr(x), _ptr(out), rows, cols, _dtype_code(x.dtype), _stream(stream))
    if rc != FA_OK:
        raise FattnError(rc, "fa_logsumexp_rows")
    return out


def device_status(reset: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device status word (FA_OK or an error code)."""
    return lib().fa_device_status(_stream(stream), int(bool(reset)))


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> int:
    return lib().fa_selftest_wait_timeout(int(limit_us), _stream(stream))
