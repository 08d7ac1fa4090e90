"""fp64 CPU oracle for the attention forward and row-wise softmax / LSE.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` leg are the only callers.
The product package never imports this module and this module never imports
the product package; both sides meet only through the seeded input generators
(``online_softmax_10_gb300.inputs``), which hold none of the method's
arithmetic.

``oracle.c`` computes the plain three-pass definitions:
  * softmax and log-sum-exp -- "从原始Softmax到在线Softmax", section
    "softmax形式推导"; "什么是 online softmax and flash attention", section
    "Safe softmax", eq (2);
  * attention -- "什么是 online softmax and flash attention", section
    "Attention的数学表达", eq (8)-(9), with an explicit ``scale`` and an optional
    top-left causal mask (key j kept for query i iff j <= i).

``online.py`` restates the pages' online recurrences (sequential and
block-wise) for small inputs; it is pinned against the same worked examples.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain -O2, no fast-math,
    no FMA contraction, so the host arithmetic is the same on x86 and Arm)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            lib.oracle_softmax_rows.argtypes = [dp, ctypes.c_long, ctypes.c_long, dp, dp, ctypes.c_int]
            lib.oracle_softmax_rows.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, ctypes.c_long, ctypes.c_double, ctypes.c_int,
                                             lp, ctypes.c_long, dp, dp, ctypes.c_int]
            lib.oracle_attn_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def as_f64(a) -> np.ndarray:
    """Widen an array (numpy, or a CPU torch tensor of any float dtype) to a
    contiguous float64 numpy array.  bf16/fp32 -> fp64 is exact."""
    if hasattr(a, "detach") and hasattr(a, "double"):
        a = a.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softmax_rows(X, want_p: bool = True, nthreads: int | None = None):
    """Row-wise softmax of X[rows, cols] in fp64.  Returns (P or None, LSE)."""
    X = as_f64(X)
    if X.ndim != 2 or X.shape[1] == 0:
        raise ValueError("X must be [rows, cols] with cols > 0")
    rows, cols = X.shape
    P = np.empty_like(X) if want_p else None
    LSE = np.empty(rows, dtype=np.float64)
    lib = _load()
    rc = lib.oracle_softmax_rows(_dptr(X), rows, cols, _dptr(P) if P is not None else None,
                                 _dptr(LSE), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_softmax_rows failed ({rc})")
    return P, LSE


def logsumexp_rows(X, nthreads: int | None = None) -> np.ndarray:
    return softmax_rows(X, want_p=False, nthreads=nthreads)[1]


def log_softmax_rows(X, nthreads: int | None = None):
    """log p = z - LSE(z) per row ("从原始Softmax到在线Softmax", section
    "softmax形式推导", the log-softmax identity).  Returns (logP, LSE)."""
    X = as_f64(X)
    lse = logsumexp_rows(X, nthreads)
    return X - lse[:, None], lse


def cross_entropy_rows(X, labels, nthreads: int | None = None):
    """Per-row cross-entropy -log p_label = LSE(z) - z_label, the log-softmax
    followed by the label's negative log-probability of the page's
    cross_entropy_loss sketch ("从原始Softmax到在线Softmax", section
    "softmax实际代码实现"), without its batch mean.  Labels outside
    [0, cols) give 0 (an ignored row).  Returns (loss, LSE)."""
    X = as_f64(X)
    lab = np.asarray(labels.cpu() if hasattr(labels, "cpu") else labels, dtype=np.int64).reshape(-1)
    if lab.shape[0] != X.shape[0]:
        raise ValueError("one label per row")
    lse = logsumexp_rows(X, nthreads)
    loss = np.zeros(X.shape[0], dtype=np.float64)
    ok = (lab >= 0) & (lab < X.shape[1])
    rows = np.nonzero(ok)[0]
    loss[rows] = lse[rows] - X[rows, lab[rows]]
    return loss, lse


def attn_fwd(Q, K, V, scale: float, causal=False, rows=None, nthreads: int | None = None):
    """Attention forward in fp64.  causal: 0/False none, 1/True top-left
    (key j for query i iff j <= i), 2 bottom-right (iff j <= i + M - N); a
    query with no kept key gets O = 0, LSE = -inf.

    Q [B,H,N,d], K [B,H,M,d], V [B,H,M,d] (numpy or CPU torch; widened exactly).
    ``rows``: optional 1-D array of flat query indices (b*H + h)*N + i.
    Returns (O, LSE): O [B,H,N,d] and LSE [B,H,N] when rows is None, otherwise
    O [len(rows), d] and LSE [len(rows)].
    """
    Q, K, V = as_f64(Q), as_f64(K), as_f64(V)
    if Q.ndim != 4 or K.ndim != 4 or V.ndim != 4:
        raise ValueError("Q, K, V must be 4-D [B,H,*,d]")
    B, H, N, d = Q.shape
    M = K.shape[2]
    if K.shape != (B, H, M, d) or V.shape != (B, H, M, d):
        raise ValueError("shape mismatch")
    lib = _load()
    if rows is None:
        nsel = B * H * N
        sel_p = None
    else:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        nsel = sel.shape[0]
        sel_p = sel.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    O = np.empty((nsel, d), dtype=np.float64)
    LSE = np.empty(nsel, dtype=np.float64)
    rc = lib.oracle_attn_rows(_dptr(Q), _dptr(K), _dptr(V), B, H, N, M, d, float(scale), int(causal),
                              sel_p, nsel, _dptr(O), _dptr(LSE), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    if rows is None:
        return O.reshape(B, H, N, d), LSE.reshape(B, H, N)
    return O, LSE
