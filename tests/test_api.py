"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/fattn.h declares, and rejects bad arguments before any
CUDA call (so these calls are safe on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

from online_softmax_10_gb300 import build as fbuild
from online_softmax_10_gb300 import fattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")

INVALID, UNSUPPORTED, MISALIGNED = fattn.FA_ERR_INVALID_ARG, fattn.FA_ERR_UNSUPPORTED, fattn.FA_ERR_MISALIGNED


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fattn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_attn_fwd", "fa_softmax_rows", "fa_logsumexp_rows", "fa_status_string", "fa_version",
              "fa_device_status", "fa_selftest_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    for n in names:
        assert hasattr(L, n), n
    # the binding's signature table covers the header exactly
    assert sorted(fattn.SIGNATURES) == names


def test_version_and_status_strings(L):
    assert fattn.version() == 100
    assert fattn.status_string(0) == "FA_OK"
    assert fattn.status_string(5) == "FA_ERR_DEVICE_TIMEOUT"
    assert fattn.status_string(12345) == "FA_ERR_UNKNOWN"


P = 1 << 20  # a 16-byte-aligned fake address: never dereferenced, every call below fails validation first


def attn(L, Q=P, K=P, V=P, O=P, LSE=P, B=1, H=1, N=8, M=8, d=64, scale=0.125, causal=0, i=1, o=1):
    return L.fa_attn_fwd(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, i, o, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(Q=None), INVALID), (dict(K=None), INVALID), (dict(V=None), INVALID), (dict(O=None), INVALID),
    (dict(B=0), INVALID), (dict(H=-1), INVALID), (dict(N=0), INVALID), (dict(M=0), INVALID), (dict(d=0), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(causal=3), INVALID), (dict(causal=-1), INVALID),
    (dict(i=7), UNSUPPORTED), (dict(o=9), UNSUPPORTED), (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED),
    (dict(i=0, o=1), UNSUPPORTED), (dict(i=0, d=48), UNSUPPORTED), (dict(B=300, H=300), UNSUPPORTED),
    (dict(Q=P + 8), MISALIGNED), (dict(O=P + 2), MISALIGNED), (dict(LSE=P + 4), MISALIGNED),
    (dict(B=1 << 30, H=1, N=1 << 30, M=1 << 30), INVALID),
])
def test_attn_argument_errors(L, kw, expect):
    assert attn(L, **kw) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, P, P, 4, 8, 1, 1), INVALID), ((P, None, P, 4, 8, 1, 1), INVALID), ((P, P, P, 0, 8, 1, 1), INVALID),
    ((P, P, P, 4, 0, 1, 1), INVALID), ((P, P, P, 4, -3, 1, 1), INVALID), ((P, P, P, 4, 8, 3, 1), UNSUPPORTED),
    ((P, P, P, 4, 8, 1, 5), UNSUPPORTED), ((P + 1, P, P, 4, 8, 1, 1), MISALIGNED),
    ((P, P + 4, P, 4, 8, 1, 1), MISALIGNED), ((P, P, P + 8, 4, 8, 1, 1), MISALIGNED),
    ((P, P, P, 1 << 40, 1 << 40, 1, 1), INVALID),
])
def test_softmax_rows_argument_errors(L, args, expect):
    assert L.fa_softmax_rows(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, P, 4, 8, 1), INVALID), ((P, None, 4, 8, 1), INVALID), ((P, P, 0, 8, 1), INVALID),
    ((P, P, 4, 0, 1), INVALID), ((P, P, 4, 8, 2), UNSUPPORTED), ((P + 2, P, 4, 8, 1), MISALIGNED),
])
def test_logsumexp_rows_argument_errors(L, args, expect):
    assert L.fa_logsumexp_rows(*args, None) == expect


def test_selftest_rejects_bad_limit(L):
    assert L.fa_selftest_wait_timeout(0, None) == INVALID
    assert L.fa_selftest_wait_timeout(2000000, None) == INVALID


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        fattn.softmax_rows(x)
    with pytest.raises(ValueError):
        fattn.attn_fwd(torch.zeros(1, 1, 2, 64), torch.zeros(1, 1, 2, 64), torch.zeros(1, 1, 2, 64))


def test_splitkv_workspace_bytes_host_arithmetic(L):
    # partial O fp32 [S][BH][N][d], 256-byte aligned, then partial LSE fp32 [S][BH][N]
    S, B, H, N, d = 5, 2, 3, 77, 128
    o = S * B * H * N * d * 4
    assert L.fa_attn_splitkv_workspace_bytes(B, H, N, d, S) == (o + 255) // 256 * 256 + S * B * H * N * 4
    assert L.fa_attn_splitkv_workspace_bytes(B, H, N, d, 1) == 0
    assert L.fa_attn_splitkv_workspace_bytes(B, H, N, d, 0) == -1
    assert L.fa_attn_splitkv_workspace_bytes(B, H, N, d, 65) == -1
    assert L.fa_attn_splitkv_workspace_bytes(0, H, N, d, 2) == -1


def test_splitkv_argument_errors(L):
    f = L.fa_attn_fwd_splitkv
    base = [P, P, P, P, P, 1, 2, 64, 4096, 128, 0.1, 0]
    assert f(*base, 65, P, 1 << 30, 1, 1, None) == INVALID          # too many splits
    assert f(*base, -1, P, 1 << 30, 1, 1, None) == INVALID
    assert f(*base, 4, None, 1 << 30, 1, 1, None) == INVALID        # no workspace
    assert f(*base, 4, P, 16, 1, 1, None) == INVALID                # workspace too small
    assert f(*base, 4, P + 16, 1 << 30, 1, 1, None) == MISALIGNED   # not 256-byte aligned
    assert f(*[P, P, P, P, P, 1, 2, 64, 4096, 64, 0.1, 0], 4, P, 1 << 30, 0, 0, None) == UNSUPPORTED  # fp32 split
    assert f(None, P, P, P, P, 1, 2, 64, 4096, 128, 0.1, 0, 4, P, 1 << 30, 1, 1, None) == INVALID


def test_row_extras_argument_errors(L):
    assert L.fa_log_softmax_rows(None, P, P, 4, 8, 1, 1, None) == INVALID
    assert L.fa_log_softmax_rows(P, None, P, 4, 8, 1, 1, None) == INVALID
    assert L.fa_log_softmax_rows(P, P + 8, P, 4, 8, 1, 1, None) == MISALIGNED
    assert L.fa_log_softmax_rows(P, P, P, 4, 8, 1, 7, None) == UNSUPPORTED
    assert L.fa_cross_entropy_rows(P, None, P, P, 4, 8, 1, None) == INVALID   # no labels
    assert L.fa_cross_entropy_rows(P, P, None, P, 4, 8, 1, None) == INVALID   # no loss
    assert L.fa_cross_entropy_rows(P, P, P, P, 0, 8, 1, None) == INVALID
    assert L.fa_cross_entropy_rows(P, P + 8, P, None, 4, 8, 1, None) == MISALIGNED
    assert L.fa_cross_entropy_rows(P, P, P, None, 4, 8, 3, None) == UNSUPPORTED


def test_strided_argument_errors(L):
    import ctypes
    arr = lambda *v: (ctypes.c_longlong * 3)(*v)
    good = arr(1 << 20, 64 * 8, 64 * 4)                   # bf16: multiples of 8 elements
    f = L.fa_attn_fwd_strided
    base = [P, P, P, P, P, 1, 4, 8, 8, 64]
    assert f(*base, None, good, good, good, 0.1, 0, 1, 1, None) == INVALID
    assert f(*base, good, good, good, None, 0.1, 0, 1, 1, None) == INVALID
    assert f(*base, arr(1 << 20, 64 * 8, 60), good, good, good, 0.1, 0, 1, 1, None) == MISALIGNED  # 120 B rows
    assert f(*base, good, arr(0, 64, 64), good, good, 0.1, 0, 1, 1, None) == MISALIGNED              # zero stride
    assert f(*base, good, good, good, arr(1 << 20, 64 * 8, 66), 0.1, 0, 1, 1, None) == MISALIGNED
    assert f(*base, good, good, good, good, 0.1, 3, 1, 1, None) == INVALID                           # causal mode
    # fp32 needs 16-byte strides too: 4 elements
    assert f(*[P, P, P, P, P, 1, 4, 8, 8, 64], arr(4096, 512, 66), good, good, good, 0.1, 0, 0, 0, None) == MISALIGNED
