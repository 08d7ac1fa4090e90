"""fa_attn_fwd_splitkv_noalloc, the split-KV entry point for callers that
cannot allocate device memory (their memory belongs to another allocator, or
they must not call cudaMalloc/cudaFree): its partial results go to a scratch
array built into the library instead of a caller workspace.

It is called through the C ABI and checked on two calls in a row that solve
different problems (other inputs, other shapes), so partials left in the
shared scratch by the first call would corrupt the second if any were not
rewritten.  Each call is compared with the existing entry point
fa_attn_fwd_splitkv (a torch-allocated workspace) and with the fp64 oracle:
O as computed (fp32) within 1e-2 of the oracle and equal to the split entry
point's; bf16 O equal to RN of the fp32 O bit for bit; LSE relative 1e-3.
The file name sorts last so that a run that stops at the first failure has
already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_10_gb300 import fattn, inputs
from parity import O_TOL_BF16, bf16_bits_equal_rn, ensure_built, lse_ok, nan_full, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _noalloc_c_abi(q, k, v, o, lse, scale, causal, splits):
    B, H, N, d = q.shape
    M = k.shape[2]
    L = fattn.lib()
    out_code = fattn.FA_BF16 if o.dtype == torch.bfloat16 else fattn.FA_F32
    return L.fa_attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, N, M, d, ctypes.c_float(scale), int(causal), splits,
                                         fattn.FA_BF16, out_code,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc(q, k, v, scale, causal, splits, out_dtype):
    B, H, N, d = q.shape
    o = nan_full((B, H, N, d), out_dtype)
    lse = nan_full((B, H, N), torch.float32)
    rc = _noalloc_c_abi(q, k, v, o, lse, scale, causal, splits)
    assert rc == fattn.FA_OK, fattn.status_string(rc)
    assert fattn.device_status() == fattn.FA_OK
    return o, lse


# Pairs of problems run back to back: the second call's rows overlap the
# first call's partials in the scratch, with other values.
PAIRS = [
    ((1, 8, 256, 16384, 128, False, 0, 1), (1, 8, 256, 12000, 128, False, 0, 2)),
    ((1, 2, 300, 2100, 64, True, 7, 3), (2, 3, 129, 4000, 64, True, 5, 4)),
    ((2, 3, 129, 4000, 128, True, 5, 5), (1, 2, 300, 2100, 128, 2, 7, 6)),
]


@pytest.mark.parametrize("first,second", PAIRS)
def test_noalloc_two_calls_match_splitkv_and_oracle(first, second):
    for B, H, N, M, d, causal, splits, seed in (first, second):
        scale = 1.0 / math.sqrt(d)
        qc, kc, vc = inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=seed)
        q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
        o32, lse = _noalloc(q, k, v, scale, causal, splits, torch.float32)
        o16, lse16 = _noalloc(q, k, v, scale, causal, splits, torch.bfloat16)
        assert bf16_bits_equal_rn(o16, o32) and torch.equal(lse16, lse)
        # the existing entry point, with a caller workspace
        ref_o, ref_l = fattn.attn_fwd_splitkv(q, k, v, scale, causal, num_splits=splits, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(o32, ref_o) and torch.equal(lse, ref_l)
        # the oracle
        O_ref, L_ref = oracle.attn_fwd(qc, kc, vc, scale, causal)
        og = to_np(o32)
        assert not np.any(np.isnan(og))
        assert float(np.max(np.abs(og - O_ref))) <= O_TOL_BF16
        ok, rel = lse_ok(to_np(lse), L_ref)
        assert ok, rel


def test_noalloc_python_wrapper():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 4, 200, 3000, 128, torch.bfloat16, seed=9))
    o = nan_full(q.shape, torch.bfloat16)
    lse = nan_full(q.shape[:3], torch.float32)
    fattn.attn_fwd_splitkv_noalloc(q, k, v, causal=True, num_splits=6, out=o, lse=lse)
    assert fattn.device_status() == fattn.FA_OK
    ref_o, ref_l = fattn.attn_fwd_splitkv(q, k, v, causal=True, num_splits=6)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    with pytest.raises(ValueError):
        fattn.attn_fwd_splitkv_noalloc(q, k, v, out=o)


def test_noalloc_rejects_problems_beyond_the_scratch():
    # B*H*N*d*4*S far beyond 32 MiB: refused before anything is enqueued
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 16, 2048, 2048, 128, torch.bfloat16, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty((1, 16, 2048), dtype=torch.float32, device="cuda")
    need = fattn.splitkv_workspace_bytes(1, 16, 2048, 128, 8)
    assert need > fattn.NOALLOC_SCRATCH_BYTES
    assert _noalloc_c_abi(q, k, v, o, lse, 0.08, False, 8) == fattn.FA_ERR_INVALID_ARG
    assert _noalloc_c_abi(q, k, v, o, lse, 0.08, False, 65) == fattn.FA_ERR_INVALID_ARG  # above the split maximum
