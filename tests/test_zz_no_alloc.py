"""fa_attn_fwd_splitkv_noalloc, the split-KV entry point for callers that
cannot allocate device memory (their memory belongs to another allocator, or
they must not call cudaMalloc/cudaFree): its partial results go to a scratch
array built into the library instead of a caller workspace.

It is checked through the C ABI against the existing entry point
fa_attn_fwd_splitkv (given a torch-allocated workspace) on two calls in a row,
at the attention tests' tolerance (bf16 O: 1e-2 plus the bf16 store's half ulp
of |O|; LSE 1e-3 * max(1, |LSE|)).  The file name sorts last so that a run
that stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import BF16_HALF_ULP_REL, LSE_REL, O_TOL_BF16, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _noalloc_c_abi(q, k, v, o, lse, scale, causal, splits):
    B, H, N, d = q.shape
    M = k.shape[2]
    L = fattn.lib()
    return L.fa_attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, N, M, d, ctypes.c_float(scale), int(causal), splits,
                                         fattn.FA_BF16, fattn.FA_BF16,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,H,N,M,d,causal,splits", [
    (1, 8, 256, 16384, 128, False, 0), (1, 2, 300, 2100, 64, True, 7), (2, 3, 129, 4000, 128, True, 5)])
def test_noalloc_matches_splitkv_twice(B, H, N, M, d, causal, splits):
    scale = d ** -0.5
    q, k, v = (t.cuda() for t in inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=B + N + M))
    ref_o, ref_l = fattn.attn_fwd_splitkv(q, k, v, scale, causal, num_splits=splits)
    torch.cuda.synchronize()
    tol = O_TOL_BF16 + BF16_HALF_ULP_REL * ref_o.float().abs()
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc_c_abi(q, k, v, o, lse, scale, causal, splits)
        assert rc == fattn.FA_OK, fattn.status_string(rc)
        assert fattn.device_status() == fattn.FA_OK
        assert torch.all((o.float() - ref_o.float()).abs() <= tol).item()
        assert torch.all((lse - ref_l).abs() <= LSE_REL * ref_l.abs().clamp(min=1.0)).item()


def test_noalloc_rejects_problems_beyond_the_scratch():
    # B*H*N*d*4*S far beyond 32 MiB: refused before anything is enqueued
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 16, 2048, 2048, 128, torch.bfloat16, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty((1, 16, 2048), dtype=torch.float32, device="cuda")
    need = fattn.splitkv_workspace_bytes(1, 16, 2048, 128, 8)
    assert need > fattn.NOALLOC_SCRATCH_BYTES
    assert _noalloc_c_abi(q, k, v, o, lse, 0.08, False, 8) == fattn.FA_ERR_INVALID_ARG
