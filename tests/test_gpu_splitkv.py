"""Split-KV attention (fa_attn_fwd_splitkv) against the fp64 oracle: the key
range of each query block is split over several CTAs and the normalised
partials are merged by their log-sum-exp.  Same tolerances as fa_attn_fwd
(bf16 inputs: |dO| <= 1e-2 for fp32 O, plus the bf16 store's half ulp for
bf16 O; LSE relative 1e-3)."""
import math

import numpy as np
import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import attn_case, ensure_built, lse_ok, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _split_case(q, k, v, causal, splits, out_dtype=None, rows=None):
    """attn_case, but through the split entry point (patched in for the call)."""
    orig = fattn.attn_fwd

    def split_fwd(q_, k_, v_, scale, causal_, out_dtype=None, stream=None):
        return fattn.attn_fwd_splitkv(q_, k_, v_, scale, causal_, num_splits=splits, out_dtype=out_dtype,
                                      stream=stream)
    fattn.attn_fwd = split_fwd
    try:
        return attn_case(q, k, v, causal, out_dtype=out_dtype, rows=rows)
    finally:
        fattn.attn_fwd = orig


@pytest.mark.parametrize("splits", [2, 3, 7, 16, 0])
@pytest.mark.parametrize("B,H,N,M,d,causal", [
    (1, 2, 300, 2100, 128, False), (1, 2, 300, 2100, 64, True), (2, 1, 129, 1000, 128, True),
    (1, 3, 64, 8192, 128, False), (1, 2, 1000, 1000, 64, True), (1, 2, 300, 2100, 128, 2), (1, 2, 2100, 300, 64, 2)])
def test_splitkv_matches_oracle(splits, B, H, N, M, d, causal):
    q, k, v = inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=N + M + splits)
    for out in (None, torch.float32):
        err, ratio, ok, rel = _split_case(q, k, v, causal, splits, out_dtype=out)
        assert ratio <= 1.0, (out, err)
        assert ok, rel


def test_splitkv_close_to_unsplit():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 4, 256, 16384, 128, torch.bfloat16, seed=1))
    o1, l1 = fattn.attn_fwd(q, k, v, 0.09, False, out_dtype=torch.float32)
    o2, l2 = fattn.attn_fwd_splitkv(q, k, v, 0.09, False, num_splits=12, out_dtype=torch.float32)
    assert (o1 - o2).abs().max().item() < 2e-3
    assert (l1 - l2).abs().max().item() < 1e-4


def test_splitkv_auto_choice_and_workspace():
    n = fattn.splitkv_num_splits(1, 8, 256, 65536, 128, False)
    assert 2 <= n <= 64
    assert fattn.splitkv_num_splits(2, 32, 8192, 8192, 128, True) == 1  # already fills the GPU
    need = fattn.splitkv_workspace_bytes(1, 8, 256, 128, n)
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 8, 256, 4096, 128, torch.bfloat16, seed=2))
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.attn_fwd_splitkv(q, k, v, 0.1, False, num_splits=n, workspace=small)
    assert e.value.status == fattn.FA_ERR_INVALID_ARG
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.attn_fwd_splitkv(q, k, v, 0.1, False, num_splits=n, workspace=big[16:])
    assert e.value.status == fattn.FA_ERR_MISALIGNED
    o, lse = fattn.attn_fwd_splitkv(q, k, v, 0.1, False, num_splits=n, workspace=big[:need])
    assert fattn.device_status() == fattn.FA_OK
    ref, lref = fattn.attn_fwd(q, k, v, 0.1, False)
    assert (o.float() - ref.float()).abs().max().item() < 2e-2


def test_splitkv_decode_like_long_keys_sampled():
    # few query rows, long key range: the shape split-KV is for
    q, k, v = inputs.attn_inputs(1, 8, 256, 65536, 128, torch.bfloat16, seed=6)
    rows = inputs.sample_rows(8 * 256, 128, seed=6).numpy()
    err, ratio, ok, rel = _split_case(q, k, v, False, 0, out_dtype=torch.float32, rows=rows)
    assert ratio <= 1.0, err
    assert ok, rel
