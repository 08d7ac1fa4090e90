"""Maximum sizes: tensors past 2^31 elements (the kernels' element offsets
must be 64-bit) and a million-key split-KV problem, each checked on sampled
rows against the fp64 oracle.  Tolerances as in the other parity tests.

Inputs are drawn on the device (seeded, inputs.device_normal); the sampled
rows and the heads they need are copied back and given to the oracle, so both
sides see the same bits.  Outputs start as NaN.  Attention O is checked as
computed (stored as fp32) at 1e-2, and the bf16-stored O of the same inputs
must be round-to-nearest-even of it, bit for bit, over the whole tensor.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_10_gb300 import fattn, inputs
from parity import (O_TOL_BF16, P_TOL_BF16, bf16_bits_equal_rn, default_entry, ensure_built, lse_ok, run_attn,
                    rows_logsumexp, rows_softmax, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _edge_and_sample(total, count, seed):
    rows = {0, total - 1}
    rows.update(int(r) for r in inputs.sample_rows(total, count, seed=seed))
    return np.array(sorted(rows))


# (rows, cols), each past 2^31 elements: the pipelined kernel (64 KB rows; 8 KB
# rows with four consumer groups, whose LSE alone takes the warp-per-row
# kernel) and the streaming kernels (> 64K columns)
ROW_SHAPES = [(65600, 32768), (525000, 4096), (21500, 100000)]


@pytest.mark.parametrize("rows,cols", ROW_SHAPES)
def test_softmax_rows_past_2p31_elements(rows, cols):
    assert rows * cols > 2 ** 31
    x = inputs.device_normal((rows, cols), seed=rows + cols, sigma=3.0)
    p, lse = rows_softmax(x)
    lse2 = rows_logsumexp(x)
    assert fattn.device_status() == fattn.FA_OK
    sel = _edge_and_sample(rows, 30, seed=cols)
    idx = torch.as_tensor(sel, device=x.device)
    P_ref, L_ref = oracle.softmax_rows(x[idx].cpu())
    assert not torch.isnan(p).any().item() and not torch.isnan(lse).any().item()
    err = float(np.max(np.abs(to_np(p[idx]) - P_ref)))
    assert err <= P_TOL_BF16, err
    for got in (lse, lse2):
        ok, rel = lse_ok(to_np(got[idx]), L_ref)
        assert ok, rel
    sums = p.sum(dim=1, dtype=torch.float32)
    assert torch.all((sums - 1).abs() <= 1e-2).item()


def test_attention_past_2p31_elements():
    # B=17 H=64 N=M=16384 d=128: 2.28e9 elements per tensor, causal
    B, H, N, d = 17, 64, 16384, 128
    q = inputs.device_normal((B, H, N, d), seed=71)
    k = inputs.device_normal((B, H, N, d), seed=72)
    v = inputs.device_normal((B, H, N, d), seed=73)
    assert q.numel() > 2 ** 31
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attn(default_entry, q, k, v, scale, True, torch.float32)
    o16, lse16 = run_attn(default_entry, q, k, v, scale, True, torch.bfloat16)
    assert bf16_bits_equal_rn(o16, o) and torch.equal(lse16, lse)
    del o16, lse16
    assert not torch.isnan(o).any().item() and not torch.isnan(lse).any().item()
    for (b, h) in [(0, 0), (8, 31), (B - 1, H - 1)]:
        sel = _edge_and_sample(N, 14, seed=b * H + h)
        qh, kh, vh = (t[b:b + 1, h:h + 1].cpu() for t in (q, k, v))
        O_ref, L_ref = oracle.attn_fwd(qh, kh, vh, scale, True, rows=sel)
        O_g = to_np(o[b, h])[sel]
        assert float(np.max(np.abs(O_g - O_ref))) <= O_TOL_BF16, float(np.max(np.abs(O_g - O_ref)))
        ok, rel = lse_ok(to_np(lse[b, h])[sel], L_ref)
        assert ok, rel
    del q, k, v, o, lse


def test_splitkv_million_keys():
    # decode-like: 64 queries per head against 2^20 keys, split over CTAs
    B, H, N, M, d = 1, 2, 64, 1 << 20, 128
    q = inputs.device_normal((B, H, N, d), seed=81)
    k = inputs.device_normal((B, H, M, d), seed=82)
    v = inputs.device_normal((B, H, M, d), seed=83)
    scale = 1.0 / math.sqrt(d)
    assert fattn.splitkv_num_splits(B, H, N, M, d, False) > 1
    S = fattn.splitkv_num_splits(B, H, N, M, d, False)
    ws = torch.full((fattn.splitkv_workspace_bytes(B, H, N, d, S),), 255, dtype=torch.uint8, device="cuda")
    o, lse = run_attn(lambda *a: fattn.attn_fwd_splitkv(*a[:5], num_splits=S, workspace=ws, out=a[5], lse=a[6],
                                                        stream=a[7]), q, k, v, scale, False, torch.float32)
    sel = _edge_and_sample(B * H * N, 14, seed=5)
    O_ref, L_ref = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(), scale, False, rows=sel)
    O_g = to_np(o).reshape(-1, d)[sel]
    assert float(np.max(np.abs(O_g - O_ref))) <= O_TOL_BF16
    ok, rel = lse_ok(to_np(lse).reshape(-1)[sel], L_ref)
    assert ok, rel
