"""The seeded input generators: deterministic, the stated shapes, the stated
distributions (loosely), and the structure (the +20 spike, K row scaling)."""
import torch

from online_softmax_10_gb300 import inputs


def test_attn_inputs_deterministic_and_shaped():
    a = inputs.attn_inputs(2, 3, 17, 19, 64, torch.bfloat16, seed=5)
    b = inputs.attn_inputs(2, 3, 17, 19, 64, torch.bfloat16, seed=5)
    c = inputs.attn_inputs(2, 3, 17, 19, 64, torch.bfloat16, seed=6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    assert a[0].shape == (2, 3, 17, 64) and a[1].shape == (2, 3, 19, 64) and a[2].shape == (2, 3, 19, 64)
    assert all(t.dtype == torch.bfloat16 for t in a)


def test_attn_inputs_distributions():
    q, k, v = inputs.attn_inputs(1, 4, 512, 512, 64, torch.float32, seed=1)
    assert abs(q.mean().item()) < 0.02 and abs(q.std().item() - 1) < 0.02
    u = inputs.attn_inputs(1, 1, 64, 64, 64, torch.float32, seed=0, dist="uniform")[0]
    assert u.min() >= 0 and u.max() < 1
    q2, k2, v2 = inputs.attn_inputs(1, 4, 512, 512, 64, torch.float32, seed=1, k_row_scale=(0.5, 2.0))
    assert torch.equal(q, q2) and torch.equal(v, v2)
    ratio = (k2 / k).reshape(-1, 64)
    # one factor per key row, in [0.5, 2)
    assert torch.allclose(ratio, ratio[:, :1].expand_as(ratio), rtol=1e-5)
    assert ratio.min() >= 0.5 and ratio.max() < 2.0


def test_rows_inputs_spike_and_distribution():
    x = inputs.rows_inputs(64, 4096, torch.float32, seed=1)
    assert torch.all((x == 20.0).sum(1) == 1)
    body = x[x != 20.0]
    assert abs(body.std().item() - 3.0) < 0.05
    y = inputs.rows_inputs(64, 4096, torch.bfloat16, seed=1)
    assert y.dtype == torch.bfloat16 and torch.equal(y, x.to(torch.bfloat16))
    z = inputs.rows_inputs(4, 100, torch.float32, seed=1, spike=None)
    assert not torch.any(z == 20.0)


def test_workloads_match_their_specification():
    w = inputs.WORKLOADS
    assert len(w) == 5
    c4 = inputs.ATTN_B2H32_8192_D128_CAUSAL
    assert (c4.B, c4.H, c4.N, c4.M, c4.d, c4.causal, c4.seed) == (2, 32, 8192, 8192, 128, True, 3)
    assert abs(c4.flops() - 4 * 2 * 32 * 8192 * 8192 * 128 / 2) < 1
    assert inputs.ATTN_F32_64.dist == "uniform" and inputs.ATTN_F32_64.dtype == torch.float32
    assert inputs.ROWS_4096x32768.rows == 4096 and inputs.ROWS_4096x32768.cols == 32768


def test_sample_rows_includes_edges():
    s = inputs.sample_rows(1000, 20)
    assert s[0] == 0 and s[-1] == 999 and len(torch.unique(s)) == len(s)
    assert torch.equal(inputs.sample_rows(5, 20), torch.arange(5))
