"""Parity of fa_attn_fwd (C ABI) with the fp64 oracle.

Tolerances: max-abs 1e-5 on O for fp32 inputs; max-abs 1e-2 on O for bf16
inputs with fp32 accumulation when O is stored as fp32, plus the bf16 store's
half-ulp rounding (|O| * 2^-8) when O is stored as bf16; relative 1e-3 on LSE, gated as
|dLSE| <= 1e-3 * max(1, |LSE|) because a causal first row's LSE is a single
score that can be close to zero.
Full-size workloads are checked on a seeded sample of query rows (each row of
attention is independent, so a sampled row is an exact check of that row).
"""
import math

import numpy as np
import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import O_TOL_BF16, attn_case, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


# ----------------------------------------------------------------- fp32 path
def test_f32_workload_n64_d64_uniform():
    w = inputs.ATTN_F32_64
    q, k, v = inputs.workload_attn_inputs(w)
    err, ratio, ok, rel = attn_case(q, k, v, w.causal)
    assert ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,M", [(1, 1), (63, 65), (130, 70), (70, 130), (200, 200)])
def test_f32_shapes(d, causal, N, M):
    q, k, v = inputs.attn_inputs(2, 2, N, M, d, torch.float32, seed=N * 7 + M + d)
    err, ratio, ok, rel = attn_case(q, k, v, causal)
    assert ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("d", [16, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_many_row_blocks(d, causal):
    """Enough 64-row blocks (32 heads x 10) to fill the GPU twice over: the
    kernel takes 64 rows per CTA instead of 16; ragged last block."""
    q, k, v = inputs.attn_inputs(4, 8, 610, 610, d, torch.float32, seed=610 + d)
    err, ratio, ok, rel = attn_case(q, k, v, causal)
    assert ratio <= 1.0, err
    assert ok, rel


# ----------------------------------------------------------------- bf16 tensor-core path
BF16_SHAPES = [(1, 1), (1, 300), (127, 127), (128, 128), (129, 129), (255, 255), (256, 256), (257, 257),
               (300, 100), (100, 300), (513, 2100), (1000, 1000)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,M", BF16_SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_shapes(d, causal, N, M, out):
    q, k, v = inputs.attn_inputs(1, 2, N, M, d, torch.bfloat16, seed=N + 3 * M + d + causal)
    err, ratio, ok, rel = attn_case(q, k, v, causal, out_dtype=torch.float32 if out == "f32" else None)
    assert ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_fp32_output(d):
    q, k, v = inputs.attn_inputs(2, 3, 700, 900, d, torch.bfloat16, seed=d)
    err, ratio, ok, rel = attn_case(q, k, v, True, out_dtype=torch.float32)
    assert err <= O_TOL_BF16 and ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_many_rescales(d):
    # K scaled x8 and sorted-growing score scale along the keys: the running
    # max rises repeatedly, exercising the conditional rescale of o~.
    q, k, v = inputs.attn_inputs(1, 2, 384, 1024, d, torch.float32, seed=11)
    ramp = torch.linspace(0.5, 8.0, 1024).reshape(1, 1, 1024, 1)
    k = (k * ramp).to(torch.bfloat16)
    err, ratio, ok, rel = attn_case(q.to(torch.bfloat16), k, v.to(torch.bfloat16), False,
                                    out_dtype=torch.float32)
    assert ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_equal_scores_closed_form(causal):
    # K = 0: every kept key weighs the same; O is the mean of the kept V rows.
    N, d = 300, 128
    q, _, v = inputs.attn_inputs(1, 1, N, N, d, torch.bfloat16, seed=4)
    k = torch.zeros_like(q)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), 1.0 / math.sqrt(d), causal, out_dtype=torch.float32)
    o, lse = o.cpu().double(), lse.cpu().double()
    vd = v.double()[0, 0]
    if causal:
        ref = torch.cumsum(vd, 0) / torch.arange(1, N + 1, dtype=torch.float64)[:, None]
        lref = torch.log(torch.arange(1, N + 1, dtype=torch.float64))
    else:
        ref = vd.mean(0).expand(N, d)
        lref = torch.full((N,), math.log(N), dtype=torch.float64)
    assert (o[0, 0] - ref).abs().max().item() <= O_TOL_BF16
    assert (lse[0, 0] - lref).abs().max().item() <= 1e-3 * max(1.0, math.log(N))


def test_bf16_causal_first_row_is_first_value():
    q, k, v = inputs.attn_inputs(2, 2, 260, 260, 64, torch.bfloat16, seed=9)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), 0.125, True)
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])


def _workload_sampled(w, nsample):
    """The full-size workload in the benchmark's launch configuration (bf16 O),
    then the same inputs with fp32 O; a seeded sample of rows vs the oracle."""
    q, k, v = inputs.workload_attn_inputs(w)
    rows = inputs.sample_rows(w.B * w.H * w.N, nsample, seed=w.seed).numpy()
    for out in (None, torch.float32):
        err, ratio, ok, rel = attn_case(q, k, v, w.causal, out_dtype=out, rows=rows)
        assert ratio <= 1.0, (out, err)
        assert ok, rel


def test_bf16_workload_b4_h16_n2048_d64():
    _workload_sampled(inputs.ATTN_B4H16_2048_D64, 1024)


def test_bf16_workload_b2_h32_n8192_d128_causal():
    _workload_sampled(inputs.ATTN_B2H32_8192_D128_CAUSAL, 512)


def test_bf16_workload_b1_h16_n32768_d128_causal_kscaled():
    _workload_sampled(inputs.ATTN_B1H16_32768_D128_CAUSAL, 256)


def test_bf16_deterministic():
    w = inputs.ATTN_B4H16_2048_D64
    q, k, v = (t.cuda() for t in inputs.workload_attn_inputs(w))
    o1, l1 = fattn.attn_fwd(q, k, v, w.scale, w.causal)
    o2, l2 = fattn.attn_fwd(q, k, v, w.scale, w.causal)
    o3, l3 = fattn.attn_fwd(q, k, v, w.scale, w.causal)
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    assert torch.equal(l1, l2) and torch.equal(l1, l3)


def test_bf16_side_stream_and_no_lse():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 4, 600, 600, 128, torch.bfloat16, seed=3))
    ref, _ = fattn.attn_fwd(q, k, v, 0.1, True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, lse = fattn.attn_fwd(q, k, v, 0.1, True, want_lse=False)
    s.synchronize()
    assert lse is None
    assert torch.equal(o, ref)


# ----------------------------------------------------------------- bottom-right causal
BR_SHAPES = [(300, 100), (100, 300), (257, 1000), (1000, 257), (1, 300), (300, 1), (129, 129)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,M", BR_SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_bottom_right_causal(d, N, M, out):
    # key j kept for query i iff j <= i + (M - N); with N > M the first N - M
    # queries keep no key and must come back as O = 0, LSE = -inf
    q, k, v = inputs.attn_inputs(1, 2, N, M, d, torch.bfloat16, seed=N * 3 + M + d)
    err, ratio, ok, rel = attn_case(q, k, v, 2, out_dtype=torch.float32 if out == "f32" else None)
    assert ratio <= 1.0, err
    assert ok, rel


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("N,M", [(70, 130), (130, 70), (1, 40), (40, 1)])
def test_f32_bottom_right_causal(d, N, M):
    q, k, v = inputs.attn_inputs(2, 2, N, M, d, torch.float32, seed=N + M + d)
    err, ratio, ok, rel = attn_case(q, k, v, 2)
    assert ratio <= 1.0, err
    assert ok, rel


# ----------------------------------------------------------------- strided layouts
def _oracle_check(q, k, v, causal, o, lse, o_tol_rel=None):
    import oracle
    d = q.shape[-1]
    O_ref, L_ref = oracle.attn_fwd(q, k, v, 1.0 / math.sqrt(d), causal)
    og = o.float().cpu().double().numpy()
    tol = (1e-5 if q.dtype == torch.float32 else 1e-2) + (2.0 ** -8 * np.abs(O_ref) if o.dtype == torch.bfloat16 else 0)
    assert np.all(np.abs(og - O_ref) <= tol), float(np.max(np.abs(og - O_ref)))
    from parity import lse_ok
    ok, rel = lse_ok(lse.cpu().double().numpy(), L_ref)
    assert ok, rel


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.bfloat16, 128), (torch.float32, 64)])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_strided_bshd_layout(dtype, d, causal):
    B, H, N, M = 2, 3, 300, 520
    q, k, v = inputs.attn_inputs(B, H, N, M, d, dtype, seed=d + causal)
    # the same values laid out [B, N, H, d]
    qs, ks, vs = (t.permute(0, 2, 1, 3).contiguous().cuda() for t in (q, k, v))
    o, lse = fattn.attn_fwd_strided(qs, ks, vs, causal=causal, layout="bshd")
    assert fattn.device_status() == fattn.FA_OK
    assert o.shape == (B, N, H, d)
    _oracle_check(q, k, v, causal, o.permute(0, 2, 1, 3), lse)


def test_strided_padded_rows_bf16():
    # [B, H, N, d] views cut out of wider rows (row stride 2d) and an output
    # with a padded row stride as well
    B, H, N, M, d = 1, 2, 200, 333, 128
    q, k, v = inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=8)
    wide = lambda t: torch.cat([t, torch.zeros_like(t)], -1).cuda()[..., :d]
    qw, kw, vw = wide(q), wide(k), wide(v)
    ow = torch.zeros(B, H, N, 2 * d, dtype=torch.bfloat16, device="cuda")[..., :d]
    o, lse = fattn.attn_fwd_strided(qw, kw, vw, causal=1, out=ow, layout="bhsd")
    assert fattn.device_status() == fattn.FA_OK
    _oracle_check(q, k, v, 1, o, lse)
    assert torch.all(ow.as_strided((B, H, N, d), (H * N * 2 * d, N * 2 * d, 2 * d, 1), d) == 0)  # padding untouched
