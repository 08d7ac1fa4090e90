"""Parity of fa_attn_fwd (C ABI) with the fp64 oracle.

Tolerances: max-abs 1e-5 on O for fp32 inputs; max-abs 1e-2 on O for bf16
inputs with fp32 accumulation, on O as the kernel computes it (stored as
fp32); the bf16-stored O must be round-to-nearest-even of that fp32 O bit for
bit (its own max-abs is reported, not bounded); relative 1e-3 on LSE, gated as
|dLSE| <= 1e-3 * max(1, |LSE|) because a causal first row's LSE is a single
score that can be close to zero.  Every output buffer starts as NaN.
The two mid-size workloads are checked on every row; the 32768-key workload
on the first and last row of every 128-row query tile of every head (every
CTA and both of its tiles) plus a seeded sample.
"""
import math

import numpy as np
import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import O_TOL_BF16, attn_case, default_entry, ensure_built, nan_full, run_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


# ----------------------------------------------------------------- fp32 path
def test_f32_workload_n64_d64_uniform():
    w = inputs.ATTN_F32_64
    q, k, v = inputs.workload_attn_inputs(w)
    attn_case(q, k, v, w.causal, name=w.name).assert_ok()


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,M", [(1, 1), (63, 65), (130, 70), (70, 130), (200, 200)])
def test_f32_shapes(d, causal, N, M):
    q, k, v = inputs.attn_inputs(2, 2, N, M, d, torch.float32, seed=N * 7 + M + d)
    attn_case(q, k, v, causal).assert_ok()


@pytest.mark.parametrize("d", [16, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_many_row_blocks(d, causal):
    """Enough 64-row blocks (32 heads x 10) to fill the GPU twice over: the
    kernel takes 64 rows per CTA instead of 16; ragged last block."""
    q, k, v = inputs.attn_inputs(4, 8, 610, 610, d, torch.float32, seed=610 + d)
    attn_case(q, k, v, causal).assert_ok()


# ----------------------------------------------------------------- bf16 tensor-core path
BF16_SHAPES = [(1, 1), (1, 300), (127, 127), (128, 128), (129, 129), (255, 255), (256, 256), (257, 257),
               (300, 100), (100, 300), (513, 2100), (1000, 1000)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,M", BF16_SHAPES)
def test_bf16_shapes(d, causal, N, M):
    # fp32 O against the oracle, bf16 O bit-exact RN of it (attn_case)
    q, k, v = inputs.attn_inputs(1, 2, N, M, d, torch.bfloat16, seed=N + 3 * M + d + causal)
    attn_case(q, k, v, causal).assert_ok()


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_batched_heads_ragged(d):
    q, k, v = inputs.attn_inputs(2, 3, 700, 900, d, torch.bfloat16, seed=d)
    attn_case(q, k, v, True).assert_ok()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [300, 512])
def test_bf16_last_wave_single_tile_ctas(d, N):
    """Without the causal mask, a last wave of k <= SMs/2 (head, 256-row block)
    units runs as 2k CTAs of one 128-row tile each.  SMs + 8 units put 8 units
    there; with N = 300 some of those halves hold 44 rows or none."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = (sms + 8) // 2
    q, k, v = inputs.attn_inputs(1, H, N, 500, d, torch.bfloat16, seed=N + d)
    attn_case(q, k, v, False).assert_ok()


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_many_rescales(d):
    # K scaled x8 and sorted-growing score scale along the keys: the running
    # max rises repeatedly, exercising the conditional rescale of o~.
    q, k, v = inputs.attn_inputs(1, 2, 384, 1024, d, torch.float32, seed=11)
    ramp = torch.linspace(0.5, 8.0, 1024).reshape(1, 1, 1024, 1)
    k = (k * ramp).to(torch.bfloat16)
    attn_case(q.to(torch.bfloat16), k, v.to(torch.bfloat16), False).assert_ok()


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_equal_scores_closed_form(causal):
    # K = 0: every kept key weighs the same; O is the mean of the kept V rows.
    N, d = 300, 128
    q, _, v = inputs.attn_inputs(1, 1, N, N, d, torch.bfloat16, seed=4)
    k = torch.zeros_like(q)
    o, lse = run_attn(default_entry, q.cuda(), k.cuda(), v.cuda(), 1.0 / math.sqrt(d), causal, torch.float32)
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
    o, lse = run_attn(default_entry, q.cuda(), k.cuda(), v.cuda(), 0.125, True, torch.bfloat16)
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])


def tile_edge_rows(B, H, N, tile=128):
    """Flat query rows (b*H + h)*N + i: the first and the last row of every
    `tile`-row query tile of every (batch, head)."""
    starts = np.arange(0, N, tile)
    ends = np.minimum(starts + tile, N) - 1
    per_head = np.unique(np.concatenate([starts, ends]))
    heads = np.arange(B * H)[:, None] * N
    return (heads + per_head[None, :]).reshape(-1)


def _workload_case(w, rows=None, label="all rows"):
    """A full-size workload: O as computed within 1e-2 of the oracle, and on
    these seeded inputs the bf16-stored O (what the benchmark writes) within
    the same flat 1e-2 as well."""
    q, k, v = inputs.workload_attn_inputs(w)
    res = attn_case(q, k, v, w.causal, rows=rows, name=f"{w.name} ({label})")
    res.assert_ok()
    assert res.err_bf16 <= O_TOL_BF16, res.err_bf16


def test_bf16_workload_b4_h16_n2048_d64():
    _workload_case(inputs.ATTN_B4H16_2048_D64)


def test_bf16_workload_b2_h32_n8192_d128_causal():
    _workload_case(inputs.ATTN_B2H32_8192_D128_CAUSAL)


def test_bf16_workload_b1_h16_n32768_d128_causal_kscaled():
    w = inputs.ATTN_B1H16_32768_D128_CAUSAL
    rows = np.union1d(tile_edge_rows(w.B, w.H, w.N), inputs.sample_rows(w.B * w.H * w.N, 2048, seed=w.seed).numpy())
    _workload_case(w, rows, f"{len(rows)} rows: both ends of every 128-row tile")


def test_tile_edge_rows_cover_every_tile():
    rows = tile_edge_rows(1, 2, 300)
    assert list(rows) == [0, 127, 128, 255, 256, 299, 300, 427, 428, 555, 556, 599]


def test_bf16_deterministic():
    w = inputs.ATTN_B4H16_2048_D64
    q, k, v = (t.cuda() for t in inputs.workload_attn_inputs(w))
    outs = [run_attn(default_entry, q, k, v, w.scale, w.causal, torch.bfloat16) for _ in range(3)]
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_bf16_side_stream_and_no_lse():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 4, 600, 600, 128, torch.bfloat16, seed=3))
    ref, _ = run_attn(default_entry, q, k, v, 0.1, True, torch.bfloat16)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    o = nan_full(q.shape, torch.bfloat16)
    with torch.cuda.stream(s):
        o, lse = fattn.attn_fwd(q, k, v, 0.1, True, out=o, want_lse=False)
    s.synchronize()
    assert lse is None
    assert torch.equal(o, ref)


# ----------------------------------------------------------------- bottom-right causal
BR_SHAPES = [(300, 100), (100, 300), (257, 1000), (1000, 257), (1, 300), (300, 1), (129, 129)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,M", BR_SHAPES)
def test_bf16_bottom_right_causal(d, N, M):
    # key j kept for query i iff j <= i + (M - N); with N > M the first N - M
    # queries keep no key and must come back as O = 0, LSE = -inf
    q, k, v = inputs.attn_inputs(1, 2, N, M, d, torch.bfloat16, seed=N * 3 + M + d)
    attn_case(q, k, v, 2).assert_ok()


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("N,M", [(70, 130), (130, 70), (1, 40), (40, 1)])
def test_f32_bottom_right_causal(d, N, M):
    q, k, v = inputs.attn_inputs(2, 2, N, M, d, torch.float32, seed=N + M + d)
    attn_case(q, k, v, 2).assert_ok()


# ----------------------------------------------------------------- strided layouts
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.bfloat16, 128), (torch.float32, 64)])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_strided_bshd_layout(dtype, d, causal):
    B, H, N, M = 2, 3, 300, 520
    q, k, v = inputs.attn_inputs(B, H, N, M, d, dtype, seed=d + causal)

    def entry(q_, k_, v_, scale, causal_, out, lse, stream=None):
        # the same values laid out [B, N, H, d]; O written [B, N, H, d] in place
        qs, ks, vs = (t.permute(0, 2, 1, 3).contiguous() for t in (q_, k_, v_))
        o_bshd = torch.full((B, N, H, d), float("nan"), dtype=out.dtype, device=out.device)
        o2, _ = fattn.attn_fwd_strided(qs, ks, vs, scale, causal_, out=o_bshd, lse=lse, layout="bshd",
                                       stream=stream)
        assert o2.shape == (B, N, H, d)
        out.copy_(o_bshd.permute(0, 2, 1, 3))

    attn_case(q, k, v, causal, entry=entry).assert_ok()


def test_strided_padded_rows_bf16():
    # [B, H, N, d] views cut out of wider rows (row stride 2d) and an output
    # with a padded row stride as well; the padding must stay untouched
    B, H, N, M, d = 1, 2, 200, 333, 128
    q, k, v = inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=8)
    pads = []

    def entry(q_, k_, v_, scale, causal_, out, lse, stream=None):
        wide = lambda t: torch.cat([t, torch.zeros_like(t)], -1)[..., :d]
        ow_full = torch.zeros(B, H, N, 2 * d, dtype=out.dtype, device=out.device)
        ow_full[..., :d] = float("nan")
        ow = ow_full[..., :d]
        fattn.attn_fwd_strided(wide(q_), wide(k_), wide(v_), scale, causal_, out=ow, lse=lse, layout="bhsd",
                               stream=stream)
        pads.append(ow_full[..., d:].clone())
        out.copy_(ow)

    attn_case(q, k, v, 1, entry=entry).assert_ok()
    assert all(torch.all(p == 0).item() for p in pads)  # padding untouched
