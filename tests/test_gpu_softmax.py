"""Parity of fa_softmax_rows / fa_logsumexp_rows (C ABI) with the fp64 oracle.

Tolerances: probabilities max-abs 4e-3 when stored as bf16 (about one bf16
ulp at 1; the method states none) and 1e-5 when stored as fp32; LSE relative
1e-3 (gated as |dLSE| <= 1e-3 * max(1, |LSE|)); every row sums to 1 within
1e-2 (bf16) / 1e-5 (fp32).  Every output buffer starts as NaN, so an element
the kernels never write fails.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_10_gb300 import fattn, inputs
from parity import (P_TOL_BF16, P_TOL_F32, ensure_built, lse_ok, report, to_np, rows_log_softmax as log_softmax,
                    rows_logsumexp as logsumexp, rows_softmax as softmax)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(x_cpu, p, lse, rows=None, name=None):
    X = x_cpu if rows is None else x_cpu[torch.as_tensor(rows)]
    P_ref, L_ref = oracle.softmax_rows(X)
    pg = to_np(p if rows is None else p[torch.as_tensor(rows, device=p.device)])
    lg = to_np(lse if rows is None else lse[torch.as_tensor(rows, device=lse.device)])
    assert not np.any(np.isnan(pg)) and not np.any(np.isnan(lg)), "an output element was never written"
    tol = P_TOL_BF16 if p.dtype == torch.bfloat16 else P_TOL_F32
    err = float(np.max(np.abs(pg - P_ref)))
    assert err <= tol, err
    ok, rel = lse_ok(lg, L_ref)
    assert ok, rel
    sums = p.float().sum(1)
    stol = 1e-2 if p.dtype == torch.bfloat16 else 1e-5
    assert torch.all((sums - 1).abs() <= stol).item()
    if name is not None:
        report(name, rows=int(X.shape[0]), p_maxabs=err, lse_max_rel=rel,
               max_row_sum_err=float((sums - 1).abs().max().item()))


def test_workload_4096x32768_bf16():
    w = inputs.ROWS_4096x32768
    x = inputs.workload_rows_inputs(w)
    p, lse = softmax(x.cuda())
    assert fattn.device_status() == fattn.FA_OK
    _check(x, p, lse, name=w.name + " softmax (all rows)")   # every row against the oracle
    # the LSE-only kernel on the same input, every row
    lse2 = logsumexp(x.cuda())
    assert fattn.device_status() == fattn.FA_OK
    L_ref = oracle.logsumexp_rows(x)
    ok, rel = lse_ok(to_np(lse2), L_ref)
    assert ok, rel
    report(w.name + " logsumexp (all rows)", rows=w.rows, lse_max_rel=rel)
    assert torch.allclose(lse, lse2, rtol=1e-5, atol=1e-5)


COLS = [1, 2, 7, 8, 9, 31, 255, 256, 257, 1000, 2048, 2049, 4096, 8192, 32768, 65536, 65537, 100000]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("din,dout", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                      (torch.float32, torch.float32), (torch.float32, torch.bfloat16)])
def test_shapes_and_dtypes(cols, din, dout):
    rows = 5 if cols <= 65536 else 3
    x = inputs.rows_inputs(rows, cols, din, seed=cols, spike=20.0 if cols > 1 else None)
    p, lse = softmax(x.cuda(), out_dtype=dout)
    assert fattn.device_status() == fattn.FA_OK
    _check(x, p, lse)


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("din", [torch.bfloat16, torch.float32])
def test_logsumexp_shapes(cols, din):
    x = inputs.rows_inputs(6, cols, din, seed=cols + 1)
    lse = logsumexp(x.cuda())
    ok, rel = lse_ok(to_np(lse), oracle.logsumexp_rows(x))
    assert ok, rel


@pytest.mark.parametrize("cols,din", [(32776, torch.bfloat16), (131072, torch.bfloat16), (229376, torch.bfloat16),
                                      (262144, torch.bfloat16), (16388, torch.float32), (131072, torch.float32)])
@pytest.mark.parametrize("dout", [torch.bfloat16, torch.float32])
def test_cluster_rows(cols, din, dout):
    """Rows above 64 KB of whole 16-byte vectors: a cluster of 2 to 8 CTAs per
    row, each holding a 64 KB slice (the last one partly past the row end), the
    row's (max, sum) exchanged through distributed shared memory; more rows
    than clusters, so each cluster loops over rows (both exchange-slot sets)."""
    rows = 400 if cols * (2 if din == torch.bfloat16 else 4) <= 300000 else 160
    x = inputs.rows_inputs(rows, cols, din, seed=cols + rows)
    p, lse = softmax(x.cuda(), out_dtype=dout)
    lse2 = logsumexp(x.cuda())
    y, lse3 = log_softmax(x.cuda(), out_dtype=torch.float32)
    assert fattn.device_status() == fattn.FA_OK
    sample = inputs.sample_rows(rows, 24, seed=cols).numpy()
    _check(x, p, lse, sample)
    sub = x[torch.as_tensor(sample)]
    L_ref = oracle.logsumexp_rows(sub)
    for got in (lse2, lse3):
        ok, rel = lse_ok(to_np(got)[sample], L_ref)
        assert ok, rel
    Y, _ = oracle.log_softmax_rows(sub)
    yg = to_np(y)[sample]
    assert np.all(np.abs(yg - Y) <= 1e-5 + 1e-6 * np.abs(Y)), float(np.max(np.abs(yg - Y)))


@pytest.mark.parametrize("rows", [64, 153, 1000])
@pytest.mark.parametrize("cols,din", [(4096, torch.bfloat16), (4352, torch.bfloat16), (5000, torch.bfloat16),
                                      (6144, torch.bfloat16), (8192, torch.bfloat16),
                                      (16384, torch.bfloat16), (24576, torch.bfloat16), (32768, torch.bfloat16),
                                      (2560, torch.float32), (4096, torch.float32), (16384, torch.float32)])
@pytest.mark.parametrize("dout", [torch.bfloat16, torch.float32])
def test_pipelined_rows(rows, cols, din, dout):
    # rows of 8-64 KB take the persistent pipelined kernel (four consumer
    # groups up to 16 KB, eight for the LSE alone, some with part of each
    # thread's slice past the row end: 4352 and 5000 columns on 12 vectors per
    # thread); with more rows than SMs each CTA cycles its ring several times
    x = inputs.rows_inputs(rows, cols, din, seed=rows + cols)
    p, lse = softmax(x.cuda(), out_dtype=dout)
    lse2 = logsumexp(x.cuda())
    assert fattn.device_status() == fattn.FA_OK
    sample = inputs.sample_rows(rows, 40, seed=cols).numpy()
    _check(x, p, lse, sample)
    ok, rel = lse_ok(to_np(lse2)[sample], oracle.logsumexp_rows(x[torch.as_tensor(sample)]))
    assert ok, rel


@pytest.mark.parametrize("cols", [40, 1000, 8192, 32768, 100000])
@pytest.mark.parametrize("din", [torch.bfloat16, torch.float32])
def test_masked_rows_minus_inf(cols, din):
    """Masked logits (-inf), as padding masks make them: row r keeps only its
    first k_r entries (k_r from 1 to cols) and the last row a random tenth.
    exp(-inf - m) = 0, so p = 0 and log p = -inf there, and LSE is that of
    the kept entries.  Long masked runs leave whole per-thread slices at -inf."""
    x = inputs.rows_inputs(8, cols, torch.float32, seed=cols + 5)
    for r, k in enumerate([1, 3, 100, cols // 3, cols // 2 + 1, cols - 1, cols]):
        x[r, max(1, min(k, cols)):] = float("-inf")
    g = torch.Generator().manual_seed(cols)
    drop = torch.rand(cols, generator=g) < 0.9
    drop[0] = False
    x[7, drop] = float("-inf")
    x = x.to(din)
    p, lse = softmax(x.cuda())
    assert fattn.device_status() == fattn.FA_OK
    assert not torch.isnan(p).any().item()
    _check(x, p, lse)
    lse2 = logsumexp(x.cuda())
    ok, rel = lse_ok(to_np(lse2), oracle.logsumexp_rows(x))
    assert ok, rel
    y, _ = log_softmax(x.cuda(), out_dtype=torch.float32)
    Y, _ = oracle.log_softmax_rows(x)
    yg = to_np(y)
    assert np.array_equal(np.isneginf(yg), np.isneginf(Y))
    fin = np.isfinite(Y)
    assert np.all(np.abs(yg[fin] - Y[fin]) <= 1e-5 + 1e-6 * np.abs(Y[fin]))


@pytest.mark.parametrize("cols,din", [(1024, torch.bfloat16), (2048, torch.bfloat16), (4096, torch.bfloat16),
                                      (1024, torch.float32), (520, torch.float32)])
def test_many_rows_per_warp(cols, din):
    """More rows than resident warps: rows of up to 4 KB (8 KB for the LSE
    alone) go to one warp per row, each warp looping over rows with the next
    row loaded ahead; a seeded sample of rows against the oracle."""
    rows = 6000
    x = inputs.rows_inputs(rows, cols, din, seed=cols + 11)
    p, lse = softmax(x.cuda())
    lse2 = logsumexp(x.cuda())
    y, _ = log_softmax(x.cuda(), out_dtype=torch.float32)
    assert fattn.device_status() == fattn.FA_OK
    sample = inputs.sample_rows(rows, 64, seed=cols).numpy()
    _check(x, p, lse, sample)
    sub = x[torch.as_tensor(sample)]
    ok, rel = lse_ok(to_np(lse2)[sample], oracle.logsumexp_rows(sub))
    assert ok, rel
    Y, _ = oracle.log_softmax_rows(sub)
    yg = to_np(y)[sample]
    assert np.all(np.abs(yg - Y) <= 1e-5 + 1e-6 * np.abs(Y)), float(np.max(np.abs(yg - Y)))


def test_many_short_rows():
    x = inputs.rows_inputs(70000, 40, torch.bfloat16, seed=2)
    p, lse = softmax(x.cuda())
    rows = inputs.sample_rows(70000, 300).numpy()
    _check(x, p, lse, rows)


def test_shift_invariance_and_large_logits():
    x = inputs.rows_inputs(8, 4096, torch.float32, seed=3)
    xs = x + 1024.0                     # exp(x) alone would overflow fp32
    p0, l0 = softmax(x.cuda())
    p1, l1 = softmax(xs.cuda())
    assert torch.all(torch.isfinite(p1)).item()
    # exact against the oracle on the shifted (rounded) input
    _check(xs, p1, l1)
    # and close to the unshifted result: x + 1024 rounds x to 2^-13 in fp32
    assert (p1 - p0).abs().max().item() <= 2e-3
    assert ((l1 - 1024.0) - l0).abs().max().item() <= 1e-3


def test_constant_rows_closed_form():
    x = torch.full((4, 3000), -7.5, dtype=torch.bfloat16)
    p, lse = softmax(x.cuda(), out_dtype=torch.float32)
    assert (p - 1.0 / 3000).abs().max().item() <= 1e-9
    assert (lse.cpu().double() - (-7.5 + np.log(3000))).abs().max().item() <= 1e-5


def test_deterministic():
    x = inputs.rows_inputs(64, 32768, torch.bfloat16, seed=1).cuda()
    a, la = softmax(x)
    b, lb = softmax(x)
    assert torch.equal(a, b) and torch.equal(la, lb)
