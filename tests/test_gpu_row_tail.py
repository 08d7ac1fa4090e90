"""Run-time tail rows in the pipelined row kernels.

Rows of 8-64 KB go through a persistent kernel with one CTA per SM.  The
LSE-only kernel on rows above 16 KB and the softmax kernel on rows of 8-16 KB
take their first rounds of rows statically and the last rounds a chunk of rows
per request from a counter in device memory.  Each CUDA stream gets a counter
of its own, so launches that share a counter run one after another, and the
last CTA of a launch zeroes it for the next.  A row's arithmetic does not
depend on the CTA that computes it, so every launch of the same input must
give the same bits, and every row must be written: outputs start as NaN, so a
row that no CTA took fails.  Checked for launches back to back on one stream,
for launches on four streams at once, on 300 fresh streams at once (more than
the 256 counters: the rest split statically), and for the same calls captured
once in a CUDA graph and replayed (a captured launch keeps the static split:
the replays must still write every row, with the same bits as the direct
launch); the first result of each case is compared with the fp64 oracle (LSE
on every row, P on 64 sampled rows).  The fused cross-entropy (LSE kernel) and
the log-softmax (softmax kernel) are checked with tail rows too.  Tolerances
as in the row softmax tests: P max-abs 4e-3 (bf16) / 1e-5 (fp32), LSE relative
1e-3.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from online_softmax_10_gb300 import fattn, inputs
from parity import (LSE_REL, P_TOL_BF16, P_TOL_F32, ensure_built, lse_ok, nan_full, rows_cross_entropy,
                    rows_log_softmax, to_np)

pytestmark = pytest.mark.gpu

# (rows, cols, input dtype).  LSE kernel, tail rows above 16 KB: 64 KB rows
# one per request, 32 KB two; softmax kernel, tail rows of 8-16 KB: 16 KB
# rows four per request, 12 KB five, 16 KB fp32 four.  The tail is on when
# every CTA has at least 16 rounds of 64 KB (152 SMs: 2432 rows of 64 KB, 4864
# of 32 KB, 9728 of 16 KB, 12160 of 12 KB); ragged row counts.  (The other
# kernel splits the same rows statically, and so does the softmax kernel on
# the 8 KB fp32 rows.)
SHAPES = [(2500, 32768, torch.bfloat16), (4900, 16384, torch.bfloat16), (10000, 8192, torch.bfloat16),
          (12500, 6144, torch.bfloat16), (2500, 16384, torch.float32), (10001, 4096, torch.float32),
          (20000, 2048, torch.float32), (16 * 152 + 3, 32768, torch.bfloat16)]
P_SAMPLE = 64  # rows of P compared with the oracle (LSE: every row)


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _oracle_check(x_cpu, p, lse, lse_only):
    L_ref = oracle.logsumexp_rows(x_cpu)
    for got in (lse, lse_only):
        ok, rel = lse_ok(to_np(got), L_ref)
        assert ok, rel
    assert not torch.isnan(p).any().item(), "a row was never written"
    rows = inputs.sample_rows(x_cpu.shape[0], P_SAMPLE, seed=x_cpu.shape[1]).numpy()
    P_ref, _ = oracle.softmax_rows(x_cpu[torch.as_tensor(rows)])
    pg = to_np(p[torch.as_tensor(rows, device=p.device)])
    tol = P_TOL_BF16 if p.dtype == torch.bfloat16 else P_TOL_F32
    assert float(np.max(np.abs(pg - P_ref))) <= tol


def _run(x, p, lse, lse_only, stream=None):
    fattn.softmax_rows(x, out=p, lse=lse, stream=stream)
    fattn.logsumexp_rows(x, out=lse_only, stream=stream)


def _fresh(x):
    rows = x.shape[0]
    return nan_full(x.shape, x.dtype), nan_full((rows,), torch.float32), nan_full((rows,), torch.float32)


@pytest.mark.parametrize("rows,cols,din", SHAPES)
def test_back_to_back_launches(rows, cols, din):
    x_cpu = inputs.rows_inputs(rows, cols, din, seed=rows + cols, spike=12.0)
    x = x_cpu.cuda()
    outs = [_fresh(x) for _ in range(6)]
    for o in outs:  # no synchronisation between the launches
        _run(x, *o)
    assert fattn.device_status() == fattn.FA_OK
    _oracle_check(x_cpu, *outs[0])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


@pytest.mark.parametrize("rows,cols,din", [SHAPES[0], SHAPES[2], SHAPES[5]])
def test_graph_replays(rows, cols, din):
    x_cpu = inputs.rows_inputs(rows, cols, din, seed=rows * 3 + cols)
    x = x_cpu.cuda()
    ref = _fresh(x)
    _run(x, *ref)
    assert fattn.device_status() == fattn.FA_OK
    _oracle_check(x_cpu, *ref)
    out = _fresh(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _run(x, *out)  # the kernels' one-time set-up happens outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(x, *out)
    for _ in range(6):
        for t in out:
            t.fill_(float("nan"))
        g.replay()
        assert fattn.device_status() == fattn.FA_OK
        for a, b in zip(ref, out):
            assert torch.equal(a, b)


def test_streams_at_once():
    shapes = [SHAPES[0], SHAPES[2], SHAPES[3], SHAPES[5]]
    xs_cpu = [inputs.rows_inputs(r, c, d, seed=r + 7 * c) for r, c, d in shapes]
    xs = [x.cuda() for x in xs_cpu]
    streams = [torch.cuda.Stream() for _ in shapes]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[_fresh(x) for _ in range(6)] for x in xs]
    for k in range(6):  # interleaved, no synchronisation between the streams
        for x, s, o in zip(xs, streams, outs):
            with torch.cuda.stream(s):
                _run(x, *o[k], stream=s)
    for s in streams:
        assert fattn.device_status(stream=s) == fattn.FA_OK
    for x_cpu, o in zip(xs_cpu, outs):
        _oracle_check(x_cpu, *o[0])
        for other in o[1:]:
            for a, b in zip(o[0], other):
                assert torch.equal(a, b)


@pytest.mark.parametrize("rows,cols,din", [SHAPES[0], SHAPES[7]])
def test_cross_entropy_with_tail_rows(rows, cols, din):
    """The fused cross-entropy runs in the LSE kernel, so with tail rows the
    loss and LSE of each row must come from that row's label (the row index
    the ring carries), including ignored labels (-100, out of range)."""
    x_cpu = inputs.rows_inputs(rows, cols, din, seed=rows + 3 * cols)
    g = torch.Generator().manual_seed(rows)
    labels = torch.randint(0, cols, (rows,), generator=g)
    labels[::17] = -100
    labels[5::23] = cols + 3
    x, lab = x_cpu.cuda(), labels.cuda()
    for _ in range(3):  # back to back: each launch takes the counter over
        loss, lse = rows_cross_entropy(x, lab, want_lse=True)
    assert fattn.device_status() == fattn.FA_OK
    ref, L = oracle.cross_entropy_rows(x_cpu, labels)
    lg = to_np(loss)
    assert np.all(np.abs(lg - ref) <= LSE_REL * np.maximum(1.0, np.abs(ref))), float(np.max(np.abs(lg - ref)))
    assert np.all(lg[labels.numpy() < 0] == 0)
    ok, rel = lse_ok(to_np(lse), L)
    assert ok, rel


@pytest.mark.parametrize("rows,cols,din", [SHAPES[2], SHAPES[5]])
def test_log_softmax_with_tail_rows(rows, cols, din):
    """log p = x - LSE from the softmax kernel's log form with tail rows
    (rows of 8-16 KB): every row written, sampled rows against the oracle."""
    x_cpu = inputs.rows_inputs(rows, cols, din, seed=rows + 5 * cols)
    x = x_cpu.cuda()
    for _ in range(3):
        y, lse = rows_log_softmax(x, out_dtype=torch.float32)
    assert fattn.device_status() == fattn.FA_OK
    assert not torch.isnan(y).any().item(), "a row was never written"
    ok, rel = lse_ok(to_np(lse), oracle.logsumexp_rows(x_cpu))
    assert ok, rel
    sample = inputs.sample_rows(rows, P_SAMPLE, seed=cols).numpy()
    Y, _ = oracle.log_softmax_rows(x_cpu[torch.as_tensor(sample)])
    yg = to_np(y[torch.as_tensor(sample, device=y.device)])
    assert np.all(np.abs(yg - Y) <= 1e-5 + 1e-6 * np.abs(Y)), float(np.max(np.abs(yg - Y)))


class _RawStream:
    """A CUDA stream handle in the form the binding takes (``.cuda_stream``)."""

    def __init__(self, handle):
        self.cuda_stream = handle


def test_more_streams_than_counters():
    """Each stream keeps the counter it got first; once the 256 counters of the
    device are taken, further streams split their rows statically.  300 fresh
    non-blocking streams (created through the driver API: the framework's own
    stream objects come from a small pool), one launch on each, all in flight
    together: every result the same bits, and equal to the oracle.  (Runs last
    in this file: afterwards no new stream of this process gets a counter.)"""
    try:
        libcuda = ctypes.CDLL("libcuda.so.1")
    except OSError:
        pytest.skip("driver library not loadable")
    rows, cols, din = SHAPES[0]
    x_cpu = inputs.rows_inputs(rows, cols, din, seed=17)
    x = x_cpu.cuda()
    outs = [nan_full((rows,), torch.float32) for _ in range(300)]
    torch.cuda.synchronize()  # inputs and outputs ready before the non-blocking streams run
    handles = []
    try:
        for _ in range(300):
            h = ctypes.c_void_p()
            assert libcuda.cuStreamCreate(ctypes.byref(h), 1) == 0  # CU_STREAM_NON_BLOCKING
            handles.append(h)
        for h, o in zip(handles, outs):
            fattn.logsumexp_rows(x, out=o, stream=_RawStream(h.value))
        for h in handles:
            assert libcuda.cuStreamSynchronize(h) == 0
    finally:
        for h in handles:
            libcuda.cuStreamDestroy_v2(h)
    assert fattn.device_status() == fattn.FA_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ok, rel = lse_ok(to_np(outs[0]), oracle.logsumexp_rows(x_cpu))
    assert ok, rel
