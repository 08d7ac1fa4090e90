"""fa_log_softmax_rows and fa_cross_entropy_rows (C ABI) against the fp64 oracle.

Tolerances: log-softmax 1e-5 + 1e-6 |y| when stored as fp32, plus the bf16
store's half ulp (|y| * 2^-8) when stored as bf16; cross-entropy loss and LSE
gated like LSE everywhere: |d| <= 1e-3 * max(1, |value|).  Every output
buffer starts as NaN."""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_10_gb300 import fattn, inputs
from parity import LSE_REL, ensure_built, lse_ok, rows_cross_entropy, rows_log_softmax, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


COLS = [1, 7, 256, 1000, 8192, 32768, 65536, 100000]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [3, 200])
@pytest.mark.parametrize("din,dout", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                      (torch.float32, torch.float32)])
def test_log_softmax(cols, rows, din, dout):
    if rows * cols > 4_000_000:
        rows = 40
    x = inputs.rows_inputs(rows, cols, din, seed=cols + rows, spike=20.0 if cols > 1 else None)
    y, lse = rows_log_softmax(x.cuda(), out_dtype=dout)
    assert fattn.device_status() == fattn.FA_OK
    Y, L = oracle.log_softmax_rows(x)
    yg = to_np(y)
    tol = 1e-5 + (2.0 ** -8 if dout == torch.bfloat16 else 1e-6) * np.abs(Y)
    assert np.all(np.abs(yg - Y) <= tol), float(np.max(np.abs(yg - Y) - tol))
    ok, rel = lse_ok(to_np(lse), L)
    assert ok, rel


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("din", [torch.bfloat16, torch.float32])
def test_cross_entropy(cols, din):
    rows = 300 if cols <= 32768 else 60
    x = inputs.rows_inputs(rows, cols, din, seed=cols + 7)
    g = torch.Generator().manual_seed(cols)
    labels = torch.randint(0, cols, (rows,), generator=g)
    labels[::17] = -100          # ignored rows
    labels[5::23] = cols + 3     # out of range: ignored too
    loss, lse = rows_cross_entropy(x.cuda(), labels.cuda(), want_lse=True)
    assert fattn.device_status() == fattn.FA_OK
    ref, L = oracle.cross_entropy_rows(x, labels)
    lg = to_np(loss)
    assert np.all(np.abs(lg - ref) <= LSE_REL * np.maximum(1.0, np.abs(ref))), float(np.max(np.abs(lg - ref)))
    assert np.all(lg[labels.numpy() < 0] == 0)
    ok, rel = lse_ok(to_np(lse), L)
    assert ok, rel


def test_cross_entropy_worked_example():
    x = torch.tensor([[2.0, 1.0, 0.1]], dtype=torch.float32).cuda()
    loss, _ = rows_cross_entropy(x, torch.tensor([0]).cuda())
    assert abs(loss.item() - 0.4170) < 5e-4   # the page's printed value
