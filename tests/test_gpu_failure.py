"""Failure detection on the GPU without a fault: a kernel waits on an
mbarrier that nothing completes, its bounded wait gives up, the kernel
records FA_ERR_DEVICE_TIMEOUT in the device status word and returns, and the
CUDA context stays usable."""
import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_bounded_wait_times_out_and_context_survives():
    assert fattn.device_status(reset=True) == fattn.FA_OK
    assert fattn.selftest_wait_timeout(20000) == fattn.FA_ERR_DEVICE_TIMEOUT
    # the status was reset by the self-test; a normal call works afterwards
    assert fattn.device_status() == fattn.FA_OK
    x = inputs.rows_inputs(4, 1000, torch.float32, seed=0).cuda()
    p, _ = fattn.softmax_rows(x)
    torch.cuda.synchronize()
    assert abs(p.sum(1) - 1).max().item() < 1e-5
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 1, 256, 256, 128, torch.bfloat16, seed=1))
    fattn.attn_fwd(q, k, v, 0.1, True)
    assert fattn.device_status() == fattn.FA_OK
