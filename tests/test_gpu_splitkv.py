"""Split-KV attention (fa_attn_fwd_splitkv) against the fp64 oracle: the key
range of each query block is split over several CTAs and the normalised
partials are merged by their log-sum-exp.  Same tolerances as fa_attn_fwd
(bf16 inputs: |dO| <= 1e-2 on O as computed, stored as fp32; the bf16-stored O
equal to RN of it bit for bit; LSE relative 1e-3).  Outputs and the workspace
start as NaN (all bytes 0xFF), so a partial or an output the kernels never
write cannot pass."""
import pytest
import torch

from online_softmax_10_gb300 import fattn, inputs
from parity import attn_case, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def split_entry(splits):
    """An attention entry for parity.attn_case that goes through
    fa_attn_fwd_splitkv with a NaN-filled workspace."""
    def entry(q, k, v, scale, causal, out, lse, stream=None):
        B, H, N, d = q.shape
        S = splits if splits > 0 else fattn.splitkv_num_splits(B, H, N, k.shape[2], d, causal)
        need = fattn.splitkv_workspace_bytes(B, H, N, d, S)
        ws = torch.full((max(need, 1),), 255, dtype=torch.uint8, device=q.device) if need > 0 else None
        fattn.attn_fwd_splitkv(q, k, v, scale, causal, num_splits=S, workspace=ws, out=out, lse=lse, stream=stream)
    return entry


@pytest.mark.parametrize("splits", [2, 3, 7, 16, 0])
@pytest.mark.parametrize("B,H,N,M,d,causal", [
    (1, 2, 300, 2100, 128, False), (1, 2, 300, 2100, 64, True), (2, 1, 129, 1000, 128, True),
    (1, 3, 64, 8192, 128, False), (1, 2, 1000, 1000, 64, True), (1, 2, 300, 2100, 128, 2), (1, 2, 2100, 300, 64, 2)])
def test_splitkv_matches_oracle(splits, B, H, N, M, d, causal):
    q, k, v = inputs.attn_inputs(B, H, N, M, d, torch.bfloat16, seed=N + M + splits)
    attn_case(q, k, v, causal, entry=split_entry(splits)).assert_ok()


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
    rows = inputs.sample_rows(8 * 256, 512, seed=6).numpy()
    attn_case(q, k, v, False, rows=rows, entry=split_entry(0), name="splitkv B1 H8 N256 M65536 d128 (512 rows)"
              ).assert_ok()
