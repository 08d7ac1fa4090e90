"""Shared helpers of the GPU parity tests: run a case through the C ABI and
compare with the oracle at the stated tolerances.

Every output buffer handed to the library is filled with NaN first, so an
element the kernels never write cannot pass (a fresh allocation could
otherwise return an earlier call's correct values).

bf16 inputs are run twice, once storing O as fp32 and once as bf16.  The fp32
O is what the kernel computed and is held to max-abs 1e-2.  The bf16 O must be
bit-identical to round-to-nearest-even of the fp32 O (both epilogues round the
same fp32 products), and its own max-abs error against the oracle is reported
as it stands (``report``), not held to a widened bound.
"""
import json
import math
import os

import numpy as np
import torch

import oracle
from online_softmax_10_gb300 import build as fbuild
from online_softmax_10_gb300 import fattn, inputs

# Tolerances (stated for the method; see the module docstrings of the tests)
O_TOL_F32 = 1e-5      # max-abs on O, fp32 inputs
O_TOL_BF16 = 1e-2     # max-abs on O, bf16 inputs, fp32 accumulation (O as computed, stored as fp32)
LSE_REL = 1e-3        # relative on LSE (gated as |dLSE| <= 1e-3 * max(1, |LSE|))
P_TOL_BF16 = 4e-3     # max-abs on softmax probabilities stored as bf16 (about one bf16 ulp at 1)
P_TOL_F32 = 1e-5      # max-abs on softmax probabilities stored as fp32


def ensure_built():
    fbuild.build()
    fattn.lib()


def report(case: str, **values):
    """Append one JSON line of measured parity figures to the file named by
    FATTN_PARITY_REPORT (nothing happens when it is unset)."""
    path = os.environ.get("FATTN_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": case, **values}) + "\n")


def nan_full(shape, dtype, device="cuda"):
    """An output buffer poisoned with NaN."""
    return torch.full(tuple(shape), float("nan"), dtype=dtype, device=device)


def lse_ok(lse_gpu, lse_ref):
    """|dLSE| <= 1e-3 * max(1, |LSE|); an LSE of -inf (a query with no kept
    key) must be -inf on both sides."""
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    if np.any(np.isnan(lse_gpu)):
        return False, float("nan")
    empty = np.isneginf(lse_ref)
    if not np.array_equal(np.isneginf(lse_gpu), empty):
        return False, float("inf")
    g, r = lse_gpu[~empty], lse_ref[~empty]
    if g.size == 0:
        return True, 0.0
    d = np.abs(g - r)
    return bool(np.all(d <= LSE_REL * np.maximum(1.0, np.abs(r)))), float(np.max(d / np.maximum(np.abs(r), 1e-30)))


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def bf16_bits_equal_rn(o_bf16, o_f32):
    """True when every element of o_bf16 is round-to-nearest-even of o_f32."""
    return torch.equal(o_bf16.view(torch.int16), o_f32.to(torch.bfloat16).view(torch.int16))


def default_entry(q, k, v, scale, causal, out, lse, stream=None):
    fattn.attn_fwd(q, k, v, scale, causal, out=out, lse=lse, stream=stream)


def run_attn(entry, qd, kd, vd, scale, causal, out_dtype, stream=None):
    """One call of an attention entry point on device tensors, into
    NaN-poisoned O and LSE; returns (O, LSE) on the device."""
    B, H, N, d = qd.shape
    o = nan_full((B, H, N, d), out_dtype, qd.device)
    lse = nan_full((B, H, N), torch.float32, qd.device)
    entry(qd, kd, vd, scale, causal, o, lse, stream)
    assert fattn.device_status(stream=stream) == fattn.FA_OK
    return o, lse


class AttnResult:
    """Measured parity of one attention case."""

    def __init__(self, err, ratio, lse_ok, lse_rel, err_bf16=None, bf16_over=None, rows=0):
        self.err = err            # max-abs of O as computed (fp32 O) against the oracle
        self.ratio = ratio        # worst |dO| / tolerance
        self.lse_ok = lse_ok
        self.lse_rel = lse_rel
        self.err_bf16 = err_bf16  # max-abs of the bf16-stored O against the oracle (reported)
        self.bf16_over = bf16_over  # elements of the bf16-stored O beyond 1e-2 (reported)
        self.rows = rows          # query rows compared

    def assert_ok(self):
        assert self.ratio <= 1.0, self.err
        assert self.lse_ok, self.lse_rel


def attn_case(q, k, v, causal, rows=None, stream=None, entry=None, name=None, scale=None):
    """Run an attention entry point (default fa_attn_fwd) on CPU tensors q, k,
    v copied to the device, and the oracle on the same bits.

    fp32 inputs: one call, |dO| <= 1e-5.  bf16 inputs: a call with fp32 O
    (|dO| <= 1e-2) and one with bf16 O, which must equal RN(fp32 O) bit for
    bit; both calls' LSE must agree bit for bit.  ``rows`` selects flat query
    rows (b*H + h)*N + i for the comparison (all rows when None)."""
    entry = entry or default_entry
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o32, lse = run_attn(entry, qd, kd, vd, scale, causal, torch.float32, stream)
    o16 = None
    if q.dtype == torch.bfloat16:
        o16, lse16 = run_attn(entry, qd, kd, vd, scale, causal, torch.bfloat16, stream)
        assert bf16_bits_equal_rn(o16, o32), "bf16 O is not RN(fp32 O) of the same kernel"
        assert torch.equal(lse16, lse), "LSE differs between the fp32-O and bf16-O calls"
    if rows is None:
        O_ref, L_ref = oracle.attn_fwd(q, k, v, scale, causal)
        O_ref, L_ref = O_ref.reshape(-1, d), L_ref.reshape(-1)
        sel = slice(None)
    else:
        sel = np.asarray(rows)
        O_ref, L_ref = oracle.attn_fwd(q, k, v, scale, causal, rows=sel)
    O_g = to_np(o32).reshape(-1, d)[sel]
    L_g = to_np(lse).reshape(-1)[sel]
    assert not np.any(np.isnan(O_g)) and not np.any(np.isnan(L_g)), "an output element was never written"
    assert np.all(np.isfinite(O_g))
    tol = O_TOL_F32 if q.dtype == torch.float32 else O_TOL_BF16
    diff = np.abs(O_g - O_ref)
    err = float(np.max(diff))
    ok, rel = lse_ok(L_g, L_ref)
    res = AttnResult(err, err / tol, ok, rel, rows=O_ref.shape[0])
    if o16 is not None:
        d16 = np.abs(to_np(o16).reshape(-1, d)[sel] - O_ref)
        res.err_bf16 = float(np.max(d16))
        res.bf16_over = int(np.sum(d16 > O_TOL_BF16))
    if name is not None:
        report(name, rows=res.rows, o_maxabs=res.err, o_bf16_maxabs=res.err_bf16,
               o_bf16_elems_over_1e_2=res.bf16_over, lse_max_rel=res.lse_rel)
    return res


def rows_softmax(x, out_dtype=None):
    """fa_softmax_rows into NaN-filled P and LSE; returns (P, LSE)."""
    p = nan_full(x.shape, out_dtype or x.dtype, x.device)
    lse = nan_full((x.shape[0],), torch.float32, x.device)
    return fattn.softmax_rows(x, out=p, lse=lse)


def rows_logsumexp(x):
    """fa_logsumexp_rows into a NaN-filled LSE."""
    return fattn.logsumexp_rows(x, out=nan_full((x.shape[0],), torch.float32, x.device))


def rows_log_softmax(x, out_dtype=None):
    """fa_log_softmax_rows into NaN-filled Y and LSE; returns (Y, LSE)."""
    y = nan_full(x.shape, out_dtype or x.dtype, x.device)
    lse = nan_full((x.shape[0],), torch.float32, x.device)
    return fattn.log_softmax_rows(x, out=y, lse=lse)


def rows_cross_entropy(x, labels, want_lse=False):
    """fa_cross_entropy_rows into a NaN-filled loss (and LSE); returns (loss, LSE)."""
    loss = nan_full((x.shape[0],), torch.float32, x.device)
    lse = nan_full((x.shape[0],), torch.float32, x.device) if want_lse else None
    return fattn.cross_entropy_rows(x, labels, loss=loss, lse=lse, want_lse=want_lse)


def workload_attn(w):
    return inputs.workload_attn_inputs(w)
