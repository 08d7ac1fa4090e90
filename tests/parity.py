"""Shared helpers of the GPU parity tests: run a case through the C ABI and
compare with the oracle at the stated tolerances."""
import math

import numpy as np
import torch

import oracle
from online_softmax_10_gb300 import build as fbuild
from online_softmax_10_gb300 import fattn, inputs

# Tolerances (stated for the method; see the module docstrings of the tests)
O_TOL_F32 = 1e-5      # max-abs on O, fp32 inputs
O_TOL_BF16 = 1e-2     # max-abs on O, bf16 inputs, fp32 accumulation (fp32 O as stored)
BF16_HALF_ULP_REL = 2.0 ** -8  # storing O as bf16 adds up to half an ulp: <= |O| * 2^-8
LSE_REL = 1e-3        # relative on LSE (gated as |dLSE| <= 1e-3 * max(1, |LSE|))
P_TOL_BF16 = 4e-3     # max-abs on softmax probabilities stored as bf16 (about one bf16 ulp at 1)
P_TOL_F32 = 1e-5      # max-abs on softmax probabilities stored as fp32


def ensure_built():
    fbuild.build()
    fattn.lib()


def lse_ok(lse_gpu, lse_ref):
    """|dLSE| <= 1e-3 * max(1, |LSE|); an LSE of -inf (a query with no kept
    key) must be -inf on both sides."""
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
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


def attn_case(q, k, v, causal, out_dtype=None, rows=None, stream=None):
    """Run fa_attn_fwd on CPU tensors q, k, v (copied to the device) and the
    oracle on the same bits, and measure O against the tolerance.

    fp32 inputs: |dO| <= 1e-5.  bf16 inputs: |dO| <= 1e-2 when O is stored as
    fp32; when O is stored as bf16 the store's own rounding (at most half an
    ulp, |O| * 2^-8) is added to the 1e-2.
    Returns (max-abs O error, worst error / tolerance, LSE ok, LSE max rel)."""
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, causal, out_dtype=out_dtype, stream=stream)
    assert fattn.device_status(stream=stream) == fattn.FA_OK
    o, lse = to_np(o), to_np(lse)
    if rows is None:
        O_ref, L_ref = oracle.attn_fwd(q, k, v, scale, causal)
        O_g, L_g = o, lse
    else:
        rows = np.asarray(rows)
        O_ref, L_ref = oracle.attn_fwd(q, k, v, scale, causal, rows=rows)
        O_g = o.reshape(-1, d)[rows]
        L_g = lse.reshape(-1)[rows]
    assert np.all(np.isfinite(O_g)) and not np.any(np.isnan(L_g))
    diff = np.abs(O_g - O_ref)
    if q.dtype == torch.float32:
        tol = np.full_like(O_ref, O_TOL_F32)
    elif (out_dtype or q.dtype) == torch.bfloat16:
        tol = O_TOL_BF16 + BF16_HALF_ULP_REL * np.abs(O_ref)
    else:
        tol = np.full_like(O_ref, O_TOL_BF16)
    ratio = float(np.max(diff / tol))
    ok, rel = lse_ok(L_g, L_ref)
    return float(np.max(diff)), ratio, ok, rel


def workload_attn(w):
    return inputs.workload_attn_inputs(w)
