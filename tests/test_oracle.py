"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Nothing here runs on a GPU.  Each check pins the oracle to something other
than itself: the pages' printed worked examples (tests/golden), invariants the
pages state (rows sum to one, shift invariance, the online result equals the
three-pass one), closed forms, and special cases that a library routine
computes independently (torch fp64 softmax / logsumexp / SDPA on the CPU).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import online

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
TOL = GOLD["tolerance_abs"]


# ---------------------------------------------------------------- worked examples
def test_ex1_softmax_printed_values():
    ex = GOLD["ex1_softmax"]
    p, lse = oracle.softmax_rows(np.array([ex["logits"]]))
    assert np.max(np.abs(p[0] - ex["p"])) < TOL
    # sum of exp(x - max) is exp(LSE - max)
    assert abs(math.exp(lse[0] - ex["max"]) - ex["sum_exp"]) < TOL


def test_ex2_cross_entropy_printed_value():
    ex = GOLD["ex2_cross_entropy"]
    _, lse = oracle.softmax_rows(np.array([ex["logits"]]))
    # -log p_label = LSE - z_label   (log p_j = z_j - LSE)
    loss = lse[0] - ex["logits"][ex["label"]]
    assert abs(loss - ex["loss"]) < TOL


def test_ex3_attention_printed_values():
    ex = GOLD["ex3_attention"]
    Q = np.array(ex["Q"])[None, None]
    K = np.array(ex["K"])[None, None]
    V = np.array(ex["V"])[None, None]
    O, lse = oracle.attn_fwd(Q, K, V, scale=ex["scale"])
    assert np.max(np.abs(O[0, 0] - np.array(ex["O"]))) < TOL
    # the page's per-row sum of exp(S - rowmax): exp(LSE - rowmax(S))
    S = np.array(ex["S"])
    assert np.max(np.abs(np.exp(lse[0, 0] - S.max(1)) - ex["row_sum_exp"])) < 2 * TOL


def test_ex3_softmax_of_printed_scores():
    ex = GOLD["ex3_attention"]
    p, _ = oracle.softmax_rows(np.array(ex["S"]))
    assert np.max(np.abs(p - np.array(ex["P"]))) < TOL


def _ex4_as_attention():
    # one query, scores s_j = q . k_j with scale 1: q = [1, 0], k_j = [s_j, 0]
    ex = GOLD["ex4_online_merge"]
    s = np.array(ex["scores"])
    Q = np.array([[1.0, 0.0]])[None, None]
    K = np.stack([s, np.zeros_like(s)], 1)[None, None]
    V = np.array(ex["V"])[None, None]
    return ex, Q, K, V


def test_ex4_global_softmax_printed_values():
    ex, Q, K, V = _ex4_as_attention()
    O, lse = oracle.attn_fwd(Q, K, V, scale=1.0)
    assert np.max(np.abs(O[0, 0, 0] - ex["global_O"])) < TOL
    assert abs(math.exp(lse[0, 0, 0] - ex["global_max"]) - ex["global_sum_exp"]) < TOL
    p, _ = oracle.softmax_rows(np.array([ex["scores"]]))
    assert np.max(np.abs(p[0] - ex["global_probs"])) < TOL


def test_ex4_blockwise_merge_printed_values():
    ex = GOLD["ex4_online_merge"]
    x, V = np.array(ex["scores"]), np.array(ex["V"])
    # block 1 alone
    o1, m1, l1 = online.blockwise_attention_row(x[:2], V[:2], 2)
    assert m1 == ex["block1"]["m"] and abs(l1 - ex["block1"]["l"]) < TOL
    assert np.max(np.abs(o1 - ex["block1"]["o"])) < TOL
    o2, m2, l2 = online.blockwise_attention_row(x[2:], V[2:], 2)
    assert m2 == ex["block2"]["m"] and abs(l2 - ex["block2"]["l"]) < TOL
    assert np.max(np.abs(o2 - ex["block2"]["o"])) < TOL
    o, m, l = online.blockwise_attention_row(x, V, ex["blocks"])
    assert m == ex["global_max"] and abs(l - ex["merged_l"]) < TOL
    assert np.max(np.abs(o - ex["online_O"])) < TOL


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("cols", [1, 2, 7, 129, 4096])
def test_rows_sum_to_one_and_log_identity(cols):
    rng = np.random.default_rng(cols)
    X = rng.normal(0, 3, size=(5, cols))
    P, lse = oracle.softmax_rows(X)
    assert np.max(np.abs(P.sum(1) - 1)) < 1e-12
    assert np.all(P > 0)
    # log p_j = z_j - LSE(z)
    assert np.max(np.abs(np.log(P) - (X - lse[:, None]))) < 1e-10


def test_shift_invariance_and_overflow():
    rng = np.random.default_rng(7)
    X = rng.normal(0, 3, size=(4, 333))
    P, lse = oracle.softmax_rows(X)
    for c in (-50.0, 1000.0, 1e5):
        P2, lse2 = oracle.softmax_rows(X + c)
        assert np.all(np.isfinite(P2))
        # x + c is rounded to the ulp of |c|; p moves by at most about that much
        tol = 1e-12 * max(1.0, abs(c) / 100)
        assert np.max(np.abs(P2 - P)) < tol
        assert np.max(np.abs((lse2 - c) - lse)) < tol
    # the page's example lifted by 1000: a naive exp would overflow
    p, _ = oracle.softmax_rows(np.array([[1002.0, 1001.0, 1000.1]]))
    assert np.max(np.abs(p[0] - GOLD["ex1_softmax"]["p"])) < TOL


def test_two_element_closed_form():
    a, b = 0.3, -1.7
    p, lse = oracle.softmax_rows(np.array([[a, b]]))
    assert abs(p[0, 0] - 1 / (1 + math.exp(b - a))) < 1e-15
    assert abs(lse[0] - (a + math.log1p(math.exp(b - a)))) < 1e-15


def test_constant_row_closed_form():
    for n in (1, 3, 1000):
        p, lse = oracle.softmax_rows(np.full((1, n), 2.5))
        assert np.max(np.abs(p - 1.0 / n)) < 1e-15
        assert abs(lse[0] - (2.5 + math.log(n))) < 1e-12


# ---------------------------------------------------------------- library routines
@pytest.mark.parametrize("shape", [(3, 5), (17, 1000), (2, 32768)])
def test_softmax_matches_torch_fp64(shape):
    g = torch.Generator().manual_seed(sum(shape))
    X = torch.randn(*shape, generator=g, dtype=torch.float64) * 3
    P, lse = oracle.softmax_rows(X)
    assert np.max(np.abs(P - torch.softmax(X, -1).numpy())) < 1e-14
    assert np.max(np.abs(lse - torch.logsumexp(X, -1).numpy())) < 1e-12


def _torch_attention(Q, K, V, scale, causal):
    Q, K, V = (torch.as_tensor(np.asarray(t)) for t in (Q, K, V))
    return torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal, scale=scale)


@pytest.mark.parametrize("B,H,N,M,d,causal", [
    (1, 1, 1, 1, 4, False), (2, 3, 17, 17, 8, False), (2, 3, 17, 17, 8, True),
    (1, 2, 9, 31, 16, True), (1, 2, 31, 9, 16, True), (1, 1, 65, 130, 64, False)])
def test_attention_matches_torch_sdpa_fp64(B, H, N, M, d, causal):
    rng = np.random.default_rng(B * 1000 + N * 10 + M)
    Q = rng.normal(size=(B, H, N, d))
    K = rng.normal(size=(B, H, M, d))
    V = rng.normal(size=(B, H, M, d))
    scale = 1 / math.sqrt(d)
    O, lse = oracle.attn_fwd(Q, K, V, scale, causal)
    ref = _torch_attention(Q, K, V, scale, causal).numpy()
    assert np.max(np.abs(O - ref)) < 1e-12
    # LSE against torch.logsumexp of the masked score matrix
    S = torch.einsum("bhnd,bhmd->bhnm", torch.tensor(Q), torch.tensor(K)) * scale
    if causal:
        mask = torch.ones(N, M, dtype=torch.bool).tril()
        S = S.masked_fill(~mask, -math.inf)
    assert np.max(np.abs(lse - torch.logsumexp(S, -1).numpy())) < 1e-12


def test_attention_row_sample_equals_full():
    rng = np.random.default_rng(3)
    Q, K, V = (rng.normal(size=(2, 2, 40, 16)) for _ in range(3))
    O, lse = oracle.attn_fwd(Q, K, V, 0.25, True)
    rows = np.array([0, 5, 39, 40, 77, 159])
    Os, lses = oracle.attn_fwd(Q, K, V, 0.25, True, rows=rows)
    assert np.array_equal(Os, O.reshape(-1, 16)[rows])
    assert np.array_equal(lses, lse.reshape(-1)[rows])


# ---------------------------------------------------------------- closed forms
def test_uniform_scores_give_mean_of_values():
    rng = np.random.default_rng(11)
    N, d = 23, 8
    Q = rng.normal(size=(1, 1, N, d))
    K = np.zeros((1, 1, N, d))
    V = rng.normal(size=(1, 1, N, d))
    O, lse = oracle.attn_fwd(Q, K, V, 0.5, False)
    assert np.max(np.abs(O[0, 0] - V[0, 0].mean(0))) < 1e-14
    assert np.max(np.abs(lse - math.log(N))) < 1e-14
    Oc, lsec = oracle.attn_fwd(Q, K, V, 0.5, True)
    for i in range(N):
        assert np.max(np.abs(Oc[0, 0, i] - V[0, 0, :i + 1].mean(0))) < 1e-14
        assert abs(lsec[0, 0, i] - math.log(i + 1)) < 1e-14


def test_causal_first_row_is_first_value():
    rng = np.random.default_rng(5)
    Q, K, V = (rng.normal(size=(1, 2, 12, 8)) for _ in range(3))
    O, lse = oracle.attn_fwd(Q, K, V, 0.3, True)
    for h in range(2):
        assert np.array_equal(O[0, h, 0], V[0, h, 0])
        assert abs(lse[0, h, 0] - 0.3 * float(Q[0, h, 0] @ K[0, h, 0])) < 1e-15


def test_dominant_key_selects_its_value():
    d = 4
    Q = np.ones((1, 1, 1, d))
    K = np.zeros((1, 1, 5, d))
    K[0, 0, 3] = 100.0
    V = np.arange(20, dtype=np.float64).reshape(1, 1, 5, d)
    O, _ = oracle.attn_fwd(Q, K, V, 1.0, False)
    # the other keys weigh e^-400 each
    assert np.max(np.abs(O[0, 0, 0] - V[0, 0, 3])) < 1e-150


# ---------------------------------------------------------------- the online recurrences
@pytest.mark.parametrize("n", [1, 2, 10, 1000])
def test_online_normaliser_equals_three_pass(n):
    x = np.random.default_rng(n).normal(0, 4, size=n)
    m, s = online.online_normaliser(x)
    assert m == x.max()
    _, lse = oracle.softmax_rows(x[None])
    assert abs((m + math.log(s)) - lse[0]) < 1e-12 * max(1, abs(lse[0]))


@pytest.mark.parametrize("M", [1, 2, 5, 64, 300])
def test_one_pass_and_blockwise_equal_oracle(M):
    rng = np.random.default_rng(M + 100)
    d = 6
    q = rng.normal(size=d)
    K = rng.normal(size=(M, d)) * 2
    V = rng.normal(size=(M, d))
    O, lse = oracle.attn_fwd(q[None, None, None], K[None, None], V[None, None], 1.0, False)
    x = K @ q
    a, g, s = online.one_pass_attention_row(x, V)
    assert np.max(np.abs(a - O[0, 0, 0])) < 1e-12
    assert abs(g + math.log(s) - lse[0, 0, 0]) < 1e-12
    for trial in range(3):
        cuts = np.sort(rng.choice(np.arange(1, M), size=min(M - 1, 1 + trial * 3), replace=False)) if M > 1 else []
        widths = np.diff(np.concatenate([[0], cuts, [M]])).astype(int).tolist()
        o, m, l = online.blockwise_attention_row(x, V, widths)
        assert np.max(np.abs(o - O[0, 0, 0])) < 1e-12
        assert abs(m + math.log(l) - lse[0, 0, 0]) < 1e-12


def test_oracle_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.softmax_rows(np.zeros((3, 0)))
    with pytest.raises(ValueError):
        oracle.attn_fwd(np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 3, 4)), np.zeros((1, 1, 2, 4)), 1.0)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 3, 4)), np.zeros((1, 1, 3, 4)), 1.0,
                        rows=[0, 2])


# ---------------------------------------------------------------- log-softmax and cross-entropy
def test_cross_entropy_printed_value_and_ignored_rows():
    ex = GOLD["ex2_cross_entropy"]
    X = np.array([ex["logits"], ex["logits"], ex["logits"]])
    loss, _ = oracle.cross_entropy_rows(X, [ex["label"], -100, 3])
    assert abs(loss[0] - ex["loss"]) < TOL
    assert loss[1] == 0.0 and loss[2] == 0.0


def test_cross_entropy_matches_torch_fp64():
    g = torch.Generator().manual_seed(5)
    X = torch.randn(37, 1000, generator=g, dtype=torch.float64) * 3
    lab = torch.randint(0, 1000, (37,), generator=g)
    loss, lse = oracle.cross_entropy_rows(X, lab)
    ref = torch.nn.functional.cross_entropy(X, lab, reduction="none").numpy()
    assert np.max(np.abs(loss - ref)) < 1e-12


def test_log_softmax_matches_torch_and_page():
    g = torch.Generator().manual_seed(6)
    X = torch.randn(9, 777, generator=g, dtype=torch.float64) * 4
    lp, lse = oracle.log_softmax_rows(X)
    assert np.max(np.abs(lp - torch.log_softmax(X, -1).numpy())) < 1e-12
    assert np.max(np.abs(np.exp(lp).sum(1) - 1)) < 1e-12
    ex = GOLD["ex1_softmax"]
    lp1, _ = oracle.log_softmax_rows(np.array([ex["logits"]]))
    assert np.max(np.abs(np.exp(lp1[0]) - ex["p"])) < TOL


# ---------------------------------------------------------------- bottom-right causal
@pytest.mark.parametrize("N,M", [(9, 31), (31, 9), (17, 17), (1, 40), (40, 1)])
def test_bottom_right_causal_matches_torch_masked_fp64(N, M):
    rng = np.random.default_rng(N * 100 + M)
    Q, K, V = rng.normal(size=(2, 2, N, 16)), rng.normal(size=(2, 2, M, 16)), rng.normal(size=(2, 2, M, 16))
    O, lse = oracle.attn_fwd(Q, K, V, 0.25, 2)
    keep = torch.ones(N, M, dtype=torch.bool).tril(diagonal=M - N)   # key j kept iff j <= i + (M - N)
    has = keep.any(1).numpy()
    S = torch.einsum("bhnd,bhmd->bhnm", torch.tensor(Q), torch.tensor(K)) * 0.25
    S = S.masked_fill(~keep, -math.inf)
    if has.any():
        P = torch.softmax(S[:, :, has], -1)
        ref = torch.einsum("bhnm,bhmd->bhnd", P, torch.tensor(V)).numpy()
        assert np.max(np.abs(O[:, :, has] - ref)) < 1e-12
        assert np.max(np.abs(lse[:, :, has] - torch.logsumexp(S[:, :, has], -1).numpy())) < 1e-12
    # rows with no kept key: O = 0, LSE = -inf
    assert np.all(O[:, :, ~has] == 0) and np.all(np.isneginf(lse[:, :, ~has]))


def test_bottom_right_equals_top_left_when_square_and_last_row_sees_all():
    rng = np.random.default_rng(2)
    Q, K, V = (rng.normal(size=(1, 1, 12, 8)) for _ in range(3))
    assert np.array_equal(oracle.attn_fwd(Q, K, V, 0.3, 2)[0], oracle.attn_fwd(Q, K, V, 0.3, 1)[0])
    K2, V2 = rng.normal(size=(1, 1, 30, 8)), rng.normal(size=(1, 1, 30, 8))
    O_br, _ = oracle.attn_fwd(Q, K2, V2, 0.3, 2)
    O_all, _ = oracle.attn_fwd(Q, K2, V2, 0.3, 0)
    assert np.max(np.abs(O_br[0, 0, -1] - O_all[0, 0, -1])) < 1e-15
