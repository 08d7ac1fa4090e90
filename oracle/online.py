"""The pages' online recurrences, restated in fp64 for small inputs.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

These follow the recurrences in the order and notation the pages give them;
the tests pin them against the worked examples and against the three-pass
oracle, which is how the identity "the online result equals the plain
definition" (the reason the fused kernel is exact) is checked on the CPU.

* ``online_normaliser`` -- "什么是 online softmax and flash attention",
  section "Online softmax", eq (3)-(5); also "Softmax与Flash-Attention",
  section "online-softmax 推导":  m_1 = x_1, s_1 = 1,
  m_i = max(m_{i-1}, x_i),  s_i = s_{i-1} e^{m_{i-1} - m_i} + e^{x_i - m_i}.
* ``one_pass_attention_row`` -- same page, section "优化循环（2）", eq (22) and
  (26): the normalised accumulator
  A'_1 = e^{x_1-g_1}/s_1 V_1,
  A'_m = A'_{m-1} s_{m-1} e^{g_{m-1}-g_m} / s_m + e^{x_m-g_m}/s_m V_m.
* ``blockwise_attention_row`` -- "从原始Softmax到在线Softmax", section on the
  block-wise online softmax: with m^(0) = -inf, l^(0) = 0, o~^(0) = 0 and for
  each key block, m^(j+1) = max(m^(j), m^new),
  o~^(j+1) = e^{m^(j) - m^(j+1)} o~^(j) + sum_k e^{s_k - m^(j+1)} v_k,
  l^(j+1)  = e^{m^(j) - m^(j+1)} l^(j)  + sum_k e^{s_k - m^(j+1)},
  o = o~ / l.
"""
from __future__ import annotations

import math

import numpy as np


def online_normaliser(x):
    """Sequential (m_N, s_N) of a 1-D sequence."""
    x = [float(v) for v in np.asarray(x, dtype=np.float64).reshape(-1)]
    if not x:
        raise ValueError("empty sequence")
    m_prev, s_prev = x[0], 1.0
    for xi in x[1:]:
        m = max(m_prev, xi)
        s = s_prev * math.exp(m_prev - m) + math.exp(xi - m)
        m_prev, s_prev = m, s
    return m_prev, s_prev


def one_pass_attention_row(x, V):
    """A'_M for one query row: scores x[M], values V[M, d]."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    V = np.asarray(V, dtype=np.float64)
    g_prev = x[0]
    s_prev = 1.0
    a = V[0].copy()                      # e^{x_1 - g_1} / s_1 = 1
    for m in range(1, x.shape[0]):
        g = max(g_prev, x[m])
        s = s_prev * math.exp(g_prev - g) + math.exp(x[m] - g)
        a = a * (s_prev * math.exp(g_prev - g) / s) + (math.exp(x[m] - g) / s) * V[m]
        g_prev, s_prev = g, s
    return a, g_prev, s_prev


def blockwise_attention_row(x, V, block):
    """o = o~ / l for one query row, merging key blocks of width ``block``
    (an int, or a list of widths summing to len(x)).  Returns (o, m, l)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    V = np.asarray(V, dtype=np.float64)
    n = x.shape[0]
    if isinstance(block, int):
        widths = [block] * (n // block) + ([n % block] if n % block else [])
    else:
        widths = list(block)
    if sum(widths) != n or any(w <= 0 for w in widths):
        raise ValueError("block widths must be positive and cover the row")
    m = -math.inf
    l = 0.0
    o = np.zeros(V.shape[1], dtype=np.float64)
    start = 0
    for w in widths:
        s_blk = x[start:start + w]
        v_blk = V[start:start + w]
        m_new = max(m, float(s_blk.max()))
        corr = math.exp(m - m_new) if m != -math.inf else 0.0
        e = np.exp(s_blk - m_new)
        o = corr * o + e @ v_blk
        l = corr * l + float(e.sum())
        m = m_new
        start += w
    return o / l, m, l
