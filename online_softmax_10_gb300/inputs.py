"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no softmax, no dot products), so it can serve both the
CUDA library and the CPU oracle without the two sharing code.

Recipe (the same for every caller):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * attention: draw Q, then K, then V as fp32 ``[B, H, N|M, d]``; for the
    long-context workload then draw one U[0.5, 2) factor per key row and
    multiply K by it in fp32; finally round to the workload dtype
    (round-to-nearest-even for bf16);
  * row softmax: draw X ~ N(0, sigma^2) as fp32 ``[rows, cols]``, then draw one
    column per row uniformly and set it to the spike value, then round to the
    dtype.
The same bits are copied to the device and widened exactly to fp64 for the
oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    B: int
    H: int
    N: int
    M: int
    d: int
    dtype: torch.dtype
    causal: bool
    seed: int
    dist: str = "normal"          # "normal": N(0,1); "uniform": U[0,1)
    k_row_scale: tuple | None = None  # (lo, hi): per key row U[lo, hi) factor

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def flops(self) -> float:
        """4*B*H*N*M*d, halved under the causal mask (the stated convention)."""
        f = 4.0 * self.B * self.H * self.N * self.M * self.d
        return f / 2 if self.causal else f


@dataclass(frozen=True)
class RowsWorkload:
    name: str
    rows: int
    cols: int
    dtype: torch.dtype
    seed: int
    sigma: float = 3.0
    spike: float | None = 20.0


# The five workloads the library is specified on.
ATTN_F32_64 = AttnWorkload("attn_f32_N64_d64", 1, 1, 64, 64, 64, torch.float32, False, 0, dist="uniform")
ROWS_4096x32768 = RowsWorkload("softmax_rows_bf16_4096x32768", 4096, 32768, torch.bfloat16, 1)
ATTN_B4H16_2048_D64 = AttnWorkload("attn_bf16_B4_H16_N2048_d64", 4, 16, 2048, 2048, 64, torch.bfloat16, False, 2)
ATTN_B2H32_8192_D128_CAUSAL = AttnWorkload("attn_bf16_B2_H32_N8192_d128_causal", 2, 32, 8192, 8192, 128,
                                           torch.bfloat16, True, 3)
ATTN_B1H16_32768_D128_CAUSAL = AttnWorkload("attn_bf16_B1_H16_N32768_d128_causal_kscaled", 1, 16, 32768, 32768,
                                            128, torch.bfloat16, True, 4, k_row_scale=(0.5, 2.0))

WORKLOADS = {w.name: w for w in (ATTN_F32_64, ROWS_4096x32768, ATTN_B4H16_2048_D64,
                                 ATTN_B2H32_8192_D128_CAUSAL, ATTN_B1H16_32768_D128_CAUSAL)}


def attn_inputs(B: int, H: int, N: int, M: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                dist: str = "normal", k_row_scale=None):
    """Q [B,H,N,d], K [B,H,M,d], V [B,H,M,d] on the CPU, rounded to ``dtype``."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    if dist == "normal":
        draw = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    elif dist == "uniform":
        draw = lambda *s: torch.rand(*s, generator=g, dtype=torch.float32)
    else:
        raise ValueError(dist)
    q = draw(B, H, N, d)
    k = draw(B, H, M, d)
    v = draw(B, H, M, d)
    if k_row_scale is not None:
        lo, hi = k_row_scale
        f = torch.rand(B, H, M, 1, generator=g, dtype=torch.float32) * (hi - lo) + lo
        k = k * f
    return q.to(dtype), k.to(dtype), v.to(dtype)


def workload_attn_inputs(w: AttnWorkload):
    return attn_inputs(w.B, w.H, w.N, w.M, w.d, w.dtype, w.seed, w.dist, w.k_row_scale)


def rows_inputs(rows: int, cols: int, dtype=torch.bfloat16, seed: int = 1, sigma: float = 3.0,
                spike: float | None = 20.0):
    """X [rows, cols] on the CPU: N(0, sigma^2) with one column per row set to
    ``spike`` (skipped when spike is None), rounded to ``dtype``."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32) * sigma
    if spike is not None and rows > 0:
        col = torch.randint(0, cols, (rows,), generator=g)
        x[torch.arange(rows), col] = spike
    return x.to(dtype)


def workload_rows_inputs(w: RowsWorkload):
    return rows_inputs(w.rows, w.cols, w.dtype, w.seed, w.sigma, w.spike)


def device_normal(shape, seed: int, sigma: float = 1.0, dtype=torch.bfloat16, device="cuda"):
    """Seeded N(0, sigma^2) values drawn on the device and cast to ``dtype``
    (round to nearest), for inputs too large to draw on the host.  Drawn in
    slices of 2^28 values so the fp32 temporary stays at 1 GiB."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        flat[s:e] = (torch.randn(e - s, generator=g, device=device) * sigma).to(dtype)
    return out


def sample_rows(total: int, count: int, seed: int = 12345):
    """A seeded, sorted sample of ``count`` distinct indices in [0, total),
    always including the first and the last index (edge rows)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    count = max(0, min(count, total))
    if count >= total:
        return torch.arange(total, dtype=torch.int64)
    idx = torch.randperm(total, generator=g)[:count]
    idx = torch.unique(torch.cat([idx, torch.tensor([0, total - 1])]))
    return idx.to(torch.int64)
