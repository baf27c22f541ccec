"""Seeded synthetic inputs for the CSA2 layer.

Shared by the tests, the smoke check and the benchmark, so that the CUDA path and
the CPU oracle receive the same bytes.  This module holds none of the method's
arithmetic: it only draws seeded random numbers and rounds them to the input
dtypes (bf16 latents, keys and queries; fp32 head weights).

Recipe (matches the workloads described for one CSA2 layer of DeepSeek-V4.1-Flash):
* latents (512 ch), indexer keys (128 ch), indexer queries (64 x 128), attention
  queries (64 x 512) and window rows (512 ch): N(0, 1), rounded to bf16;
* head weights w: N(0, 1) fp32;
* optional outliers: round(frac x n) distinct rows multiplied by a factor before the
  bf16 rounding (1 % of entries x 8 stresses the E4M3 block scales);
* Reuse-mode indices: distinct indices drawn uniformly from the visible prefix.
"""
from __future__ import annotations

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(int(seed))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values as bf16 bit patterns (uint16)."""
    return bf16_bits(rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(scale))


def normal_f32(seed: int, shape) -> np.ndarray:
    return rng(seed).standard_normal(shape, dtype=np.float32)


def outlier_rows(seed: int, n: int, frac: float = 0.01) -> np.ndarray:
    """round(frac * n) distinct row indices, ascending."""
    m = int(round(frac * n))
    return np.sort(rng(seed).permutation(n)[:m]).astype(np.int64)


def normal_bf16_rows_with_outliers(seed: int, n: int, width: int, frac: float, factor: float):
    """[n][width] N(0,1) rows; round(frac*n) rows multiplied by `factor` before bf16 rounding."""
    x = rng(seed).standard_normal((n, width), dtype=np.float32)
    if frac > 0:
        x[outlier_rows(seed + 7919, n, frac)] *= np.float32(factor)
    return bf16_bits(x)


def distinct_indices(seed: int, n_visible: int, k: int) -> np.ndarray:
    """min(k, n_visible) distinct indices drawn uniformly from [0, n_visible), -1 padded to k."""
    g = rng(seed)
    m = min(k, n_visible)
    if n_visible <= 4 * k:
        pick = g.permutation(n_visible)[:m]
    else:
        pick = np.unique(g.integers(0, n_visible, size=2 * m))
        while pick.size < m:
            pick = np.unique(np.concatenate([pick, g.integers(0, n_visible, size=m)]))
        pick = g.permutation(pick)[:m]
    out = np.full(k, -1, np.int32)
    out[:m] = pick
    return out


# --------------------------------------------------------------- device (torch) generators

def torch_normal_bf16(seed: int, shape, device, scale: float = 1.0):
    """N(0, scale^2) bf16 tensor drawn on `device` with a seeded torch.Generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def torch_normal_f32(seed: int, shape, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def torch_distinct_indices(seed: int, n_queries: int, n_visible: int, k: int, device):
    """[n_queries][k] distinct indices uniform over [0, n_visible) (requires n_visible >= k)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty((n_queries, k), dtype=torch.int32, device=device)
    for q in range(n_queries):
        # rejection-free: a random permutation prefix is O(n_visible); use sorted unique draws
        cand = torch.randint(0, n_visible, (2 * k,), generator=g, device=device)
        u = torch.unique(cand)
        while u.numel() < k:
            u = torch.unique(torch.cat([u, torch.randint(0, n_visible, (k,), generator=g, device=device)]))
        perm = torch.randperm(u.numel(), generator=g, device=device)[:k]
        out[q] = u[perm].to(torch.int32)
    return out


def torch_normal_bf16_rows_with_outliers(seed: int, n: int, width: int, frac: float, factor: float, device):
    """Device twin of the row recipe above: [n][width] N(0,1) rows drawn directly in bf16
    with a seeded torch.Generator (the generator rounds each draw to nearest),
    round(frac*n) distinct rows (a seeded permutation's prefix) multiplied by `factor`
    (a power of two: exact in bf16)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((n, width), generator=g, device=device, dtype=torch.bfloat16)
    m = int(round(frac * n))
    if m:
        g2 = torch.Generator(device=device)
        g2.manual_seed(int(seed) + 7919)
        rows = torch.randperm(n, generator=g2, device=device)[:m]
        x[rows] *= float(factor)
    return x
