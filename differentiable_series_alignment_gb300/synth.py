"""Seeded synthetic inputs for batched Soft-DTW.

This module holds no Soft-DTW arithmetic. It only draws numbers: both the CUDA
path (through its tests and the benchmark) and the fp64 oracle read exactly the
arrays produced here. Every array is drawn in float64 with numpy's PCG64 and
cast to float32, so both sides see bit-identical inputs.

Workload shapes follow the pages:
  * the headline shape B=32, N=M=512, D=64 of the README's "Key Benchmark"
    table (SoftDTW-CUDA (PyTorch + Numba) README);
  * the Figure 1 sweep of the SoftDTW-CUDA-Torch paper (B=32; L at D=128 and
    D at L=256);
  * a long time-warped pair for the long-sequence / small-gamma regime the
    abstract motivates (contributions (1) and (2));
  * block-wave sequences for the barycenter of Figure 2.
No public dataset is named on the pages; these recipes stand in for data.

Seed convention: seed = seed_base * 1000 + repeat.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng_for",
    "iid_normal_pair",
    "warped_pair",
    "block_waves",
    "WORKLOADS",
]


def rng_for(seed_base: int, repeat: int = 0) -> np.random.Generator:
    """PCG64 generator seeded by ``seed_base * 1000 + repeat``."""
    return np.random.Generator(np.random.PCG64(seed_base * 1000 + repeat))


def iid_normal_pair(B: int, N: int, M: int, D: int, seed_base: int, repeat: int = 0):
    """x (B,N,D) and y (B,M,D), entries iid N(0,1), as float32."""
    g = rng_for(seed_base, repeat)
    x = g.standard_normal((B, N, D)).astype(np.float32)
    y = g.standard_normal((B, M, D)).astype(np.float32)
    return x, y


def _random_monotone_warp(g: np.random.Generator, L: int, segments: int = 8) -> np.ndarray:
    """Piecewise-linear monotone map phi:[0,L-1]->[0,L-1] sampled at 0..L-1.

    Knots sit at evenly spaced t; the rise of each of the `segments` pieces is a
    Dirichlet(1,...,1) share of L-1, so phi(0)=0, phi(L-1)=L-1 and phi is
    non-decreasing.
    """
    if L == 1:
        return np.zeros(1)
    knots_t = np.linspace(0.0, L - 1.0, segments + 1)
    rises = g.dirichlet(np.ones(segments)) * (L - 1.0)
    knots_v = np.concatenate([[0.0], np.cumsum(rises)])
    knots_v[-1] = L - 1.0
    return np.interp(np.arange(L, dtype=np.float64), knots_t, knots_v)


def warped_pair(B: int, L: int, D: int, seed_base: int, repeat: int = 0,
                noise: float = 0.1, segments: int = 8):
    """x ~ N(0,1) of shape (B,L,D); y[b,j] = x[b] linearly interpolated at
    phi_b(j) plus N(0, noise^2), with phi_b a random monotone piecewise-linear
    warp (one per batch element)."""
    g = rng_for(seed_base, repeat)
    x = g.standard_normal((B, L, D))
    y = np.empty_like(x)
    for b in range(B):
        phi = _random_monotone_warp(g, L, segments)
        lo = np.floor(phi).astype(np.int64)
        hi = np.minimum(lo + 1, L - 1)
        w = (phi - lo)[:, None]
        y[b] = (1.0 - w) * x[b, lo] + w * x[b, hi]
    y += noise * g.standard_normal(y.shape)
    return x.astype(np.float32), y.astype(np.float32)


def block_waves(K: int, T: int, D: int, seed_base: int, repeat: int = 0,
                pmin: float = 64.0, pmax: float = 256.0, noise: float = 0.1):
    """K sequences (K,T,D): each channel is a +-1 square wave
    s(t) = +1 if floor(2 (t + phase) / P) is even else -1, with period
    P ~ U[pmin, pmax] and phase ~ U[0, P) drawn per sequence and channel,
    plus N(0, noise^2)."""
    g = rng_for(seed_base, repeat)
    P = g.uniform(pmin, pmax, size=(K, 1, D))
    phase = g.uniform(0.0, 1.0, size=(K, 1, D)) * P
    t = np.arange(T, dtype=np.float64)[None, :, None]
    s = np.where(np.floor(2.0 * (t + phase) / P) % 2 == 0, 1.0, -1.0)
    s = s + noise * g.standard_normal((K, T, D))
    return s.astype(np.float32)


# The five workloads by name, each with the seed base its inputs are drawn with.
# Sizes only; gamma and mode per entry.
WORKLOADS = {
    "small": dict(seed=0, B=4, N=64, M=64, D=4, gammas=(1.0,), modes=("unfused",)),
    "headline": dict(seed=1, B=32, N=512, M=512, D=64, gammas=(1.0,), modes=("unfused", "fused")),
    "sweep": dict(seed=2, B=32, L_sweep=(128, 256, 512, 1024, 2048), D_at_L=128,
                  D_sweep=(1, 4, 16, 64, 128, 256), L_at_D=256, gammas=(1.0,), modes=("unfused", "fused")),
    "long_warped": dict(seed=3, B=8, N=8192, M=8192, D=128, gammas=(1.0, 0.1, 0.01), modes=("fused",)),
    "barycenter": dict(seed=4, K=64, T=1024, D=8, steps=100, lr=0.1, gammas=(1.0,), modes=("fused",)),
}
