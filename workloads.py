"""Seeded synthetic inputs for the W12 skinny-GEMM workloads.

This module holds input generation only: random draws, the weight
distributions of the five workloads and round-to-nearest-even conversion of
float32 draws to BF16 bit patterns.  It contains none of the W12 format's
arithmetic, and it is the only code shared by the oracle tests and the CUDA
path tests.

Workloads (sizes as N x K for W, M activation rows):
  tiny       W[512][256] ~ N(0, 0.02^2) x per-row U(0.5, 2); 13 entries (0.01 %)
             forced to 0 and 4 entries to +-50; x[1][256] ~ N(0, 1).
  projection q/o 5120x5120, k/v 1024x5120, gate/up 17408x5120, down 5120x17408;
             W ~ N(0, 0.02^2) x per-row U(0.5, 2), and 1e-4 of the entries
             (uniform positions, no replacement) replaced by Student-t(nu=2) x 0.5.
  heavy      Student-t(nu=1.5) x 0.02, no row scale (the heavy-tailed variant of
             the two-level-verification pair).
  x          activations ~ N(0, 1), rounded to BF16.
"""
from __future__ import annotations

import numpy as np

# the projections of one dense decoder layer with hidden 5120, intermediate
# 17408 and 8 KV heads of dim 128: (name, N, K)
LAYER_PROJECTIONS = (
    ("q", 5120, 5120),
    ("k", 1024, 5120),
    ("v", 1024, 5120),
    ("o", 5120, 5120),
    ("gate", 17408, 5120),
    ("up", 17408, 5120),
    ("down", 5120, 17408),
)

PROJECTION_SHAPES = ((5120, 5120), (1024, 5120), (17408, 5120), (5120, 17408))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); returns uint16 bits.

    Inputs here are finite draws, so NaN handling is not needed; overflow
    correctly rounds to +-Inf.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_rows(N: int, K: int, seed: int, sigma: float = 0.02) -> np.ndarray:
    """W ~ N(0, sigma^2) x per-row U(0.5, 2), as BF16 bits [N][K]."""
    rng = _rng(seed)
    scale = rng.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(sigma) * scale
    return f32_to_bf16_bits(w)


def tiny_weights(seed: int = 1):
    """The 512 x 256 matrix with forced zeros and +-50 outliers, and x[1][256]."""
    N, K = 512, 256
    rng = _rng(seed)
    scale = rng.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02) * scale
    n_zero = int(round(N * K * 1e-4))  # 0.01 % of the entries -> 13
    pos = rng.choice(N * K, size=n_zero + 4, replace=False)
    flat = w.reshape(-1)
    flat[pos[:n_zero]] = 0.0
    signs = rng.choice(np.array([-1.0, 1.0], dtype=np.float32), size=4)
    flat[pos[n_zero:]] = 50.0 * signs
    x = rng.standard_normal((1, K), dtype=np.float32)
    return f32_to_bf16_bits(w), f32_to_bf16_bits(x), pos[:n_zero], pos[n_zero:]


def projection_weights(N: int, K: int, seed: int, outlier_frac: float = 1e-4) -> np.ndarray:
    """Normal x row-scale weights with Student-t(2) x 0.5 outliers, BF16 bits."""
    rng = _rng(seed)
    scale = rng.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02) * scale
    n_out = int(round(N * K * outlier_frac))
    if n_out:
        pos = rng.choice(N * K, size=n_out, replace=False)
        w.reshape(-1)[pos] = (rng.standard_t(2.0, size=n_out) * 0.5).astype(np.float32)
    return f32_to_bf16_bits(w)


def heavy_weights(N: int, K: int, seed: int) -> np.ndarray:
    """Student-t(nu = 1.5) x 0.02, no row scale, BF16 bits."""
    rng = _rng(seed)
    w = (rng.standard_t(1.5, size=(N, K)) * 0.02).astype(np.float32)
    return f32_to_bf16_bits(w)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """x[M][K] ~ N(0, 1) as BF16 bits."""
    rng = _rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def projection_weights_torch(N: int, K: int, seed: int, device: str = "cuda"):
    """Same distribution as ``projection_weights``, drawn with torch on `device`.

    Used for the large benchmark layers, where drawing ~0.3 G weights per layer
    on the host would dominate the run.  Returns an int16 tensor of BF16 bits.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    scale = torch.rand((N, 1), generator=g, device=device) * 1.5 + 0.5
    w = torch.randn((N, K), generator=g, device=device) * 0.02 * scale
    n_out = int(round(N * K * 1e-4))
    if n_out:
        pos = torch.randperm(N * K, generator=g, device=device)[:n_out]
        # Student-t(2) = Z / sqrt(chi2_2 / 2), chi2_2 = -2 log U
        z = torch.randn(n_out, generator=g, device=device)
        u = torch.rand(n_out, generator=g, device=device).clamp_min(1e-30)
        t2 = z / torch.sqrt(-torch.log(u))
        w.view(-1)[pos] = t2 * 0.5
    return w.to(torch.bfloat16).view(torch.int16)
