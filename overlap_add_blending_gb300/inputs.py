"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws numbers: it holds none of the tiling, window or
selection arithmetic, so that the CUDA path and the CPU oracle can both be
fed from it without sharing any of the method.

Shapes follow the LTX-2 workloads named in the TDP / SP docs (stage 1 at
512x768x121 and the full-resolution call at 1024x1536x121, both patchified
to 32 px per latent unit and 8 frames per latent frame) and a 4K-class
3840x2176 latent.  Position intervals are in pixel units: latent frame f
spans [8f, 8f+8), row h spans [32h, 32h+32), column w spans [32w, 32w+32).
"""
from __future__ import annotations

import numpy as np

POS_SCALE = (8, 32, 32)   # pixels (or frames) per latent unit on (t, h, w)


def latent(shape, seed: int = 0) -> np.ndarray:
    """N(0, 1) float32 latent of shape (B, C, F, H, W)."""
    return np.random.default_rng(seed).standard_normal(size=tuple(shape), dtype=np.float32)


def affine_params(num_tiles: int, seed: int = 1):
    """Per-tile affine op y = a_t * x + b_t with a_t ~ U[0.5, 1.5], b_t ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.5, 1.5, size=num_tiles).astype(np.float32)
    b = rng.standard_normal(size=num_tiles).astype(np.float32)
    return a, b


def grid_positions(B: int, F: int, H: int, W: int, scale=POS_SCALE) -> np.ndarray:
    """Uniform position grid, int32 [B, 3, F*H*W, 2]; token n = (f*H + h)*W + w."""
    f, h, w = np.meshgrid(np.arange(F), np.arange(H), np.arange(W), indexing="ij")
    coords = (f.reshape(-1), h.reshape(-1), w.reshape(-1))
    pos = np.empty((B, 3, F * H * W, 2), dtype=np.int32)
    for d in range(3):
        pos[:, d, :, 0] = coords[d] * scale[d]
        pos[:, d, :, 1] = (coords[d] + 1) * scale[d]
    return pos


def random_positions(B: int, N: int, seed: int, lo: int = -1000, hi: int = 1000) -> np.ndarray:
    """Arbitrary (non-grid) intervals, int32 [B, 3, N, 2], start < end."""
    rng = np.random.default_rng(seed)
    start = rng.integers(lo, hi, size=(B, 3, N), dtype=np.int64)
    width = rng.integers(1, 64, size=(B, 3, N), dtype=np.int64)
    return np.stack([start, start + width], axis=-1).astype(np.int32)


def cond_positions(B: int, M: int, F: int, H: int, W: int, n_negative: int, seed: int = 2,
                   scale=POS_SCALE) -> np.ndarray:
    """Conditioning-token intervals, int32 [B, 3, M, 2].

    Spatial starts are uniform over the frame plus a 64 px margin on each
    side, widths 32 px times U{1, 2, 3}; `n_negative` tokens (placed at
    random indices) have a time start in [-16, -1], the rest in [0, 8F);
    time widths are 8.
    """
    rng = np.random.default_rng(seed)
    pos = np.empty((B, 3, M, 2), dtype=np.int64)
    for b in range(B):
        neg = np.zeros(M, dtype=bool)
        neg[rng.permutation(M)[:n_negative]] = True
        t0 = np.where(neg, rng.integers(-16, 0, size=M), rng.integers(0, F * scale[0], size=M))
        pos[b, 0, :, 0] = t0
        pos[b, 0, :, 1] = t0 + scale[0]
        for d, D in ((1, H), (2, W)):
            s0 = rng.integers(-64, D * scale[d] + 64, size=M)
            pos[b, d, :, 0] = s0
            pos[b, d, :, 1] = s0 + scale[d] * rng.integers(1, 4, size=M)
    return pos.astype(np.int32)
