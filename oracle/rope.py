"""Pos-vector rotary position embedding (oracle).

From antirez/ds4 PR #530, the pos-vector RoPE commit: in a batched step every
token row carries its own position (a small position array indexed by token
row) instead of ``pos0 + t``.  The pages do not print the rotation itself;
the reading taken is the common rotate-half form with base ``theta``:

    for pair i < D/2 of each head:  a_i = pos[t] * theta ** (-2 i / D)
        (x_i, x_{i+D/2}) <- (x_i cos a_i - x_{i+D/2} sin a_i,
                             x_i sin a_i + x_{i+D/2} cos a_i)

applied to every head of q and of k.  Everything here is float64.
"""
from __future__ import annotations

import numpy as np


def angles(pos: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """float64 ``a[n_tok, D/2]``."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.power(np.float64(theta), -2.0 * i / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope_posvec(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate ``x[n_tok, H, D]`` by each token's own position; float64 result."""
    x = np.asarray(x, dtype=np.float64)
    n_tok, _, d = x.shape
    if len(pos) != n_tok:
        raise ValueError("one position per token row")
    a = angles(pos, d, theta)[:, None, :]
    c, s = np.cos(a), np.sin(a)
    half = d // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def head_rmsnorm_rope(x: np.ndarray, pos: np.ndarray, theta: float, w, eps: float) -> np.ndarray:
    """Per-head RMS norm, then the pos-vector RoPE (the ds4 page's fused head
    norm + RoPE tail and its position-vector twin, read as: every head vector
    of ``x[n_tok, H, D]`` is scaled by ``1 / sqrt(mean(x^2) + eps)`` and by the
    per-dimension weight ``w[D]``, then rotated as ``rope_posvec``).  ``w``
    None: no norm.  float64 result."""
    x = np.asarray(x, dtype=np.float64)
    if w is not None:
        ms = np.mean(x * x, axis=-1, keepdims=True)
        x = x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)
    return rope_posvec(x, pos, theta)
