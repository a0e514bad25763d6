"""Pos-vector rotary position embedding (oracle).

From antirez/ds4 PR #530, the pos-vector RoPE commit: in a batched step every
token row carries its own position (a small position array indexed by token
row) instead of ``pos0 + t``.  The pages do not print the rotation itself;
the reading taken is the common rotate-half form with base ``theta``:

    for pair i < D/2 of each head:  a_i = pos[t] * theta ** (-2 i / D)
        (x_i, x_{i+D/2}) <- (x_i cos a_i - x_{i+D/2} sin a_i,
                             x_i sin a_i + x_{i+D/2} cos a_i)

applied to every head of q and of k.  Everything here is float64.

The same page tests a "plain and YaRN" path of that RoPE without printing the
YaRN rule.  The reading taken is YaRN as published (Peng, Quesnelle, Fan,
Shippole 2023, "YaRN: Efficient Context Window Extension of Large Language
Models", sections 3.2 "NTK-by-parts" and 3.3 "YaRN"), in the form that ramps
over the pair index:

    scale s = extended / original context L;  per pair i the rotation count
    over L is r_i = L / (2 pi / f_i) with the plain frequency f_i;
    corr(b) = pair index where r = b:  D ln(L / (2 pi b)) / (2 ln theta);
    low = max(floor(corr(beta_fast)), 0), high = min(ceil(corr(beta_slow)), D - 1)
    ramp_i = clamp((i - low) / max(high - low, 0.001), 0, 1)
    f'_i = f_i (1 - ramp_i) + (f_i / s) ramp_i     (extrapolate fast pairs,
                                                    interpolate slow ones)
    every rotated value is multiplied by m = 0.1 ln s + 1 (the paper's
    sqrt(1/t), applied to q and k through the rotation)

with beta_fast = 32, beta_slow = 1 by default.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Yarn:
    """YaRN parameters: ``factor`` s > 1, ``orig_ctx`` L (the original context)."""
    factor: float
    orig_ctx: int
    beta_fast: float = 32.0
    beta_slow: float = 1.0


def yarn_correction_range(head_dim: int, theta: float, yarn: Yarn):
    """(low, high) pair indices bounding the ramp."""
    def corr(b):
        return head_dim * math.log(yarn.orig_ctx / (2.0 * math.pi * b)) / (2.0 * math.log(theta))
    low = max(math.floor(corr(yarn.beta_fast)), 0)
    high = min(math.ceil(corr(yarn.beta_slow)), head_dim - 1)
    return low, high


def yarn_mscale(yarn) -> float:
    return 1.0 if yarn is None else 0.1 * math.log(yarn.factor) + 1.0


def frequencies(head_dim: int, theta: float, yarn=None) -> np.ndarray:
    """float64 per-pair frequency ``f[D/2]`` (YaRN-blended when ``yarn``)."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    f = np.power(np.float64(theta), -2.0 * i / head_dim)
    if yarn is None:
        return f
    low, high = yarn_correction_range(head_dim, theta, yarn)
    ramp = np.clip((i - low) / max(high - low, 0.001), 0.0, 1.0)
    return f * (1.0 - ramp) + (f / yarn.factor) * ramp


def angles(pos: np.ndarray, head_dim: int, theta: float, yarn=None) -> np.ndarray:
    """float64 ``a[n_tok, D/2]``."""
    f = frequencies(head_dim, theta, yarn)
    return np.asarray(pos, dtype=np.float64)[:, None] * f[None, :]


def rope_posvec(x: np.ndarray, pos: np.ndarray, theta: float, yarn=None) -> np.ndarray:
    """Rotate ``x[n_tok, H, D]`` by each token's own position; float64 result.
    With ``yarn``: YaRN frequencies and the magnitude factor m."""
    x = np.asarray(x, dtype=np.float64)
    n_tok, _, d = x.shape
    if len(pos) != n_tok:
        raise ValueError("one position per token row")
    a = angles(pos, d, theta, yarn)[:, None, :]
    m = yarn_mscale(yarn)
    c, s = np.cos(a) * m, np.sin(a) * m
    half = d // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def head_rmsnorm_rope(x: np.ndarray, pos: np.ndarray, theta: float, w, eps: float, yarn=None) -> np.ndarray:
    """Per-head RMS norm, then the pos-vector RoPE (the ds4 page's fused head
    norm + RoPE tail and its position-vector twin, read as: every head vector
    of ``x[n_tok, H, D]`` is scaled by ``1 / sqrt(mean(x^2) + eps)`` and by the
    per-dimension weight ``w[D]``, then rotated as ``rope_posvec``).  ``w``
    None: no norm.  float64 result."""
    x = np.asarray(x, dtype=np.float64)
    if w is not None:
        ms = np.mean(x * x, axis=-1, keepdims=True)
        x = x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)
    return rope_posvec(x, pos, theta, yarn)
