"""The small per-token stages of a decode step (oracle).

The ds4 page ("What") lists the memory-bound dense stages a batched step runs
once for all sessions -- attention projections, output head, RoPE/norm --
around the matmuls.  The llama-style stages used here, written out in float64:

    rmsnorm(x)  = x / sqrt(mean(x^2) + eps) * w
    silu_mul    = g / (1 + exp(-g)) * u
    residual    = a + b
    embedding   = the q8_0 row of the token id, dequantised
"""
from __future__ import annotations

import numpy as np

from . import q8_0


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g)) * np.asarray(u, dtype=np.float64)


def residual_add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64) + np.asarray(b, dtype=np.float64)


def embedding(table_blocks: np.ndarray, token_ids) -> np.ndarray:
    """Dequantised rows ``[n_tok, hidden]`` of a q8_0 embedding table."""
    return q8_0.dequantize_rows(np.asarray(table_blocks)[np.asarray(token_ids)])
