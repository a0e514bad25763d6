"""Narrow-batch q8_0 matmul (oracle).

From antirez/ds4 PR #530 ("Why it's worth it -- the narrow-batch matmul" and
the narrow-batch q8_0 matmul commit): every output row is the dot product of a
q8_0 weight row with each of the ``n_tok`` pre-quantised q8_0 activation rows,
block by block.  Written out:

    isum[t, r, i] = sum_{k<32} qW[r, i, k] * qX[t, i, k]          (exact integer)
    y[t, r]       = sum_{i<nb} float(dW[r, i]) * float(dX[t, i]) * isum[t, r, i]

``isum`` is exact (|isum| <= 32 * 127 * 127 = 516128 fits int32); ``y`` is
accumulated here in float64.  The output is token-major ``y[n_tok, R]``.
"""
from __future__ import annotations

import numpy as np

from . import q8_0

ISUM_BOUND = 32 * 127 * 127


ROW_CHUNK = 4096  # output rows evaluated per pass (memory bound only; rows are independent)


def block_dots(w_blocks: np.ndarray, x_blocks: np.ndarray, rows=None) -> np.ndarray:
    """int64 ``isum[n_tok, R', nb]`` for weight rows ``rows`` (default all)."""
    qw, _ = q8_0.unpack(w_blocks)
    qx, _ = q8_0.unpack(x_blocks)
    if rows is not None:
        qw = qw[np.asarray(rows)]
    if qw.shape[1] != qx.shape[1]:
        raise ValueError("weight and activation rows have different block counts")
    qx64 = qx.astype(np.int64)
    out = np.empty((qx.shape[0], qw.shape[0], qw.shape[1]), dtype=np.int64)
    for r0 in range(0, qw.shape[0], ROW_CHUNK):
        out[:, r0:r0 + ROW_CHUNK] = np.einsum("rik,tik->tri", qw[r0:r0 + ROW_CHUNK].astype(np.int64), qx64)
    assert np.all(np.abs(out) <= ISUM_BOUND)
    return out


def matmul_q8_0(w_blocks: np.ndarray, x_blocks: np.ndarray, rows=None) -> np.ndarray:
    """float64 ``y[n_tok, R']`` = q8_0 weight rows ``rows`` (default all) times
    each q8_0 activation row."""
    _, dw = q8_0.unpack(w_blocks)
    _, dx = q8_0.unpack(x_blocks)
    if rows is not None:
        rows = np.asarray(rows)
        dw = dw[rows]
        w_blocks = np.asarray(w_blocks)[rows]
    y = np.empty((dx.shape[0], dw.shape[0]), dtype=np.float64)
    dx64 = dx.astype(np.float64)
    for r0 in range(0, dw.shape[0], ROW_CHUNK):
        isum = block_dots(w_blocks[r0:r0 + ROW_CHUNK], x_blocks).astype(np.float64)
        scale = dx64[:, None, :] * dw[r0:r0 + ROW_CHUNK].astype(np.float64)[None, :, :]
        y[:, r0:r0 + ROW_CHUNK] = np.sum(scale * isum, axis=2)
    return y
