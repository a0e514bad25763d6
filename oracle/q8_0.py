"""q8_0 block codec (oracle).

Format.  A q8_0 block covers 32 consecutive values of a row and takes 34
bytes: the fp16 scale ``d`` (little-endian) first, then the 32 int8 codes.
Value k of the block is ``float(d) * q[k]``.  A row of ``cols`` values
(``cols % 32 == 0``) is ``cols / 32`` blocks laid end to end; a matrix is its
rows laid end to end.  The ds4 page ("Why it's worth it -- the narrow-batch
matmul") names the 32-weight block and the pre-quantised ("preq") q8_0
activations; the block layout itself is the page's silent point, read here as
scale-then-codes.

Quantisation of one block (the workload definition: scale = max|x| / 127,
code = round(x / scale)), every operation an IEEE float32 operation:

    a = max_k |x_k|                      (exact)
    d = a / 127                           (float32 division, round to nearest)
    q_k = clamp(round(x_k / d), -127, 127)   (float32 division; round half
                                              away from zero), q = 0 if d == 0
    stored scale = fp16(d)                (round to nearest even)

The codes use the float32 ``d`` before its fp16 rounding.
"""
from __future__ import annotations

import numpy as np

QK = 32
BLOCK_BYTES = 34


def quantize_rows(x: np.ndarray) -> np.ndarray:
    """Quantise float32 rows ``x[..., cols]`` to q8_0 bytes ``[..., cols/32*34]``."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    cols = x.shape[-1]
    if cols % QK:
        raise ValueError("row length must be a multiple of 32")
    nb = cols // QK
    lead = x.shape[:-1]
    blk = x.reshape(-1, nb, QK)
    amax = np.max(np.abs(blk), axis=-1)                      # float32, exact
    d = (amax / np.float32(127.0)).astype(np.float32)        # one float32 division
    safe = np.where(d == 0, np.float32(1.0), d).astype(np.float32)
    v = (blk / safe[..., None]).astype(np.float32)           # float32 division per value
    v64 = v.astype(np.float64)
    r = np.sign(v64) * np.floor(np.abs(v64) + 0.5)           # half away from zero, exact in f64
    r = np.where(d[..., None] == 0, 0.0, r)
    q = np.clip(r, -127, 127).astype(np.int8)
    out = np.empty((blk.shape[0], nb, BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = d.astype(np.float16).astype("<f2").view(np.uint8).reshape(blk.shape[0], nb, 2)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(lead + (nb * BLOCK_BYTES,))


def unpack(blocks: np.ndarray):
    """Split q8_0 bytes ``[..., nb*34]`` into (codes int8 ``[..., nb, 32]``,
    scales float16 ``[..., nb]``)."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    if b.shape[-1] % BLOCK_BYTES:
        raise ValueError("byte length must be a multiple of 34")
    nb = b.shape[-1] // BLOCK_BYTES
    lead = b.shape[:-1]
    b3 = b.reshape(lead + (nb, BLOCK_BYTES))
    d = np.ascontiguousarray(b3[..., 0:2]).view("<f2").reshape(lead + (nb,))
    q = np.ascontiguousarray(b3[..., 2:]).view(np.int8)
    return q, d


def dequantize_rows(blocks: np.ndarray) -> np.ndarray:
    """float64 values ``[..., cols]`` represented by q8_0 bytes."""
    q, d = unpack(blocks)
    v = q.astype(np.float64) * d.astype(np.float64)[..., None]
    return v.reshape(v.shape[:-2] + (v.shape[-2] * QK,))
