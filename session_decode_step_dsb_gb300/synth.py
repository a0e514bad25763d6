"""Seeded synthetic inputs shared by the CUDA path, its tests and the bench.

This module only draws random numbers and shapes them; it holds none of the
decode step's arithmetic (no quantisation, no RoPE, no attention).  Every
array is a pure function of ``(seed, stream, shape, ...)``, drawn with
numpy's PCG64 generator seeded through ``SeedSequence([seed, stream, ...])``,
so the x86 host and the Arm GPU host produce identical bytes.

Large matrices are drawn in fixed row chunks of :data:`ROW_CHUNK` rows, each
chunk from its own sub-stream, so that a caller can regenerate any row range
(for sampled checks at full size) without drawing the whole matrix.
"""
from __future__ import annotations

import numpy as np

ROW_CHUNK = 1024

# Sub-stream ids, one per logical tensor kind.  A tensor's stream is
# ``kind * 1_000_003 + index`` so that e.g. layer 3's QKV weight and layer 4's
# never share a stream.
STREAM_W = 11
STREAM_X = 13
STREAM_KCACHE = 17
STREAM_VCACHE = 19
STREAM_Q = 23
STREAM_K = 29
STREAM_V = 31
STREAM_META = 37
STREAM_TOKENS = 41
STREAM_EMBED = 43


def stream_id(kind: int, index: int = 0) -> int:
    return int(kind) * 1_000_003 + int(index)


def _rng(seed: int, *keys: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(k) for k in keys]))


def normal_rows(seed: int, stream: int, rows: int, cols: int, std: float = 1.0,
                row_lo: int = 0, row_hi: int | None = None) -> np.ndarray:
    """Rows ``[row_lo, row_hi)`` of a ``rows x cols`` float32 matrix of N(0, std^2).

    Rows are drawn in chunks of ROW_CHUNK; chunk ``c`` comes from sub-stream
    ``(seed, stream, c)``, so any row range is reproducible on its own.
    """
    if row_hi is None:
        row_hi = rows
    if not (0 <= row_lo <= row_hi <= rows):
        raise ValueError("row range out of bounds")
    out = np.empty((row_hi - row_lo, cols), dtype=np.float32)
    c0, c1 = row_lo // ROW_CHUNK, (row_hi - 1) // ROW_CHUNK if row_hi > row_lo else -1
    for c in range(c0, c1 + 1):
        base = c * ROW_CHUNK
        n = min(ROW_CHUNK, rows - base)
        chunk = _rng(seed, stream, c).standard_normal((n, cols), dtype=np.float32)
        if std != 1.0:
            chunk *= np.float32(std)
        lo, hi = max(row_lo, base), min(row_hi, base + n)
        out[lo - row_lo:hi - row_lo] = chunk[lo - base:hi - base]
    return out


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """A float32 N(0, std^2) tensor of any shape (rows = all leading dims)."""
    shape = tuple(int(s) for s in shape)
    cols = shape[-1] if shape else 1
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    return normal_rows(seed, stream, rows, cols, std).reshape(shape)


def uniform_int(seed: int, stream: int, lo: int, hi: int, n: int) -> np.ndarray:
    """``n`` int32 values uniform on the closed range [lo, hi]."""
    return _rng(seed, stream).integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def distinct_slots(seed: int, stream: int, n: int, full_batch_size: int) -> np.ndarray:
    """``n`` distinct int32 slot ids drawn from [0, full_batch_size)."""
    if not 0 <= n <= full_batch_size:
        raise ValueError("n must lie in [0, full_batch_size]")
    return _rng(seed, stream).permutation(full_batch_size)[:n].astype(np.int32)


def cache_bits(seed: int, stream: int, shape, dtype: str) -> np.ndarray:
    """Initial KV-cache contents: N(0,1) values already in the cache dtype.

    Returned as uint16 bit patterns of shape ``shape``.  ``"f16"`` draws use
    numpy's float16 cast; ``"bf16"`` draws keep the top 16 bits of the float32
    draw (truncation).  Either is just a way of drawing values that are
    representable in the cache dtype; the KV write of the step itself (which
    rounds to nearest even) is not done here.
    """
    x = normal(seed, stream, shape)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError("dtype must be 'f16' or 'bf16'")


def cache_bits_rows(seed: int, stream: int, shape, dtype: str, row_lo: int, row_hi: int) -> np.ndarray:
    """Rows ``[row_lo, row_hi)`` of :func:`cache_bits` viewed as a 2-D
    ``(prod(shape[:-1]), shape[-1])`` matrix, without drawing the rest."""
    rows = int(np.prod(shape[:-1]))
    x = normal_rows(seed, stream, rows, int(shape[-1]), 1.0, row_lo, row_hi)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError("dtype must be 'f16' or 'bf16'")
