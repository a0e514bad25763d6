"""KV-cache write through batch_index (oracle), with the fp32 -> fp16 / bf16
conversions it needs.

From quic/efficient-transformers PR #1305 ("Objective"): the retained KV cache
is always sized for ``full_batch_size`` and a live batch of ``b`` sequences
addresses it through ``batch_index``.  From antirez/ds4 PR #530 (the
batched-decode encoder commit): each sequence appends its own K/V inside the
batched step.  Written out, for sequence ``s < b``, draft token ``j < T`` and
token row ``t = s*T + j``:

    K[batch_index[s], h, pos[t], :] = cvt(k[t, h, :])   for every kv head h
    V[batch_index[s], h, pos[t], :] = cvt(v[t, h, :])

and nothing else in the cache changes.  ``cvt`` rounds a float32 to the cache
dtype, to nearest with ties to even; both converters below are written from
the IEEE 754 binary16 and the bfloat16 (top half of binary32) definitions.
"""
from __future__ import annotations

import numpy as np


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE binary32 -> binary16, round to nearest, ties to even (uint16 bits).

    A finite binary32 value is ``num * 2**vexp`` with ``num`` its 24-bit
    significand.  The binary16 grid spacing at magnitude ``2**top`` is
    ``2**max(top - 10, -24)`` (10 fraction bits; the subnormal spacing is
    2^-24); the value is divided by that spacing with round-half-even, and a
    carry out of the significand moves to the next binade.  Exponents past
    binary16's range give infinity.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.int64)
    sign = (u >> 31) & 1
    e = (u >> 23) & 0xFF
    m = u & 0x7FFFFF
    special = e == 0xFF
    tiny = e == 0                                   # float32 zero/subnormal: |x| < 2^-126 -> +-0
    num = m | 0x800000
    vexp = e - 150
    top = e - 127
    grid = np.maximum(top - 10, -24)
    shift = np.clip(grid - vexp, 1, 26)             # always >= 13 for finite normal inputs
    k = num >> shift
    rem = num & ((np.int64(1) << shift) - 1)
    half = np.int64(1) << (shift - 1)
    k = k + ((rem > half) | ((rem == half) & ((k & 1) == 1))).astype(np.int64)
    carry = k == 0x800
    k = np.where(carry, 0x400, k)
    grid = grid + carry.astype(np.int64)
    E = grid + 25
    normal_bits = np.where(E >= 31, 0x7C00, (E << 10) | (k & 0x3FF))
    h = np.where(grid == -24, k, normal_bits)      # subnormal grid: the count itself is the encoding
    h = np.where(tiny, 0, h)
    h = np.where(special, 0x7C00 | np.where(m != 0, 0x200, 0), h)
    return (h | (sign << 15)).astype(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 (the top 16 bits), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi = u >> np.uint64(16)
    lo = u & np.uint64(0xFFFF)
    is_nan = ((u >> np.uint64(23)) & np.uint64(0xFF) == 0xFF) & ((u & np.uint64(0x7FFFFF)) != 0)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    r = hi + up.astype(np.uint64)
    r = np.where(is_nan, hi | np.uint64(0x40), r)
    return r.astype(np.uint16)


def f16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bits_to_f64(b: np.ndarray, dtype: str) -> np.ndarray:
    return f16_bits_to_f64(b) if dtype == "f16" else bf16_bits_to_f64(b)


def convert(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_f16_bits(x) if dtype == "f16" else f32_to_bf16_bits(x)


def kv_scatter(k_cache: np.ndarray, v_cache: np.ndarray, batch_index, tokens_per_seq: int,
               pos, k: np.ndarray, v: np.ndarray, dtype: str):
    """Return copies of the uint16 caches ``[F, Hkv, C, D]`` with the step's
    rows written; ``k, v`` are float32 ``[n_tok, Hkv, D]``."""
    kc, vc = k_cache.copy(), v_cache.copy()
    batch_index = np.asarray(batch_index)
    pos = np.asarray(pos)
    kb, vb = convert(k, dtype), convert(v, dtype)
    for s, slot in enumerate(batch_index):
        for j in range(tokens_per_seq):
            t = s * tokens_per_seq + j
            kc[slot, :, pos[t], :] = kb[t]
            vc[slot, :, pos[t], :] = vb[t]
    return kc, vc
