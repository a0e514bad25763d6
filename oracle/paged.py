"""Paged and ring (sliding-window) KV geometry per sequence (oracle).

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use this module; the library never does.

From antirez/ds4 PR #530 (the multi-sequence decode attention commit): every
sequence of a batched decode attention carries its own view of its cache --
its own cache location and ring geometry -- so that sequences of different
shapes and ring offsets share one launch.  From hw-native-sys/pypto-lib PR #841
(its paged attention and ``pa_max_blocks``): the cache is paged and a
sequence finds its keys through a table of blocks.

The pages name the geometry, not its layout; the reading taken:

* Page pool: ``[n_pages, Hkv, P, D]`` with ``P = 128`` keys per page (one
  attention chunk), K and V each in their own pool.
* Sequence ``s``: block table ``bt[s, 0 .. n_blocks[s])`` of page indices and a
  window ``W[s]`` (0: no window).
* The key at absolute position ``p`` is row ``p % P`` of page ``bt[s, i]``
  with ``i = p // P`` (linear, ``W = 0``) or ``i = (p // P) % n_blocks[s]``
  (ring, ``W > 0``: the newest ``n_blocks * P`` positions live in the ring).
* Draft token ``j`` of ``T`` sits at ``pos = seq_lens[s] - T + j`` and sees
  keys ``lo .. pos`` with ``lo = max(0, pos - W + 1)`` under a window, else 0.
* A ring must still hold every key a draft token sees after the step's ``T``
  writes: ``n_blocks * P >= W + T - 1``; a linear table must cover the
  sequence: ``ceil(seq_lens[s] / P) <= n_blocks``.
"""
from __future__ import annotations

import numpy as np

from . import attention, kv

PAGE = 128


def locate(p: int, bt_row, n_blocks: int, window: int):
    """(page, row) of absolute key position ``p`` of one sequence."""
    i = p // PAGE
    if window > 0:
        i %= n_blocks
    elif i >= n_blocks:
        raise ValueError("position beyond the sequence's block table")
    return int(bt_row[i]), p % PAGE


def visible_range(seq_len: int, tokens_per_seq: int, j: int, window: int):
    """Half-open range of key positions draft token ``j`` sees."""
    hi = attention.visible_keys(seq_len, tokens_per_seq, j)
    lo = max(0, hi - window) if window > 0 else 0
    return lo, hi


def check_geometry(block_table, n_blocks, window, tokens_per_seq: int, seq_lens):
    for s, L in enumerate(np.asarray(seq_lens)):
        nb, w = int(n_blocks[s]), int(window[s])
        if w > 0:
            if nb * PAGE < w + tokens_per_seq - 1:
                raise ValueError("ring smaller than window + T - 1")
        elif -(-int(L) // PAGE) > nb:
            raise ValueError("block table does not cover the sequence")


def scatter(k_pool: np.ndarray, v_pool: np.ndarray, block_table, n_blocks, window, tokens_per_seq: int,
            pos, k: np.ndarray, v: np.ndarray, dtype: str):
    """Copies of the uint16 pools ``[n_pages, Hkv, P, D]`` with the step's
    rows written at their (page, row); ``k, v`` float32 ``[n_tok, Hkv, D]``."""
    kp, vp = k_pool.copy(), v_pool.copy()
    kb, vb = kv.convert(k, dtype), kv.convert(v, dtype)
    pos = np.asarray(pos)
    n_seq = len(n_blocks)
    for s in range(n_seq):
        for j in range(tokens_per_seq):
            t = s * tokens_per_seq + j
            page, row = locate(int(pos[t]), block_table[s], int(n_blocks[s]), int(window[s]))
            kp[page, :, row, :] = kb[t]
            vp[page, :, row, :] = vb[t]
    return kp, vp


def attention_paged(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_table, n_blocks, window,
                    tokens_per_seq: int, seq_lens, heads=None) -> np.ndarray:
    """Decode attention through the paged geometry, float64.  ``k_pool,
    v_pool``: float values ``[n_pages, Hkv, P, D]``; returns
    ``out[n_tok, Hq, D]`` (rows of heads outside ``heads`` are NaN)."""
    n_tok, hq, d = q.shape
    hkv = k_pool.shape[1]
    group = hq // hkv
    out = np.full((n_tok, hq, d), np.nan)
    heads = range(hq) if heads is None else heads
    for s, L in enumerate(np.asarray(seq_lens)):
        for j in range(tokens_per_seq):
            t = s * tokens_per_seq + j
            lo, hi = visible_range(int(L), tokens_per_seq, j, int(window[s]))
            where = [locate(p, block_table[s], int(n_blocks[s]), int(window[s])) for p in range(lo, hi)]
            pages = np.array([w[0] for w in where])
            rows = np.array([w[1] for w in where])
            for h in heads:
                g = h // group
                keys = k_pool[pages, g, rows]
                vals = v_pool[pages, g, rows].astype(np.float64)
                out[t, h] = attention.weights(q[t, h], keys) @ vals
    return out
