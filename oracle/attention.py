"""Multi-sequence GQA decode attention (oracle).

From antirez/ds4 PR #530, the multi-sequence decode attention commit: one
launch serves several sequences; sequence ``s`` reads its own query rows,
attends to its own cache with decode semantics and writes its own output rows,
so the result for a sequence is what an independent single-sequence run
gives.  From hw-native-sys/pypto-lib PR #841 (commit message): the live batch
and the per-sequence lengths come from the ``seq_lens`` descriptor.  From
quic/efficient-transformers PR #1305 ("Assumptions and limitations"): under
speculative decode each sequence carries K+1 = T query tokens.

Readings taken where the pages are silent:

* ``seq_lens[s]`` is the KV length after this step's T tokens are written;
  draft token ``j`` sits at position ``seq_lens[s] - T + j`` and sees keys
  ``0 .. seq_lens[s] - T + j`` (causal inside the draft).
* GQA: query head ``h`` uses kv head ``h // (Hq / Hkv)``.
* scores are ``q . k / sqrt(D)``; no soft-cap, no bias.

Written out in float64 with a plain (unsplit) softmax:

    p_j = exp(score_j - max score) / sum_j exp(score_j - max score)
    out = sum_j p_j V_j
"""
from __future__ import annotations

import numpy as np


def visible_keys(seq_len: int, tokens_per_seq: int, j: int) -> int:
    """Number of keys that draft token ``j`` of a sequence sees."""
    return seq_len - tokens_per_seq + j + 1


def weights(q_row: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Softmax weights of one query row over ``keys[L, D]`` (float64)."""
    d = keys.shape[-1]
    score = keys.astype(np.float64) @ q_row.astype(np.float64) / np.sqrt(np.float64(d))
    e = np.exp(score - np.max(score))
    return e / np.sum(e)


def attention_decode_multi(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           batch_index, tokens_per_seq: int, seq_lens,
                           heads=None) -> np.ndarray:
    """Decode attention for every token row of the live batch.

    ``q``: ``[n_tok, Hq, D]``; ``k_cache, v_cache``: float values
    ``[F, Hkv, C, D]``.  Returns float64 ``out[n_tok, Hq, D]``.  ``heads``
    restricts the computation to a subset of query heads (other rows are NaN).
    """
    n_tok, hq, d = q.shape
    hkv = k_cache.shape[1]
    if hq % hkv:
        raise ValueError("query heads must be a multiple of kv heads")
    group = hq // hkv
    out = np.full((n_tok, hq, d), np.nan)
    heads = range(hq) if heads is None else heads
    for s, slot in enumerate(np.asarray(batch_index)):
        for j in range(tokens_per_seq):
            t = s * tokens_per_seq + j
            vis = visible_keys(int(seq_lens[s]), tokens_per_seq, j)
            for h in heads:
                g = h // group
                p = weights(q[t, h], k_cache[slot, g, :vis])
                out[t, h] = p @ v_cache[slot, g, :vis].astype(np.float64)
    return out
