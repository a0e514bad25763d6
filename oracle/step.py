"""One llama-style batched decode step composed from the oracle's pieces.

The ds4 page ("What", "Design note") runs the dense stages once for all live
sessions with n_tokens = n_seqs and keeps KV append and attention per
sequence; the QAIC page ("Objective") addresses a retained cache of
full_batch_size slots through batch_index.  The layer order used here (the
pages do not print one) is the plain pre-norm llama layer:

    h   = embedding(token)
    per layer:
        x = quant(rmsnorm(h));  [q|k|v] = Wqkv x;  q, k <- rope(pos)
        cache[batch_index] <- k, v at pos;  a = attention(q, cache, seq_lens)
        h = h + Wo quant(a)
        x = quant(rmsnorm(h));  [g|u] = Wgu x;  h = h + Wdown quant(silu(g) u)
    logits = Whead quant(rmsnorm(h))

``quant`` rounds the float64 activation to float32 and applies the q8_0
codec: activations enter every matmul pre-quantised, as on the ds4 page.

No page prints an end-to-end value.  The composition is pinned by closed
forms instead (CPU tests): with some of a layer's matrices zero, whole stages
vanish and the step reduces to a short formula of the pinned pieces (the
head of the normed embedding; the embedding plus O times the mean of the
visible V rows; the FFN residual), which fixes the residual placement, the
norm of each stage, the gate / up order, the V slice and the write-before-
attend order.  The GPU step is compared with these pieces stage by stage.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import attention, glue, kv, matmul, paged, q8_0, rope


@dataclass(frozen=True)
class Shape:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_layers: int
    eps: float = 1e-6
    theta: float = 10000.0
    yarn: object = None   # rope.Yarn, or None for the plain RoPE


def quant(x: np.ndarray) -> np.ndarray:
    return q8_0.quantize_rows(np.asarray(x, dtype=np.float64).astype(np.float32))


def positions(seq_lens, tokens_per_seq: int) -> np.ndarray:
    """pos[s*T + j] = seq_lens[s] - T + j."""
    return np.array([int(L) - tokens_per_seq + j for L in seq_lens for j in range(tokens_per_seq)],
                    dtype=np.int64)


def decode_step(shape: Shape, w: dict, k_caches: list, v_caches: list, cache_dtype: str,
                token_ids, batch_index, tokens_per_seq: int, seq_lens, geometry=None):
    """Returns ``(logits float64 [n_tok, vocab], new k_caches, new v_caches)``.

    ``w`` may also hold per-layer float32 ``q_norm[l], k_norm[l]`` (width
    head_dim): a per-head RMS norm of q and k before their rotation.
    ``w`` holds q8_0 byte arrays ``embed, head`` and per layer ``wqkv[l],
    wo[l], wgu[l], wdown[l]`` plus float32 norm weights ``attn_norm[l],
    ffn_norm[l], final_norm``.  Caches are uint16 bit arrays ``[F, Hkv, C, D]``.

    ``geometry = (block_table, n_blocks, window)``: the caches are page pools
    ``[n_pages, Hkv, 128, D]`` in the paged / ring geometry of ``paged``
    (``batch_index`` unused), and the KV write and the attention go through it.
    """
    sh = shape
    pos = positions(seq_lens, tokens_per_seq)
    n_tok = len(pos)
    hq, hkv, d = sh.n_q_heads, sh.n_kv_heads, sh.head_dim
    h = glue.embedding(w["embed"], token_ids)
    new_k, new_v = [], []
    for layer in range(sh.n_layers):
        x = glue.rmsnorm(h, w["attn_norm"][layer], sh.eps)
        qkv = matmul.matmul_q8_0(w["wqkv"][layer], quant(x))
        q = qkv[:, :hq * d].reshape(n_tok, hq, d)
        k = qkv[:, hq * d:(hq + hkv) * d].reshape(n_tok, hkv, d)
        v = qkv[:, (hq + hkv) * d:].reshape(n_tok, hkv, d)
        # optional per-head q / k RMS norm before the rotation (Qwen3-style
        # q_norm / k_norm weights of width head_dim)
        qn = w["q_norm"][layer] if "q_norm" in w else None
        kn = w["k_norm"][layer] if "k_norm" in w else None
        q = rope.head_rmsnorm_rope(q, pos, sh.theta, qn, sh.eps, sh.yarn)
        k = rope.head_rmsnorm_rope(k, pos, sh.theta, kn, sh.eps, sh.yarn)
        if geometry is None:
            kc, vc = kv.kv_scatter(k_caches[layer], v_caches[layer], batch_index, tokens_per_seq, pos,
                                   k.astype(np.float32), v.astype(np.float32), cache_dtype)
            a = attention.attention_decode_multi(q, kv.bits_to_f64(kc, cache_dtype),
                                                 kv.bits_to_f64(vc, cache_dtype),
                                                 batch_index, tokens_per_seq, seq_lens)
        else:
            bt, nbk, win = geometry
            kc, vc = paged.scatter(k_caches[layer], v_caches[layer], bt, nbk, win, tokens_per_seq, pos,
                                   k.astype(np.float32), v.astype(np.float32), cache_dtype)
            a = paged.attention_paged(q, kv.bits_to_f64(kc, cache_dtype), kv.bits_to_f64(vc, cache_dtype),
                                      bt, nbk, win, tokens_per_seq, seq_lens)
        new_k.append(kc)
        new_v.append(vc)
        h = glue.residual_add(h, matmul.matmul_q8_0(w["wo"][layer], quant(a.reshape(n_tok, hq * d))))
        x = glue.rmsnorm(h, w["ffn_norm"][layer], sh.eps)
        gu = matmul.matmul_q8_0(w["wgu"][layer], quant(x))
        act = glue.silu_mul(gu[:, :sh.ffn], gu[:, sh.ffn:])
        h = glue.residual_add(h, matmul.matmul_q8_0(w["wdown"][layer], quant(act)))
    x = glue.rmsnorm(h, w["final_norm"], sh.eps)
    logits = matmul.matmul_q8_0(w["head"], quant(x))
    return logits, new_k, new_v
