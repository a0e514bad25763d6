"""Workload shapes and seeded draws shared by the tests.

Shapes follow the workloads the pages measure on (llama-68m-shaped decode on
the QAIC page, Qwen3-14B-shaped decode on the pypto page, DeepSeek-class
dense stages and long context on the ds4 page).  Every value is drawn by
``session_decode_step_dsb_gb300.synth`` and is a pure function of the seed.
"""
from __future__ import annotations

import numpy as np

from session_decode_step_dsb_gb300 import synth


from session_decode_step_dsb_gb300.workloads import LLAMA68M, ModelShape  # noqa: F401

QWEN3_14B_1L = ModelShape("qwen3-14b-shaped-1-layer", 5120, 40, 8, 128, 17408, 151936, 1, 16, 4096, "bf16",
                          qk_norm=True)
# One Qwen3-14B-shaped layer (GQA 40/8, head_dim 128, FFN 17408, bf16 cache
# [16, 8, 4096, 128]) under a 4096-row head: the layer is the workload's, the
# head is cut to keep the oracle's weight draws to seconds (the full 151936-row
# head is a plain matmul shape, checked by the matmul tests).
QWEN3_14B_LAYER = ModelShape("qwen3-14b-shaped-layer", 5120, 40, 8, 128, 17408, 4096, 1, 16, 4096, "bf16",
                             qk_norm=True)
TINY = ModelShape("tiny", 256, 4, 2, 64, 512, 1000, 2, 4, 96, "f16")
TINY_BF16 = ModelShape("tiny-bf16", 512, 8, 2, 128, 768, 700, 1, 5, 300, "bf16")
# tiny shapes with the per-head q / k RMS norm before the rope
TINY_QKN = ModelShape("tiny-qknorm", 256, 4, 2, 64, 512, 1000, 2, 4, 96, "f16", qk_norm=True)
TINY_BF16_QKN = ModelShape("tiny-bf16-qknorm", 512, 8, 2, 128, 768, 700, 1, 5, 300, "bf16", qk_norm=True)
# tiny shapes with the YaRN RoPE (context extended 4x over an original 64 / 128)
TINY_YARN = ModelShape("tiny-yarn", 256, 4, 2, 64, 512, 1000, 2, 4, 256, "f16", qk_norm=True, yarn_factor=4.0,
                       yarn_orig_ctx=64)
# many sessions x long drafts: n_tok = 64 * 32 = 2048 token rows, so a captured
# step's metadata (2 n_tok + 3 b + 1 words) outgrows the first kernel's
# parameter block and is read from mapped pinned memory instead
TINY_WIDE = ModelShape("tiny-wide", 256, 4, 2, 64, 512, 1000, 1, 80, 64, "f16")
TINY_BF16_YARN = ModelShape("tiny-bf16-yarn", 512, 8, 2, 128, 768, 700, 1, 5, 300, "bf16", yarn_factor=4.0,
                            yarn_orig_ctx=128)

W_STD = 0.02


def weight_f32(seed: int, shape: ModelShape):
    """float32 weight draws {name: array}; per layer lists for layered ones."""
    sid = synth.stream_id
    out = {"wqkv": [], "wo": [], "wgu": [], "wdown": []}
    for layer in range(shape.n_layers):
        out["wqkv"].append(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * layer + 0), shape.qkv_rows, shape.hidden, W_STD))
        out["wo"].append(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * layer + 1), shape.hidden, shape.n_q_heads * shape.head_dim, W_STD))
        out["wgu"].append(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * layer + 2), 2 * shape.ffn, shape.hidden, W_STD))
        out["wdown"].append(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * layer + 3), shape.hidden, shape.ffn, W_STD))
    out["head"] = synth.normal_rows(seed, sid(synth.STREAM_W, 999_000), shape.vocab, shape.hidden, W_STD)
    out["embed"] = synth.normal_rows(seed, sid(synth.STREAM_EMBED, 0), shape.vocab, shape.hidden, W_STD)
    out["attn_norm"] = [np.ones(shape.hidden, np.float32) for _ in range(shape.n_layers)]
    out["ffn_norm"] = [np.ones(shape.hidden, np.float32) for _ in range(shape.n_layers)]
    out["final_norm"] = np.ones(shape.hidden, np.float32)
    if shape.qk_norm:   # weights around 1, as trained q / k norms are
        for name, idx in (("q_norm", 4), ("k_norm", 5)):
            out[name] = [(1.0 + synth.normal_rows(seed, sid(synth.STREAM_W, 10 * layer + idx), 1, shape.head_dim,
                                                  0.1)[0]).astype(np.float32) for layer in range(shape.n_layers)]
    return out


def cache_bits(seed: int, shape: ModelShape, layer: int, which: str):
    kind = synth.STREAM_KCACHE if which == "k" else synth.STREAM_VCACHE
    dims = (shape.full_batch_size, shape.n_kv_heads, shape.ctx, shape.head_dim)
    return synth.cache_bits(seed, synth.stream_id(kind, layer), dims, shape.cache_dtype)


def step_meta(seed: int, shape: ModelShape, b: int, T: int, min_len: int | None = None):
    """batch_index (distinct), seq_lens (>= T) and token ids for one step."""
    sid = synth.stream_id
    bi = synth.distinct_slots(seed, sid(synth.STREAM_META, 1), b, shape.full_batch_size)
    lo = max(T, min_len if min_len is not None else T)
    lens = synth.uniform_int(seed, sid(synth.STREAM_META, 2), lo, shape.ctx, b)
    toks = synth.uniform_int(seed, sid(synth.STREAM_TOKENS, 0), 0, shape.vocab - 1, b * T)
    return bi, lens, toks
