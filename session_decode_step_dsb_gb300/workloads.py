"""Shapes of the workloads the step is measured and checked on.

The pages measure on named models; only their shapes are used here, with
random N(0, 0.02) q8_0 weights (no trained weights are involved):
llama-68m-shaped decode (quic/efficient-transformers PR #1305, "Dynamic
batching decode latency performance"), Qwen3-14B-shaped decode
(hw-native-sys/pypto-lib PR #841), and DeepSeek-class dense-stage and
long-context shapes (antirez/ds4 PR #530 runs DeepSeek V4 Flash).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class ModelShape:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_layers: int
    full_batch_size: int
    ctx: int
    cache_dtype: str  # "f16" or "bf16"
    eps: float = 1e-6
    theta: float = 10000.0
    qk_norm: bool = False  # per-head RMS norm of q and k before the rope (Qwen3 layers have one)
    yarn_factor: float = 0.0  # > 1: YaRN RoPE over the original context yarn_orig_ctx
    yarn_orig_ctx: int = 0

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


# llama-68m shapes: hidden 768, 12 heads (MHA), head_dim 64, 2 layers, FFN 3072,
# vocab 32000; fp16 cache of full_batch_size 8 at ctx 2048.
LLAMA68M = ModelShape("llama-68m-shaped", 768, 12, 12, 64, 3072, 32000, 2, 8, 2048, "f16")
# Same shapes with full_batch_size 128 for the batch x speculative-decode sweep.
LLAMA68M_SPEC = ModelShape("llama-68m-shaped-spec", 768, 12, 12, 64, 3072, 32000, 2, 128, 2048, "f16")
# Qwen3-14B shapes: hidden 5120, 40 q heads, 8 kv heads, head_dim 128, FFN 17408,
# vocab 151936; bf16 cache [16, 8, 4096, 128].  The page gives no layer count
# for the measured step; the full model has 40 layers.
QWEN3_14B = ModelShape("qwen3-14b-shaped", 5120, 40, 8, 128, 17408, 151936, 40, 16, 4096, "bf16", qk_norm=True)

WEIGHT_STD = 0.02
