"""CPU oracle of the batched decode step -- TEST INFRASTRUCTURE, NOT PRODUCT.

A plain, slow, obviously correct restatement of what one batched decode step
computes, in float64 wherever the method does not fix the precision.  It is
written from the three pages that describe the method:

* antirez/ds4 PR #530, "Batched decode: co-decode N live sessions in one GPU
  pass (opt-in)" -- the narrow-batch q8_0 matmul ("Why it's worth it -- the
  narrow-batch matmul"), the pos-vector RoPE and the multi-sequence decode
  attention (the commit bodies of the walk-through), and the per-session
  invariants ("Correctness").
* quic/efficient-transformers PR #1305, "[feature] Enable Dynamic Batching" --
  the retained KV cache sized for full_batch_size and addressed through
  batch_index ("Objective"), and K+1 speculative tokens per sequence on
  input_ids axis 1 ("Assumptions and limitations").
* hw-native-sys/pypto-lib PR #841, "Add: dynamic public batch (1..16) for
  Qwen3-14B decode" -- the live batch read from the seq_lens descriptor and the
  contract 1 <= batch <= batch_pad (commit message).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
and imports nothing from it; the product never calls it.

Modules
-------
q8_0       block codec (quantise / unpack / dequantise)
matmul     narrow-batch q8_0 matmul and its int32 block dot products
rope       pos-vector rotary embedding
kv         fp32 -> fp16 / bf16 round-to-nearest-even and the batch_index scatter
attention  multi-sequence GQA decode attention (unsplit softmax)
glue       RMSNorm, SiLU-gate, residual add, embedding gather
step       one llama-style decode step composed from the above

Every function is pinned by ``tests/test_oracle_*.py`` against values the
mathematics fixes (closed forms, invariants, brute force on tiny inputs,
library routines for special cases).  ``step.decode_step`` is a composition
of pinned functions, and the composition is pinned too: with some of a
layer's matrices zero it reduces to closed forms of the pinned pieces (the
head of the normed embedding, the attention and FFN residuals), which fix the
residual placement, the norm order, the gate / up order and the V slice (see
its docstring).
"""
