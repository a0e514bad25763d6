"""dsb: the batched multi-session decode step for GB300 (sm_103a).

One step advances ``b`` live sessions (1 <= b <= full_batch_size) by one
token each, or by K+1 tokens under speculative decode, in one GPU pass:
a narrow-batch q8_0 matmul, a pos-vector RoPE, a KV scatter/read through
``batch_index`` into a cache sized for ``full_batch_size``, and a
multi-sequence GQA decode attention.

The compute lives in ``libdsb.so`` (hand-written CUDA kernels behind a C
ABI declared in ``include/dsb.h``); :mod:`.dsb` is the ctypes binding and
loads that library lazily, failing loudly if it has not been built.
:mod:`.synth` makes the seeded synthetic inputs.  Importing this package
loads nothing native.
"""

__all__ = ["dsb", "synth", "build"]
