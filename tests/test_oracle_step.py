"""Checks of the oracle's composed decode step (CPU only).

The composition is "parity unpinned" beyond its pinned parts; these tests
check the invariants the pages state for a batched step: each sequence's
result is what an independent single-sequence run gives (ds4 PR #530,
"Correctness"; the two-sessions smoke test in the session-split commit), and
cache slots not named in batch_index are untouched (the per-slot frontier
guard commit).
"""
import numpy as np

from oracle import q8_0, step
from tests import _shapes


def _oracle_weights(wf):
    w = {k: [q8_0.quantize_rows(m) for m in v] for k, v in wf.items() if k in ("wqkv", "wo", "wgu", "wdown")}
    w["head"] = q8_0.quantize_rows(wf["head"])
    w["embed"] = q8_0.quantize_rows(wf["embed"])
    w["attn_norm"], w["ffn_norm"], w["final_norm"] = wf["attn_norm"], wf["ffn_norm"], wf["final_norm"]
    return w


def _shape(ms):
    return step.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers)


def test_batched_step_equals_single_sequence_steps():
    ms = _shapes.TINY
    w = _oracle_weights(_shapes.weight_f32(0, ms))
    kc = [_shapes.cache_bits(0, ms, l, "k") for l in range(ms.n_layers)]
    vc = [_shapes.cache_bits(0, ms, l, "v") for l in range(ms.n_layers)]
    T = 2
    bi, lens, toks = _shapes.step_meta(0, ms, 3, T)
    logits, nk, nv = step.decode_step(_shape(ms), w, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    assert logits.shape == (3 * T, ms.vocab) and np.all(np.isfinite(logits))
    for s in range(3):
        one, _, _ = step.decode_step(_shape(ms), w, kc, vc, ms.cache_dtype, toks[s * T:(s + 1) * T],
                                     bi[s:s + 1], T, lens[s:s + 1])
        assert np.array_equal(one, logits[s * T:(s + 1) * T])
    untouched = np.ones(ms.full_batch_size, bool)
    untouched[bi] = False
    for l in range(ms.n_layers):
        assert np.array_equal(nk[l][untouched], kc[l][untouched])
        assert np.array_equal(nv[l][untouched], vc[l][untouched])


def test_positions_follow_seq_lens():
    assert list(step.positions([5, 3], 3)) == [2, 3, 4, 0, 1, 2]
