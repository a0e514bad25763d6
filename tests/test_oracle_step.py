"""Checks of the oracle's composed decode step (CPU only).

The composition is "parity unpinned" beyond its pinned parts (no printed
end-to-end value exists); these tests check the invariants the pages state for
a batched step: each sequence's result is what an independent single-sequence
run gives (ds4 PR #530, "Correctness"; the two-sessions smoke test in the
session-split commit), cache slots not named in batch_index are untouched (the
per-slot frontier guard commit), a T-token draft step equals T one-token steps,
and only visible history reaches the logits.
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


def _tiny_case(seed, b, T, min_len):
    ms = _shapes.TINY
    w = _oracle_weights(_shapes.weight_f32(seed, ms))
    kc = [_shapes.cache_bits(seed, ms, l, "k") for l in range(ms.n_layers)]
    vc = [_shapes.cache_bits(seed, ms, l, "v") for l in range(ms.n_layers)]
    bi, lens, toks = _shapes.step_meta(seed, ms, b, T, min_len)
    return ms, w, kc, vc, bi, lens, toks


def test_draft_tokens_equal_successive_single_token_steps():
    """A step of T draft tokens per sequence gives, for draft token j, the
    logits that the j-th of T successive one-token steps gives (each on the
    cache the previous one wrote), and leaves the same cache: token j sees the
    keys up to its own position and no later draft key (ds4 PR #530, the
    speculative verification batch; QAIC page, positions = seq_lens - 1 for
    T = 1).  A visible range that ignored j, or a position off by one, moves
    these logits."""
    T = 3
    ms, w, kc, vc, bi, lens, toks = _tiny_case(1, 2, T, 6)
    logits, nk, nv = step.decode_step(_shape(ms), w, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    ck, cv = kc, vc
    for j in range(T):
        lens_j = lens - T + j + 1
        toks_j = toks.reshape(len(bi), T)[:, j].copy()
        one, ck, cv = step.decode_step(_shape(ms), w, ck, cv, ms.cache_dtype, toks_j, bi, 1, lens_j)
        for s in range(len(bi)):
            assert np.array_equal(one[s], logits[s * T + j]), (s, j)
    for l in range(ms.n_layers):
        assert np.array_equal(ck[l], nk[l]) and np.array_equal(cv[l], nv[l])


def test_only_visible_history_reaches_the_logits():
    """Cache rows a step cannot see -- other slots, positions at or past
    seq_lens, and the rows the step's own writes replace -- do not change its
    logits; one row of visible history of one sequence changes that
    sequence's logits and no other's (the per-slot isolation of the QAIC
    page's batch_index and of ds4's per-sequence views)."""
    T = 2
    ms, w, kc, vc, bi, lens, toks = _tiny_case(2, 3, T, 8)
    base, _, _ = step.decode_step(_shape(ms), w, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    rng = np.random.default_rng(3)
    pk = [c.copy() for c in kc]
    pv = [c.copy() for c in vc]
    live = set(int(f) for f in bi)
    for l in range(ms.n_layers):
        for f in range(ms.full_batch_size):
            if f not in live:
                pk[l][f] = rng.integers(0, 0x7bff, pk[l][f].shape, dtype=np.uint16)
                pv[l][f] = rng.integers(0, 0x7bff, pv[l][f].shape, dtype=np.uint16)
        for s, f in enumerate(bi):
            lo = int(lens[s]) - T   # the step writes lo .. lens-1; nothing at or past lens is visible
            pk[l][f, :, lo:] = rng.integers(0, 0x3bff, pk[l][f, :, lo:].shape, dtype=np.uint16)
            pv[l][f, :, lo:] = rng.integers(0, 0x3bff, pv[l][f, :, lo:].shape, dtype=np.uint16)
    same, _, _ = step.decode_step(_shape(ms), w, pk, pv, ms.cache_dtype, toks, bi, T, lens)
    assert np.array_equal(same, base)
    hk = [c.copy() for c in kc]
    hk[0][bi[1], 0, 0] ^= np.uint16(0x0400)   # one visible key of sequence 1, layer 0, exponent bit
    moved, _, _ = step.decode_step(_shape(ms), w, hk, vc, ms.cache_dtype, toks, bi, T, lens)
    for s in range(len(bi)):
        rows = slice(s * T, (s + 1) * T)
        if s == 1:
            assert np.all(np.any(moved[rows] != base[rows], axis=1))
        else:
            assert np.array_equal(moved[rows], base[rows])
