"""Checks of the oracle's composed decode step (CPU only).

No page prints an end-to-end value, so the composition is pinned by closed
forms: with some of a layer's matrices zero, whole stages vanish and the step
reduces to a short formula of the separately pinned pieces (residual
placement, each stage's norm, the gate / up order, the V slice, the
write-before-attend order).  The tests also check the invariants the pages
state for a batched step: each sequence's result is what an independent
single-sequence run gives (ds4 PR #530, "Correctness"; the two-sessions smoke
test in the session-split commit), cache slots not named in batch_index are
untouched (the per-slot frontier guard commit), a T-token draft step equals T
one-token steps, and only visible history reaches the logits.
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


# ---------------------------------------------------------------------------
# Closed forms that pin the layer wiring of the composed step.  Zeroing some
# of a layer's matrices makes whole stages vanish (a q8_0 block of zeros has
# d = 0 and codes 0, so W x = 0 exactly, and silu(0) * 0 = 0), and with q = 0
# every visible key gets the same score, so attention is the plain mean of
# the visible V rows.  What is left is a short formula written out below from
# the pinned pieces; a residual that replaced h instead of adding to it, a
# norm weight taken from the wrong stage, gate and up swapped, the V slice
# taken from the wrong columns, K/V written after the attention instead of
# before, or a final norm / head in the wrong place each change the logits.
# ---------------------------------------------------------------------------
from oracle import glue, kv as okv, matmul as omm


def _q8(x):
    return q8_0.quantize_rows(np.asarray(x, dtype=np.float64).astype(np.float32))


def _pin_model(seed, zero):
    """TINY weights with the named per-layer matrices zeroed ({(layer, name)})
    and distinct norm weights per stage."""
    ms = _shapes.TINY
    wf = _shapes.weight_f32(seed, ms)
    rng = np.random.default_rng(100 + seed)
    for name in ("attn_norm", "ffn_norm"):
        wf[name] = [(1.0 + 0.3 * rng.standard_normal(ms.hidden)).astype(np.float32) for _ in range(ms.n_layers)]
    wf["final_norm"] = (1.0 + 0.3 * rng.standard_normal(ms.hidden)).astype(np.float32)
    for layer, name in zero:
        if name in ("wq", "wk", "wv"):   # one slice of the fused [q | k | v] rows
            hq, hkv, d = ms.n_q_heads, ms.n_kv_heads, ms.head_dim
            lo, hi = {"wq": (0, hq * d), "wk": (hq * d, (hq + hkv) * d), "wv": ((hq + hkv) * d, (hq + 2 * hkv) * d)}[name]
            wf["wqkv"][layer] = wf["wqkv"][layer].copy()
            wf["wqkv"][layer][lo:hi] = 0.0
        else:
            wf[name][layer] = np.zeros_like(wf[name][layer])
    return ms, _oracle_weights(wf), wf


def _run_pin(seed, zero, b=3, T=2):
    ms, w, wf = _pin_model(seed, zero)
    kc = [_shapes.cache_bits(seed, ms, l, "k") for l in range(ms.n_layers)]
    vc = [_shapes.cache_bits(seed, ms, l, "v") for l in range(ms.n_layers)]
    bi, lens, toks = _shapes.step_meta(seed, ms, b, T, 4)
    logits, nk, nv = step.decode_step(_shape(ms), w, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    return ms, w, kc, vc, bi, lens, toks, T, logits, nk, nv


def _head(ms, w, h):
    return omm.matmul_q8_0(w["head"], _q8(glue.rmsnorm(h, w["final_norm"], ms.eps)))


def _uniform_attention(ms, vcache_f64, bi, lens, T, v_new=None):
    """Attention with q = 0: the mean of the visible V rows.  Token j of
    sequence s sits at pos = lens[s] - T + j and sees rows 0..pos; rows
    lens[s] - T .. pos are the ones this step wrote (v_new, or zeros)."""
    hq, hkv, d = ms.n_q_heads, ms.n_kv_heads, ms.head_dim
    g = hq // hkv
    out = np.zeros((len(bi) * T, hq, d))
    for s, slot in enumerate(bi):
        lo = int(lens[s]) - T
        for j in range(T):
            for h in range(hq):
                rows = [vcache_f64[slot, h // g, p] for p in range(lo)]
                for jj in range(j + 1):
                    rows.append(np.zeros(d) if v_new is None else v_new[s * T + jj, h // g])
                out[s * T + j, h] = np.sum(rows, axis=0) / (lo + j + 1)
    return out.reshape(len(bi) * T, hq * d)


ALL = ("wqkv", "wo", "wgu", "wdown")


def test_step_with_zero_layers_is_the_head_of_the_normed_embedding():
    """Every layer matrix zero: h stays the embedding through both layers (the
    residuals add zero), the new K/V rows are zero, and
    logits = Whead q8(rmsnorm(embed[tok], final_norm))."""
    zero = {(l, n) for l in range(2) for n in ALL}
    ms, w, kc, vc, bi, lens, toks, T, logits, nk, nv = _run_pin(0, zero)
    want = _head(ms, w, glue.embedding(w["embed"], toks))
    assert np.allclose(logits, want, rtol=1e-12, atol=1e-12)
    for l in range(ms.n_layers):
        for s, slot in enumerate(bi):
            rows = slice(int(lens[s]) - T, int(lens[s]))
            for c in (nk[l], nv[l]):   # +0 or -0 (the rotation of a zero pair may give -0)
                assert np.all(okv.bits_to_f64(c[slot][:, rows], ms.cache_dtype) == 0)


def test_step_attention_residual_closed_form():
    """Only layer 0's O projection is nonzero: q = k = v = 0, so the attention
    is the mean of the visible V rows (old history plus the zero rows this
    step wrote before attending), and h = embed + Wo q8(mean).  Layer 0's
    down projection is nonzero too, but its input silu(0) * 0 is zero."""
    zero = {(0, "wqkv"), (0, "wgu")} | {(1, n) for n in ALL}
    ms, w, kc, vc, bi, lens, toks, T, logits, nk, nv = _run_pin(1, zero)
    a = _uniform_attention(ms, okv.bits_to_f64(vc[0], ms.cache_dtype), bi, lens, T)
    h = glue.embedding(w["embed"], toks) + omm.matmul_q8_0(w["wo"][0], _q8(a))
    assert np.allclose(logits, _head(ms, w, h), rtol=1e-9, atol=1e-12)


def test_step_v_slice_is_written_before_attention():
    """Layer 0 has only its V rows (the last Hkv*D rows of [q | k | v]) and
    O: q = k = 0, the step writes v = Wv q8(rmsnorm(embed, attn_norm)) into
    the cache before attending, and draft token j averages the old rows with
    the new rows of drafts 0..j."""
    zero = {(0, "wq"), (0, "wk"), (0, "wgu")} | {(1, n) for n in ALL}
    ms, w, kc, vc, bi, lens, toks, T, logits, nk, nv = _run_pin(2, zero)
    hq, hkv, d = ms.n_q_heads, ms.n_kv_heads, ms.head_dim
    emb = glue.embedding(w["embed"], toks)
    qkv = omm.matmul_q8_0(w["wqkv"][0], _q8(glue.rmsnorm(emb, w["attn_norm"][0], ms.eps)))
    v = qkv[:, (hq + hkv) * d:].astype(np.float32).reshape(-1, hkv, d)
    v_new = okv.bits_to_f64(okv.convert(v, ms.cache_dtype), ms.cache_dtype)
    a = _uniform_attention(ms, okv.bits_to_f64(vc[0], ms.cache_dtype), bi, lens, T, v_new)
    h = emb + omm.matmul_q8_0(w["wo"][0], _q8(a))
    assert np.allclose(logits, _head(ms, w, h), rtol=1e-9, atol=1e-12)
    for s, slot in enumerate(bi):
        for j in range(T):
            p = int(lens[s]) - T + j
            assert np.array_equal(nv[0][slot][:, p], okv.convert(v[s * T + j], ms.cache_dtype))
            assert np.all(okv.bits_to_f64(nk[0][slot][:, p], ms.cache_dtype) == 0)


def test_step_ffn_residual_closed_form_over_two_layers():
    """Layer 0 keeps only its FFN, layer 1 only its attention output path:
    h1 = embed + Wdown0 q8(silu(g) * u) with [g | u] = Wgu0 q8(rmsnorm(embed,
    ffn_norm0)) (gate columns first), then h2 = h1 + Wo1 q8(mean of layer 1's
    visible V rows), logits = Whead q8(rmsnorm(h2, final_norm))."""
    zero = {(0, "wqkv"), (0, "wo"), (1, "wqkv"), (1, "wgu")}
    ms, w, kc, vc, bi, lens, toks, T, logits, nk, nv = _run_pin(3, zero)
    emb = glue.embedding(w["embed"], toks)
    gu = omm.matmul_q8_0(w["wgu"][0], _q8(glue.rmsnorm(emb, w["ffn_norm"][0], ms.eps)))
    act = glue.silu_mul(gu[:, :ms.ffn], gu[:, ms.ffn:])
    h1 = emb + omm.matmul_q8_0(w["wdown"][0], _q8(act))
    a = _uniform_attention(ms, okv.bits_to_f64(vc[1], ms.cache_dtype), bi, lens, T)
    h2 = h1 + omm.matmul_q8_0(w["wo"][1], _q8(a))
    assert np.allclose(logits, _head(ms, w, h2), rtol=1e-9, atol=1e-12)
    # the alternatives a miswired step would compute differ
    swapped = emb + omm.matmul_q8_0(w["wdown"][0], _q8(glue.silu_mul(gu[:, ms.ffn:], gu[:, :ms.ffn])))
    assert not np.allclose(_head(ms, w, swapped + (h2 - h1)), logits, rtol=1e-3)
    wrong_norm = omm.matmul_q8_0(w["wgu"][0], _q8(glue.rmsnorm(emb, w["attn_norm"][0], ms.eps)))
    assert not np.allclose(wrong_norm, gu, rtol=1e-3)
