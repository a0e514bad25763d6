"""Pins of the oracle's decode step on paged and ring (sliding-window) KV
(``oracle.step.decode_step`` with a geometry) against the contiguous-cache
step, whose composition the closed forms of test_oracle_step.py pin, and
against itself under another block layout holding the same keys.  The page
and ring arithmetic itself is pinned in test_oracle_paged.py."""
import numpy as np

from oracle import paged as opg
from oracle import step
from tests import _shapes
from tests.test_oracle_step import _oracle_weights, _shape

P = opg.PAGE
# a tiny model over three 128-key pages per slot
MS = _shapes.ModelShape("tiny-paged", 256, 4, 2, 64, 512, 1000, 2, 4, 3 * P, "f16")


def _case(seed, b=3, T=2, min_len=None):
    w = _oracle_weights(_shapes.weight_f32(seed, MS))
    kc = [_shapes.cache_bits(seed, MS, l, "k") for l in range(MS.n_layers)]
    vc = [_shapes.cache_bits(seed, MS, l, "v") for l in range(MS.n_layers)]
    bi, lens, toks = _shapes.step_meta(seed, MS, b, T, min_len)
    return w, kc, vc, bi, lens, toks, T


def _pools(caches, perm):
    """Page pools holding every slot's blocks: block i of slot f at page perm[f * nb + i]."""
    nb = MS.ctx // P
    out = []
    for c in caches:
        pool = np.zeros((MS.full_batch_size * nb, MS.n_kv_heads, P, MS.head_dim), c.dtype)
        for f in range(MS.full_batch_size):
            for i in range(nb):
                pool[perm[f * nb + i]] = c[f, :, i * P:(i + 1) * P]
        out.append(pool)
    return out


def test_linear_pages_equal_the_contiguous_step():
    w, kc, vc, bi, lens, toks, T = _case(11)
    nb = MS.ctx // P
    perm = np.random.default_rng(5).permutation(MS.full_batch_size * nb)
    want, nk, nv = step.decode_step(_shape(MS), w, kc, vc, MS.cache_dtype, toks, bi, T, lens)
    bt = np.array([[perm[int(f) * nb + i] for i in range(nb)] for f in bi])
    geo = (bt, np.full(len(bi), nb), np.zeros(len(bi), int))
    got, pk, pv = step.decode_step(_shape(MS), w, _pools(kc, perm), _pools(vc, perm), MS.cache_dtype, toks, None,
                                   T, lens, geometry=geo)
    assert np.array_equal(got, want)
    for l in range(MS.n_layers):
        assert np.array_equal(pk[l], _pools([nk[l]], perm)[0])
        assert np.array_equal(pv[l], _pools([nv[l]], perm)[0])
    # a window no shorter than any sequence hides nothing
    wide = (bt, geo[1], np.full(len(bi), MS.ctx))
    same, _, _ = step.decode_step(_shape(MS), w, _pools(kc, perm), _pools(vc, perm), MS.cache_dtype, toks, None, T,
                                  lens, geometry=wide)
    assert np.array_equal(same, want)
    # and a short window changes the logits
    short = (bt, geo[1], np.full(len(bi), 40))
    other, _, _ = step.decode_step(_shape(MS), w, _pools(kc, perm), _pools(vc, perm), MS.cache_dtype, toks, None, T,
                                   lens, geometry=short)
    assert not np.allclose(other, want, rtol=1e-3)


def test_ring_equals_linear_pages_under_the_same_window():
    """Sequences longer than a two-page ring: the ring holds the last 256
    positions at (p / 128) mod 2, and under a window W with W + T - 1 <= 256
    every visible key is there, so the step equals the same step on linear
    pages holding the whole history."""
    w, kc, vc, bi, lens, toks, T = _case(12, min_len=2 * P + 20)
    nb, W = MS.ctx // P, 200
    perm = np.arange(MS.full_batch_size * nb)
    lin_bt = np.array([[perm[int(f) * nb + i] for i in range(nb)] for f in bi])
    win = np.full(len(bi), W)
    want, _, _ = step.decode_step(_shape(MS), w, _pools(kc, perm), _pools(vc, perm), MS.cache_dtype, toks, None, T,
                                  lens, geometry=(lin_bt, np.full(len(bi), nb), win))
    ring_bt = np.array([[2 * s + 1, 2 * s] for s in range(len(bi))])  # two pages each, swapped order
    rk, rv = [], []
    for c in (kc, vc):
        pools = []
        for l in range(MS.n_layers):
            pool = np.zeros((2 * len(bi), MS.n_kv_heads, P, MS.head_dim), c[l].dtype)
            for s, f in enumerate(bi):
                for p in range(max(0, int(lens[s]) - 2 * P), int(lens[s]) - T):
                    page, row = opg.locate(p, ring_bt[s], 2, W)
                    pool[page, :, row] = c[l][f, :, p]
            pools.append(pool)
        (rk if c is kc else rv).extend(pools)
    got, _, _ = step.decode_step(_shape(MS), w, rk, rv, MS.cache_dtype, toks, None, T, lens,
                                 geometry=(ring_bt, np.full(len(bi), 2), win))
    assert np.array_equal(got, want)
