"""Pins of the paged / ring KV geometry oracle (oracle/paged.py) against facts
that do not go through its own code path: the contiguous-cache oracle on the
same keys, brute force over an explicit key list, and a dictionary model of
ring writes."""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import kv as okv
from oracle import paged as opg

P = opg.PAGE


def _contiguous_case(seed, F=3, hkv=2, hq=4, C=3 * P, D=8, T=1, dtype="f16"):
    rng = np.random.default_rng(seed)
    kc = okv.convert(rng.standard_normal((F, hkv, C, D)).astype(np.float32), dtype)
    vc = okv.convert(rng.standard_normal((F, hkv, C, D)).astype(np.float32), dtype)
    bi = np.array([2, 0], np.int64)
    lens = np.array([C - 5, P + 3], np.int64)
    q = rng.standard_normal((len(bi) * T, hq, D))
    return kc, vc, bi, lens, q


def _pool_from_contiguous(kc, vc, perm=None):
    """Pages of the contiguous cache, slot f's block i at page f*nb + i (or
    its image under perm)."""
    F, hkv, C, D = kc.shape
    nb = C // P
    n_pages = F * nb
    perm = np.arange(n_pages) if perm is None else perm
    kp = np.zeros((n_pages, hkv, P, D), kc.dtype)
    vp = np.zeros_like(kp)
    for f in range(F):
        for i in range(nb):
            kp[perm[f * nb + i]] = kc[f, :, i * P:(i + 1) * P]
            vp[perm[f * nb + i]] = vc[f, :, i * P:(i + 1) * P]
    return kp, vp, nb, perm


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("permute", [False, True])
def test_linear_pages_equal_the_contiguous_cache(T, permute):
    kc, vc, bi, lens, _ = _contiguous_case(1, T=T)
    q = np.random.default_rng(2).standard_normal((len(bi) * T, 4, 8))
    perm = np.random.default_rng(3).permutation(kc.shape[0] * (kc.shape[2] // P)) if permute else None
    kp, vp, nb, perm = _pool_from_contiguous(kc, vc, perm)
    bt = np.array([[perm[f * nb + i] for i in range(nb)] for f in bi])
    n_blocks = np.full(len(bi), nb)
    window = np.zeros(len(bi), np.int64)
    got = opg.attention_paged(q, okv.bits_to_f64(kp, "f16"), okv.bits_to_f64(vp, "f16"), bt, n_blocks, window, T,
                              lens)
    want = oatt.attention_decode_multi(q, okv.bits_to_f64(kc, "f16"), okv.bits_to_f64(vc, "f16"), bi, T, lens)
    assert np.array_equal(got, want)


def test_window_not_shorter_than_the_sequence_changes_nothing():
    kc, vc, bi, lens, q = _contiguous_case(4)
    kp, vp, nb, perm = _pool_from_contiguous(kc, vc)
    bt = np.array([[f * nb + i for i in range(nb)] for f in bi])
    kf, vf = okv.bits_to_f64(kp, "f16"), okv.bits_to_f64(vp, "f16")
    base = opg.attention_paged(q, kf, vf, bt, np.full(2, nb), np.zeros(2, np.int64), 1, lens)
    # a ring of all nb pages with a window as long as the sequence
    wide = opg.attention_paged(q, kf, vf, bt, np.full(2, nb), np.array([int(lens[0]), int(lens[1])]), 1, lens)
    assert np.array_equal(base, wide)


@pytest.mark.parametrize("W", [1, 7, P, P + 9])
def test_window_is_attention_over_the_last_w_keys(W):
    kc, vc, bi, lens, q = _contiguous_case(5, T=2)
    q = np.random.default_rng(6).standard_normal((4, 4, 8))
    kp, vp, nb, perm = _pool_from_contiguous(kc, vc)
    bt = np.array([[f * nb + i for i in range(nb)] for f in bi])
    kf, vf = okv.bits_to_f64(kc, "f16"), okv.bits_to_f64(vc, "f16")
    got = opg.attention_paged(q, okv.bits_to_f64(kp, "f16"), okv.bits_to_f64(vp, "f16"), bt, np.full(2, nb),
                              np.full(2, W), 2, lens)
    for s, slot in enumerate(bi):
        for j in range(2):
            pos = int(lens[s]) - 2 + j
            lo = max(0, pos - W + 1)
            for h in range(4):
                keys = kf[slot, h // 2, lo:pos + 1]
                score = keys @ q[s * 2 + j, h] / np.sqrt(8.0)
                e = np.exp(score - score.max())
                want = (e / e.sum()) @ vf[slot, h // 2, lo:pos + 1]
                assert np.allclose(got[s * 2 + j, h], want, rtol=1e-12, atol=1e-12)


def test_ring_after_wraparound_holds_the_newest_keys():
    """Write positions 0..L-1 of one sequence through a 2-page ring in order;
    the ring then holds the newest 2P keys, and windowed attention over it
    equals attention over the logical last W keys."""
    rng = np.random.default_rng(7)
    hkv, hq, D = 2, 4, 8
    L = 5 * P + 17
    n_pages = 6
    bt = np.array([[4, 1]])
    n_blocks = np.array([2])
    W = P + 40
    k_all = rng.standard_normal((L, hkv, D)).astype(np.float32)
    v_all = rng.standard_normal((L, hkv, D)).astype(np.float32)
    kp = np.zeros((n_pages, hkv, P, D), np.uint16)
    vp = np.zeros_like(kp)
    model = {}
    for p in range(L):   # one token per step, as decode writes them
        kp, vp = opg.scatter(kp, vp, bt, n_blocks, np.array([W]), 1, np.array([p]), k_all[p:p + 1], v_all[p:p + 1],
                             "bf16")
        model[opg.locate(p, bt[0], 2, W)] = p
    for (page, row), p in model.items():
        assert np.array_equal(kp[page, :, row], okv.convert(k_all[p], "bf16"))
    assert min(model.values()) == L - 2 * P
    untouched = np.ones(n_pages, bool)
    untouched[[4, 1]] = False
    assert not kp[untouched].any()
    q = rng.standard_normal((1, hq, D))
    got = opg.attention_paged(q, okv.bits_to_f64(kp, "bf16"), okv.bits_to_f64(vp, "bf16"), bt, n_blocks,
                              np.array([W]), 1, np.array([L]))
    kl = okv.bits_to_f64(okv.convert(k_all[L - W:], "bf16"), "bf16")
    vl = okv.bits_to_f64(okv.convert(v_all[L - W:], "bf16"), "bf16")
    for h in range(hq):
        score = kl[:, h // 2] @ q[0, h] / np.sqrt(float(D))
        e = np.exp(score - score.max())
        assert np.allclose(got[0, h], (e / e.sum()) @ vl[:, h // 2], rtol=1e-12, atol=1e-12)


def test_scatter_writes_only_the_named_rows():
    rng = np.random.default_rng(8)
    kp = rng.integers(0, 65535, (5, 2, P, 4)).astype(np.uint16)
    vp = rng.integers(0, 65535, (5, 2, P, 4)).astype(np.uint16)
    bt = np.array([[3, 0, 4], [1, 2, 0]])
    n_blocks = np.array([3, 2])
    window = np.array([0, 130])
    pos = np.array([P + 5, P + 6, 2 * P + 1, 2 * P + 2])   # seq 1 wraps: block 2 -> ring index 0
    k = rng.standard_normal((4, 2, 4)).astype(np.float32)
    v = rng.standard_normal((4, 2, 4)).astype(np.float32)
    nk, nv = opg.scatter(kp, vp, bt, n_blocks, window, 2, pos, k, v, "f16")
    written = {(0, P + 5 - P), (0, P + 6 - P), (1, 1), (1, 2)}
    assert opg.locate(2 * P + 1, bt[1], 2, 130) == (1, 1)
    for page in range(5):
        for row in range(P):
            if (page, row) not in written:
                assert np.array_equal(nk[page, :, row], kp[page, :, row])
                assert np.array_equal(nv[page, :, row], vp[page, :, row])
    assert np.array_equal(nk[0, :, 5], okv.convert(k[0], "f16"))
    assert np.array_equal(nk[1, :, 2], okv.convert(k[3], "f16"))


def test_geometry_checks():
    opg.check_geometry(np.zeros((1, 2)), np.array([2]), np.array([200]), 57, np.array([1000]))
    with pytest.raises(ValueError):
        opg.check_geometry(np.zeros((1, 2)), np.array([2]), np.array([200]), 58, np.array([1000]))
    with pytest.raises(ValueError):
        opg.check_geometry(np.zeros((1, 2)), np.array([2]), np.array([0]), 1, np.array([2 * P + 1]))
    with pytest.raises(ValueError):
        opg.locate(2 * P, np.array([0, 1]), 2, 0)
