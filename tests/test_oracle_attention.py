"""Pins for the oracle's multi-sequence GQA decode attention (CPU only)."""
import math

import numpy as np

from oracle import attention


def _case(seed=0, F=5, hkv=2, group=2, C=32, D=8):
    rng = np.random.default_rng(seed)
    kc = rng.standard_normal((F, hkv, C, D))
    vc = rng.standard_normal((F, hkv, C, D))
    return rng, kc, vc, hkv * group


def test_weights_sum_to_one():
    rng = np.random.default_rng(0)
    for L in [1, 2, 17, 300]:
        p = attention.weights(rng.standard_normal(64), rng.standard_normal((L, 64)) * 3)
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p >= 0)


def test_one_key_returns_v_exactly():
    rng, kc, vc, hq = _case()
    q = rng.standard_normal((1, hq, 8))
    out = attention.attention_decode_multi(q, kc, vc, [3], 1, [1])
    for h in range(hq):
        assert np.array_equal(out[0, h], vc[3, h // 2, 0])


def test_equal_keys_give_mean_v():
    rng, kc, vc, hq = _case(1)
    kc[2, :, :, :] = kc[2, :, :1, :]
    q = rng.standard_normal((1, hq, 8))
    out = attention.attention_decode_multi(q, kc, vc, [2], 1, [20])
    for h in range(hq):
        assert np.allclose(out[0, h], vc[2, h // 2, :20].mean(axis=0), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_v():
    rng, kc, vc, hq = _case(2)
    q = np.zeros((1, hq, 8))
    out = attention.attention_decode_multi(q, kc, vc, [0], 1, [13])
    for h in range(hq):
        assert np.allclose(out[0, h], vc[0, h // 2, :13].mean(axis=0), rtol=0, atol=1e-12)


def test_brute_force_hand_expanded():
    rng, kc, vc, hq = _case(3, D=4)
    q = rng.standard_normal((2, hq, 4))
    out = attention.attention_decode_multi(q, kc, vc, [4, 1], 1, [3, 2])
    for s, (slot, L) in enumerate([(4, 3), (1, 2)]):
        for h in range(hq):
            g = h // 2
            sc = [sum(q[s, h, d] * kc[slot, g, j, d] for d in range(4)) / 2.0 for j in range(L)]
            m = max(sc)
            e = [math.exp(v - m) for v in sc]
            z = sum(e)
            want = [sum(e[j] / z * vc[slot, g, j, d] for j in range(L)) for d in range(4)]
            assert np.allclose(out[s, h], want, rtol=0, atol=1e-13)


def test_scale_is_one_over_sqrt_d():
    # two keys: k0 = 0, k1 = a e0; q = b e0 -> scores 0 and a b / sqrt(D)
    D, a, b = 16, 1.5, 2.0
    kc = np.zeros((1, 1, 4, D))
    vc = np.zeros((1, 1, 4, D))
    kc[0, 0, 1, 0] = a
    vc[0, 0, 0, 0] = 1.0
    vc[0, 0, 1, 1] = 1.0
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = b
    out = attention.attention_decode_multi(q, kc, vc, [0], 1, [2])
    p1 = 1.0 / (1.0 + math.exp(-a * b / 4.0))
    assert abs(out[0, 0, 1] - p1) < 1e-15 and abs(out[0, 0, 0] - (1 - p1)) < 1e-15


def test_batched_row_equals_single_run():
    rng, kc, vc, hq = _case(4)
    q = rng.standard_normal((3, hq, 8))
    bi, lens = [2, 0, 4], [7, 32, 1]
    out = attention.attention_decode_multi(q, kc, vc, bi, 1, lens)
    for s in range(3):
        single = attention.attention_decode_multi(q[s:s + 1], kc, vc, [bi[s]], 1, [lens[s]])
        assert np.array_equal(out[s], single[0])


def test_draft_tokens_are_causal():
    rng, kc, vc, hq = _case(5)
    T = 4
    q = rng.standard_normal((2 * T, hq, 8))
    bi, lens = [1, 3], [9, 30]
    out = attention.attention_decode_multi(q, kc, vc, bi, T, lens)
    for s in range(2):
        for j in range(T):
            t = s * T + j
            one = attention.attention_decode_multi(q[t:t + 1], kc, vc, [bi[s]], 1, [lens[s] - T + j + 1])
            assert np.array_equal(out[t], one[0])


def test_gqa_groups_are_contiguous():
    rng, kc, vc, hq = _case(6, hkv=2, group=3)
    q = rng.standard_normal((1, 6, 8))
    out = attention.attention_decode_multi(q, kc, vc, [0], 1, [10])
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, 1] = 1e3
    vc2[:, 1] = -1e3
    out2 = attention.attention_decode_multi(q, kc2, vc2, [0], 1, [10])
    assert np.array_equal(out[0, :3], out2[0, :3])       # heads 0..2 read kv head 0
    assert not np.allclose(out[0, 3:], out2[0, 3:])      # heads 3..5 read kv head 1
