"""Pins for the oracle's pos-vector RoPE (CPU only)."""
import math
import os

import numpy as np

from oracle import rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_d4.txt")


def test_hand_values_d4():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        p, xs, ys = (s.strip() for s in line.split("|"))
        x = np.array([float(v) for v in xs.split()]).reshape(1, 1, 4)
        want = np.array([float(v) for v in ys.split()])
        got = rope.rope_posvec(x, np.array([int(p)]), 10000.0)[0, 0]
        assert np.allclose(got, want, rtol=0, atol=1e-15), (line, got)


def test_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((3, 4, 64))
    assert np.array_equal(rope.rope_posvec(x, np.zeros(3, int), 10000.0), x)


def test_pair_norms_preserved():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 128))
    pos = rng.integers(0, 65536, 5)
    y = rope.rope_posvec(x, pos, 10000.0)
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12, atol=0)


def test_relative_position_invariance():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    dots = []
    for p in [0, 17, 1000, 40000]:
        qr = rope.rope_posvec(q, np.array([p + 5]), 10000.0)
        kr = rope.rope_posvec(k, np.array([p]), 10000.0)
        dots.append(float(np.sum(qr * kr)))
    assert np.allclose(dots, dots[0], rtol=0, atol=1e-10)


def test_d2_is_textbook_rotation():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 1, 2))
    pos = np.array([0, 1, 2, 5, 100, 12345])
    y = rope.rope_posvec(x, pos, 10000.0)
    for t, p in enumerate(pos):
        c, s = math.cos(p), math.sin(p)
        m = np.array([[c, -s], [s, c]])
        assert np.allclose(y[t, 0], m @ x[t, 0], rtol=0, atol=1e-12)


def test_each_row_uses_its_own_position():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 2, 16))
    pos = np.array([9, 0, 300, 9])
    y = rope.rope_posvec(x, pos, 10000.0)
    for t in range(4):
        assert np.array_equal(y[t], rope.rope_posvec(x[t:t + 1], pos[t:t + 1], 10000.0)[0])


def test_head_norm_rope_golden():
    """Hand-derived values (tests/golden/head_norm_rope.txt) pin the order:
    norm, then weight, then rotation."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "head_norm_rope.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        pos, eps, w, x, want = (p.strip() for p in line.split("|"))
        xv = np.array([float(v) for v in x.split()])[None, None, :]
        wv = np.array([float(v) for v in w.split()])
        got = rope.head_rmsnorm_rope(xv, np.array([int(pos)]), 10000.0, wv, float(eps))[0, 0]
        assert np.allclose(got, [float(v) for v in want.split()], rtol=0, atol=1e-14)


def test_head_norm_rope_unit_weights_give_unit_mean_square():
    """With unit weights the normed head has mean square ms / (ms + eps), and
    the rotation keeps it."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 4, 64)) * 7.0
    eps = 1e-6
    y = rope.head_rmsnorm_rope(x, np.array([0, 5, 90000]), 10000.0, np.ones(64), eps)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-12)
    assert np.array_equal(rope.head_rmsnorm_rope(x, np.array([1, 2, 3]), 10000.0, None, eps),
                          rope.rope_posvec(x, np.array([1, 2, 3]), 10000.0))


# ---------------------------------------------------------------- YaRN variant
YARN = rope.Yarn(factor=4.0, orig_ctx=4096)


def test_yarn_golden_frequencies():
    """Hand-derived frequencies, correction range and magnitude factor
    (tests/golden/yarn_d64.txt)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "yarn_d64.txt")
    vals = {}
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = (p.strip() for p in line.split("|"))
            vals[k] = float(v)
    assert rope.yarn_correction_range(64, 10000.0, YARN) == (vals["low"], vals["high"])
    assert abs(rope.yarn_mscale(YARN) - vals["mscale"]) < 1e-15
    f = rope.frequencies(64, 10000.0, YARN)
    for i in (0, 10, 16, 20, 23, 31):
        assert abs(f[i] - vals[f"f{i}"]) <= 4e-15 * vals[f"f{i}"], i


def test_yarn_correction_range_brackets_rotation_counts():
    """low is the last pair that turns at least beta_fast times over the
    original context, high the first that turns at most beta_slow times
    (rotation counts r_i = L f_i / (2 pi) computed here directly)."""
    for d, theta, L in ((64, 10000.0, 4096), (128, 1e6, 32768), (128, 10000.0, 2048), (256, 5e5, 8192)):
        y = rope.Yarn(8.0, L)
        low, high = rope.yarn_correction_range(d, theta, y)
        r = [L * theta ** (-2.0 * i / d) / (2 * math.pi) for i in range(d // 2 + 1)]
        assert r[low] >= y.beta_fast > r[low + 1], (d, theta, L, low)
        assert r[high - 1] > y.beta_slow >= r[high], (d, theta, L, high)


def test_yarn_fast_pairs_extrapolate_slow_pairs_interpolate():
    """Pairs below the ramp rotate as the plain RoPE (scaled by m); pairs
    above it, at position s*p, as the plain RoPE at position p (position
    interpolation)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 2, 64))
    p = np.array([0, 3, 1000, 7777])
    m = rope.yarn_mscale(YARN)
    low, high = rope.yarn_correction_range(64, 10000.0, YARN)
    y = rope.rope_posvec(x, p, 10000.0, YARN)
    plain = rope.rope_posvec(x, p, 10000.0) * m
    for i in list(range(low + 1)):
        for j in (i, i + 32):
            assert np.allclose(y[..., j], plain[..., j], rtol=0, atol=1e-12)
    y4 = rope.rope_posvec(x, 4 * p, 10000.0, YARN)
    for i in range(high, 32):
        for j in (i, i + 32):
            assert np.allclose(y4[..., j], plain[..., j], rtol=0, atol=1e-12)


def test_yarn_scale_one_is_plain_and_norms_scale_by_m():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 2, 128))
    pos = np.array([1, 500, 60000])
    assert np.allclose(rope.rope_posvec(x, pos, 1e6, rope.Yarn(1.0, 4096)), rope.rope_posvec(x, pos, 1e6),
                       rtol=0, atol=1e-12)
    y = rope.rope_posvec(x, pos, 1e6, rope.Yarn(16.0, 4096))
    m = 0.1 * math.log(16.0) + 1.0
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n_out, n_in * m * m, rtol=1e-12, atol=0)


def test_yarn_keeps_relative_position_invariance():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    dots = [float(np.sum(rope.rope_posvec(q, np.array([p + 9]), 10000.0, YARN) *
                         rope.rope_posvec(k, np.array([p]), 10000.0, YARN))) for p in (0, 11, 5000, 90000)]
    assert np.allclose(dots, dots[0], rtol=0, atol=1e-10)
