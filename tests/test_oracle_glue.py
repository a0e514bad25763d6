"""Pins for the oracle's step glue (CPU only)."""
import math

import numpy as np

from oracle import glue, q8_0


def test_rmsnorm_constant_vector():
    x = np.full((1, 64), 3.0)
    w = np.linspace(0.5, 1.5, 64)
    y = glue.rmsnorm(x, w, eps=1e-6)
    assert np.allclose(y[0], w * 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15, atol=0)


def test_rmsnorm_scale_invariant_without_eps():
    x = np.random.default_rng(0).standard_normal((3, 48))
    w = np.ones(48)
    assert np.allclose(glue.rmsnorm(7.5 * x, w, 0.0), glue.rmsnorm(x, w, 0.0), rtol=1e-14, atol=0)
    y = glue.rmsnorm(x, w, 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)


def test_silu_known_values():
    assert glue.silu_mul(np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert abs(glue.silu_mul(np.array([1.0]), np.array([1.0]))[0] - 0.7310585786300049) < 1e-15
    assert abs(glue.silu_mul(np.array([-1.0]), np.array([2.0]))[0] - 2 * -0.2689414213699951) < 1e-15
    assert abs(glue.silu_mul(np.array([40.0]), np.array([0.5]))[0] - 20.0) < 1e-12


def test_residual_add():
    a = np.arange(5.0)
    assert np.array_equal(glue.residual_add(a, a), 2 * a)


def test_embedding_is_dequantised_row():
    rng = np.random.default_rng(1)
    table = q8_0.quantize_rows(rng.standard_normal((10, 64)).astype(np.float32))
    e = glue.embedding(table, [3, 3, 9])
    q, d = q8_0.unpack(table[3])
    want = (q.astype(np.float64) * d.astype(np.float64)[:, None]).reshape(64)
    assert np.array_equal(e[0], want) and np.array_equal(e[1], want)


def test_silu_odd_part_is_the_identity():
    """x*sigmoid(x) - (-x)*sigmoid(-x) = x*(sigmoid(x) + sigmoid(-x)) = x; a
    sign slip in the exponent breaks it."""
    x = np.linspace(-30.0, 30.0, 121)
    one = np.ones_like(x)
    assert np.allclose(glue.silu_mul(x, one) - glue.silu_mul(-x, one), x, rtol=1e-14, atol=1e-14)


def test_rmsnorm_rows_are_independent():
    x = np.random.default_rng(2).standard_normal((4, 32)) * np.array([[1e-3], [1.0], [1e3], [0.0]])
    w = np.linspace(0.1, 2.0, 32)
    full = glue.rmsnorm(x, w, 1e-6)
    for t in range(4):
        assert np.array_equal(full[t], glue.rmsnorm(x[t:t + 1], w, 1e-6)[0])
    assert not full[3].any()   # an all-zero row stays zero
