"""Pins for the oracle's q8_0 codec (CPU only).

Each check rests on something other than the codec's own code: hand-derived
bytes (tests/golden/q8_0_hand_blocks.txt), exact rational arithmetic, and
the codec's error bound.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import q8_0

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_0_hand_blocks.txt")


def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, vals, hexes = (p.strip() for p in line.split("|"))
        x = np.array([float(v) for v in vals.split()], dtype=np.float32)
        b = np.array([int(h, 16) for h in hexes.split()], dtype=np.uint8)
        assert x.size == 32 and b.size == 34, name
        cases.append((name, x, b))
    return cases


@pytest.mark.parametrize("name,x,expected", _golden_cases(), ids=lambda v: v if isinstance(v, str) else "")
def test_hand_blocks(name, x, expected):
    got = q8_0.quantize_rows(x[None, :])[0]
    assert got.tobytes() == expected.tobytes(), (name, got, expected)


def test_unpack_roundtrip_layout():
    x = np.random.default_rng(0).standard_normal((3, 96)).astype(np.float32)
    b = q8_0.quantize_rows(x)
    assert b.shape == (3, 3 * 34)
    q, d = q8_0.unpack(b)
    assert q.shape == (3, 3, 32) and d.shape == (3, 3)
    # scale is the first two bytes of each block, codes follow
    assert np.array_equal(b.reshape(3, 3, 34)[..., 2:].view(np.int8), q)
    assert np.array_equal(b.reshape(3, 3, 34)[..., :2].copy().view("<f2")[..., 0], d)


def _exact_nearest_away(x32, d32):
    """Nearest integer to the exact rational x/d (ties away from zero)."""
    r = Fraction(float(x32)) / Fraction(float(d32))
    a = abs(r)
    n = int(a)
    if a - n >= Fraction(1, 2):
        n += 1
    return n if r >= 0 else -n, r


def test_codes_are_nearest_to_float32_scale():
    """q_k must be the integer nearest x_k / d with d the *float32* scale
    (not its fp16 rounding); checked in exact rational arithmetic, skipping
    quotients within float32 rounding of a half-integer tie."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 32)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float32)
    b = q8_0.quantize_rows(x)
    q, _ = q8_0.unpack(b)
    q = q.reshape(64, 32)
    amax = np.max(np.abs(x), axis=1)
    d32 = (amax / np.float32(127)).astype(np.float32)
    checked = 0
    for r in range(64):
        for k in range(32):
            n, exact = _exact_nearest_away(x[r, k], d32[r])
            frac = abs(exact) - int(abs(exact))
            if abs(frac - Fraction(1, 2)) < Fraction(1, 2 ** 16):
                continue
            assert q[r, k] == max(-127, min(127, n)), (r, k)
            checked += 1
    assert checked > 2000


def test_fp16_scale_differs_from_float32_scale_sometimes():
    """Guards the reading that codes use the float32 scale: on random data
    the fp16-rounded scale would give different codes for some values."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((512, 32)).astype(np.float32)
    q, d16 = q8_0.unpack(q8_0.quantize_rows(x))
    d16 = d16.astype(np.float32).reshape(512, 1)
    alt = np.clip(np.sign(x / d16) * np.floor(np.abs(x / d16) + 0.5), -127, 127)
    assert np.any(alt != q.reshape(512, 32))


def test_roundtrip_error_bound():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((200, 256)) * 0.02).astype(np.float32)
    b = q8_0.quantize_rows(x)
    deq = q8_0.dequantize_rows(b).reshape(200, 8, 32)
    xb = x.reshape(200, 8, 32).astype(np.float64)
    amax = np.max(np.abs(xb), axis=-1, keepdims=True)
    d32 = amax / 127.0
    _, d16 = q8_0.unpack(b)
    d16 = d16.astype(np.float64)[..., None]
    # |x - d16*q| <= |x - d32*q| + |d32 - d16| * |q|  <=  d32/2 (1+2^-20) + 127 |d32 - d16|
    bound = d32 / 2 * (1 + 2.0 ** -20) + 127 * np.abs(d32 - d16)
    assert np.all(np.abs(xb - deq) <= bound)


def test_extremes_hit_127():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, 32)).astype(np.float32)
    q, _ = q8_0.unpack(q8_0.quantize_rows(x))
    q = q.reshape(50, 32)
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(q[np.arange(50), am]) == 127)
    assert np.all(np.abs(q) <= 127)


def test_rejects_ragged_rows():
    with pytest.raises(ValueError):
        q8_0.quantize_rows(np.zeros((2, 33), np.float32))
