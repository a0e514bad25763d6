"""Pins for the oracle's narrow-batch q8_0 matmul (CPU only)."""
import numpy as np
import pytest

from oracle import matmul, q8_0


def _blocks(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Pack int8 codes [R, nb, 32] and float16 scales [R, nb] into q8_0 bytes
    directly (independent of the quantiser)."""
    r, nb, _ = codes.shape
    out = np.empty((r, nb, 34), np.uint8)
    out[..., :2] = scales.astype("<f2").reshape(r, nb, 1).view(np.uint8)
    out[..., 2:] = codes.astype(np.int8).view(np.uint8)
    return out.reshape(r, nb * 34)


def test_all_ones_closed_form():
    nb = 7
    w = _blocks(np.ones((5, nb, 32), np.int8), np.ones((5, nb), np.float16))
    x = _blocks(np.ones((3, nb, 32), np.int8), np.ones((3, nb), np.float16))
    y = matmul.matmul_q8_0(w, x)
    assert y.shape == (3, 5)
    assert np.all(y == 32 * nb)


def test_one_hot_selects_single_activation():
    rng = np.random.default_rng(0)
    nb, n_tok = 4, 3
    xc = rng.integers(-127, 128, (n_tok, nb, 32)).astype(np.int8)
    xs = rng.uniform(0.001, 0.1, (n_tok, nb)).astype(np.float16)
    x = _blocks(xc, xs)
    codes = np.zeros((1, nb, 32), np.int8)
    codes[0, 2, 17] = 1
    ws = np.full((1, nb), 0.5, np.float16)
    y = matmul.matmul_q8_0(_blocks(codes, ws), x)
    for t in range(n_tok):
        assert y[t, 0] == 0.5 * float(xs[t, 2]) * int(xc[t, 2, 17])


def test_brute_force_tiny():
    rng = np.random.default_rng(1)
    r, nb, n_tok = 3, 2, 2
    wc = rng.integers(-127, 128, (r, nb, 32))
    xc = rng.integers(-127, 128, (n_tok, nb, 32))
    ws = rng.uniform(1e-3, 1e-1, (r, nb)).astype(np.float16)
    xs = rng.uniform(1e-3, 1e-1, (n_tok, nb)).astype(np.float16)
    y = matmul.matmul_q8_0(_blocks(wc, ws), _blocks(xc, xs))
    for t in range(n_tok):
        for row in range(r):
            acc = 0.0
            for i in range(nb):
                s = 0
                for k in range(32):
                    s += int(wc[row, i, k]) * int(xc[t, i, k])
                acc += float(ws[row, i]) * float(xs[t, i]) * s
            assert abs(y[t, row] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_block_dots_extremes_fit_int32():
    nb = 2
    w = _blocks(np.full((1, nb, 32), 127, np.int8), np.ones((1, nb), np.float16))
    x = _blocks(np.full((2, nb, 32), -127, np.int8), np.ones((2, nb), np.float16))
    isum = matmul.block_dots(w, x)
    assert np.all(isum == -32 * 127 * 127)
    assert matmul.ISUM_BOUND == 516128 < 2 ** 31


def test_column_equals_single_run():
    rng = np.random.default_rng(2)
    w = q8_0.quantize_rows((rng.standard_normal((40, 256)) * 0.02).astype(np.float32))
    x = q8_0.quantize_rows(rng.standard_normal((16, 256)).astype(np.float32))
    y = matmul.matmul_q8_0(w, x)
    for j in range(16):
        assert np.array_equal(y[j], matmul.matmul_q8_0(w, x[j:j + 1])[0])


def test_row_subset_matches_full():
    rng = np.random.default_rng(4)
    w = q8_0.quantize_rows((rng.standard_normal((50, 128)) * 0.02).astype(np.float32))
    x = q8_0.quantize_rows(rng.standard_normal((3, 128)).astype(np.float32))
    rows = [0, 7, 49, 13]
    assert np.array_equal(matmul.matmul_q8_0(w, x, rows), matmul.matmul_q8_0(w, x)[:, rows])


def test_scaling_is_exact():
    rng = np.random.default_rng(6)
    wc = rng.integers(-127, 128, (4, 3, 32))
    ws = rng.uniform(1e-3, 1e-1, (4, 3)).astype(np.float16)
    xc = rng.integers(-127, 128, (2, 3, 32))
    xs = rng.uniform(1e-3, 1e-1, (2, 3)).astype(np.float16)
    y1 = matmul.matmul_q8_0(_blocks(wc, ws), _blocks(xc, xs))
    y2 = matmul.matmul_q8_0(_blocks(wc, ws), _blocks(xc, (xs * 2).astype(np.float16)))
    assert np.array_equal(2 * y1, y2)


def test_mismatched_widths_rejected():
    w = _blocks(np.ones((1, 2, 32), np.int8), np.ones((1, 2), np.float16))
    x = _blocks(np.ones((1, 3, 32), np.int8), np.ones((1, 3), np.float16))
    with pytest.raises(ValueError):
        matmul.matmul_q8_0(w, x)
