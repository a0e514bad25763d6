"""Pins for the oracle's cache-dtype converters and the batch_index scatter."""
import numpy as np
import pytest

from oracle import kv


def _probe_values():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(50000).astype(np.float32) * (np.float32(10.0) ** rng.integers(-9, 6, 50000)).astype(np.float32)
    edge = np.array([0.0, -0.0, 1.0, -1.0, 65504, 65519.996, 65520, 1e9, -1e9, 6.0e-8, 2.9802322e-8,
                     2.9802326e-8, 5.9604645e-8, 6.1035156e-5, 6.1028e-5, np.inf, -np.inf,
                     1.0009765625, 1.00048828125, 1.00146484375, 3.0e-39], np.float32)
    # every float32 that lies exactly half way between two fp16 neighbours near 1.0
    halves = (np.float32(1.0) + np.arange(1, 200, 2, dtype=np.float32) * np.float32(2.0 ** -11)).astype(np.float32)
    return np.concatenate([x, edge, halves, -halves])


def test_f16_matches_library_cast():
    x = _probe_values()
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(kv.f32_to_f16_bits(x), want)


def _bf16_brute(x: np.float32) -> int:
    """Nearest bfloat16 by enumerating the two candidates around x."""
    u = int(np.array([x], np.float32).view(np.uint32)[0])
    lo = u >> 16
    cands = [lo, lo + 1]
    vals = [float(np.array([c << 16], np.uint32).view(np.float32)[0]) for c in cands]
    dist = [abs(v - float(x)) for v in vals]
    if dist[0] < dist[1]:
        return cands[0]
    if dist[1] < dist[0]:
        return cands[1]
    return cands[0] if cands[0] % 2 == 0 else cands[1]


def test_bf16_matches_brute_force_nearest_even():
    x = _probe_values()
    x = x[np.isfinite(x) & (np.abs(x) < 3e38)][:20000]
    got = kv.f32_to_bf16_bits(x)
    for xi, gi in zip(x, got):
        assert int(gi) == _bf16_brute(xi), xi


def test_bf16_matches_library_cast():
    torch = pytest.importorskip("torch")
    x = _probe_values()
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kv.f32_to_bf16_bits(x), want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_scatter_writes_only_named_rows(dtype):
    rng = np.random.default_rng(1)
    F, H, C, D, T = 6, 3, 40, 8, 2
    kc = rng.integers(0, 2 ** 16, (F, H, C, D)).astype(np.uint16)
    vc = rng.integers(0, 2 ** 16, (F, H, C, D)).astype(np.uint16)
    bi = np.array([4, 1, 5])
    seq_lens = np.array([10, 2, 40])
    pos = np.array([L - T + j for L in seq_lens for j in range(T)])
    k = rng.standard_normal((6, H, D)).astype(np.float32)
    v = rng.standard_normal((6, H, D)).astype(np.float32)
    kc2, vc2 = kv.kv_scatter(kc, vc, bi, T, pos, k, v, dtype)
    written = np.zeros((F, H, C, D), bool)
    for s, slot in enumerate(bi):
        for j in range(T):
            t = s * T + j
            written[slot, :, pos[t], :] = True
            assert np.array_equal(kc2[slot, :, pos[t]], kv.convert(k[t], dtype))
            assert np.array_equal(vc2[slot, :, pos[t]], kv.convert(v[t], dtype))
    assert np.array_equal(kc2[~written], kc[~written])
    assert np.array_equal(vc2[~written], vc[~written])
    assert written.sum() == 3 * T * H * D
