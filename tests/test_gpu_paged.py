"""GPU parity of the paged / ring KV geometry (dsb_kv_scatter_paged,
dsb_attention_decode_paged) against the oracle, through the C ABI.

The KV write is bit-exact (a conversion of the same float32 values) and
touches no other page row; the attention is held to the attention tolerance.
A linear paged view of a contiguous cache is bitwise equal to the contiguous
kernel: the pages coincide with its 128-key chunks, so the arithmetic is the
same."""
import numpy as np
import pytest

from oracle import kv as okv
from oracle import paged as opg
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import ATTN_ATOL, ATTN_RTOL, assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu

DT = {"f16": 0, "bf16": 1}
P = 128


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _bits_dev(bits):
    import torch
    return to_dev(bits.view(np.int16)).view(torch.int16)


def _pools(seed, n_pages, hkv, D, dtype):
    shape = (n_pages, hkv, P, D)
    return (synth.cache_bits(seed, synth.stream_id(synth.STREAM_KCACHE, 40), shape, dtype),
            synth.cache_bits(seed, synth.stream_id(synth.STREAM_VCACHE, 40), shape, dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_paged_scatter_bit_exact(cuda_device, dtype):
    d = _dsb()
    hkv, D, n_pages, T = 3, 64, 9, 2
    kp, vp = _pools(1, n_pages, hkv, D, dtype)
    bt = np.array([[7, 2, 5, 0], [1, 8, 0, 0], [3, 4, 6, 0]], np.int32)
    n_blocks = np.array([3, 2, 3], np.int32)
    window = np.array([0, 200, 300], np.int32)
    lens = np.array([3 * P - 1, 5 * P + 3, 2 * P + 70], np.int32)   # seq 1 and 2 wrap around their rings
    pos = np.array([L - T + j for L in lens for j in range(T)], np.int32)
    k = synth.normal(1, synth.stream_id(synth.STREAM_K, 40), (len(pos), hkv, D)) * np.float32(50.0)
    v = synth.normal(1, synth.stream_id(synth.STREAM_V, 40), (len(pos), hkv, D))
    kd, vd = _bits_dev(kp), _bits_dev(vp)
    kv = d.kv_pages(kd, vd, DT[dtype])
    d.kv_scatter_paged(kv, bt, n_blocks, window, T, pos, to_dev(k), to_dev(v), d.Workspace(len(pos), hkv, D, 16))
    want_k, want_v = opg.scatter(kp, vp, bt, n_blocks, window, T, pos, k, v, dtype)
    assert np.array_equal(to_host(kd).view(np.uint16), want_k)
    assert np.array_equal(to_host(vd).view(np.uint16), want_v)


def _attn_case(seed, hq, hkv, D, dtype, T, lens, window, n_blocks, max_blocks, n_pages):
    rng = np.random.default_rng(seed)
    kp, vp = _pools(seed, n_pages, hkv, D, dtype)
    perm = rng.permutation(n_pages).astype(np.int32)
    bt = np.zeros((len(lens), max_blocks), np.int32)
    used = 0
    for s, nb in enumerate(n_blocks):
        bt[s, :nb] = perm[used:used + nb]
        used += nb
    q = synth.normal(seed, synth.stream_id(synth.STREAM_Q, 41), (len(lens) * T, hq, D))
    return kp, vp, bt, q


@pytest.mark.parametrize("hq,hkv,D,dtype,T", [(12, 12, 64, "f16", 1), (40, 8, 128, "bf16", 1), (8, 2, 64, "bf16", 4),
                                              (4, 4, 128, "f16", 8)])
def test_paged_attention_matches_oracle(cuda_device, hq, hkv, D, dtype, T):
    d = _dsb()
    lens = np.array([5 * P + 17, 300, 2 * P, 900], np.int32)
    window = np.array([0, 0, 150, 200], np.int32)
    n_blocks = np.array([6, 3, 2, 3], np.int32)      # seq 2, 3: rings of 2 and 3 pages (the 900-key one wrapped)
    kp, vp, bt, q = _attn_case(2, hq, hkv, D, dtype, T, lens, window, n_blocks, 6, 20)
    opg.check_geometry(bt, n_blocks, window, T, lens)
    kv = d.kv_pages(_bits_dev(kp), _bits_dev(vp), DT[dtype])
    got = to_host(d.attention_decode_paged(to_dev(q), kv, bt, n_blocks, window, T, lens,
                                           d.Workspace(len(lens) * T, hq, D, 6 * P)))
    want = opg.attention_paged(q, okv.bits_to_f64(kp, dtype), okv.bits_to_f64(vp, dtype), bt, n_blocks, window, T,
                               lens)
    assert_close(got, want, ATTN_RTOL, ATTN_ATOL, f"paged {hq}/{hkv} D={D} T={T}")


@pytest.mark.parametrize("T", [1, 3])
def test_linear_pages_bitwise_equal_contiguous(cuda_device, T):
    """The pages of a contiguous cache, permuted, read through a linear block
    table give the contiguous kernel's bits."""
    import torch
    d = _dsb()
    F, hkv, hq, C, D = 4, 2, 8, 4 * P, 64
    kc = synth.cache_bits(3, synth.stream_id(synth.STREAM_KCACHE, 42), (F, hkv, C, D), "f16")
    vc = synth.cache_bits(3, synth.stream_id(synth.STREAM_VCACHE, 42), (F, hkv, C, D), "f16")
    bi = np.array([3, 0, 2], np.int32)
    lens = np.array([C, 2 * P + 5, 77], np.int32)
    q = to_dev(synth.normal(3, synth.stream_id(synth.STREAM_Q, 42), (len(bi) * T, hq, D)))
    ws = d.Workspace(len(bi) * T, hq, D, C)
    kcd, vcd = _bits_dev(kc), _bits_dev(vc)
    contiguous = to_host(d.attention_decode_multi(q, d.kv_cache(kcd, vcd, 0), bi, T, lens, ws))
    nb = C // P
    perm = np.random.default_rng(4).permutation(F * nb).astype(np.int32)
    kp = torch.empty((F * nb, hkv, P, D), dtype=torch.int16, device="cuda")
    vp = torch.empty_like(kp)
    src_k = kcd.view(F, hkv, nb, P, D).permute(0, 2, 1, 3, 4).reshape(F * nb, hkv, P, D)
    src_v = vcd.view(F, hkv, nb, P, D).permute(0, 2, 1, 3, 4).reshape(F * nb, hkv, P, D)
    kp[torch.from_numpy(perm).long().cuda()] = src_k
    vp[torch.from_numpy(perm).long().cuda()] = src_v
    bt = np.stack([perm[f * nb:(f + 1) * nb] for f in bi])
    paged = to_host(d.attention_decode_paged(q, d.kv_pages(kp, vp, 0), bt, np.full(3, nb, np.int32),
                                             np.zeros(3, np.int32), T, lens, ws))
    assert np.array_equal(paged.view(np.uint32), contiguous.view(np.uint32))


def test_paged_rejects_bad_geometry(cuda_device):
    import torch
    d = _dsb()
    kp = torch.zeros((4, 2, P, 64), dtype=torch.int16, device="cuda")
    kv = d.kv_pages(kp, kp.clone(), 0)
    ws = d.Workspace(4, 2, 64, 4 * P)
    q = torch.zeros((2, 2, 64), device="cuda")
    with pytest.raises(d.DsbError):   # a ring of 1 page cannot hold window 128 + T - 1 = 129 keys
        d.attention_decode_paged(q, kv, np.array([[0, 0]]), np.array([1]), np.array([128]), 2, np.array([300]), ws)
    with pytest.raises(d.DsbError):   # linear table of 2 pages for 300 keys
        d.attention_decode_paged(q[:1], kv, np.array([[0, 1]]), np.array([2]), np.array([0]), 1, np.array([300]), ws)
    with pytest.raises(d.DsbError):   # page index out of range
        d.attention_decode_paged(q[:1], kv, np.array([[0, 4]]), np.array([2]), np.array([0]), 1, np.array([200]), ws)
    kv_in = torch.zeros((2, 2, 64), device="cuda")
    with pytest.raises(d.DsbError):   # two tokens of one call on the same row (ring of 1 page, positions 128 apart)
        d.kv_scatter_paged(kv, np.array([[1]]), np.array([1]), np.array([1]), 2, np.array([5, 133]), kv_in, kv_in, ws)
    assert not kp.any()   # nothing was written
