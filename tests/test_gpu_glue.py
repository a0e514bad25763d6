"""GPU parity of the decode step's fused glue kernels, each called on its own
through the C ABI and fed the oracle's own float32 inputs: RMS-norm + q8_0,
SiLU(gate) * up + q8_0, the q8_0 embedding gather, the per-head RMS norm +
RoPE, the fused (norm +) RoPE + KV write, and the attention with q8_0 output.

Quantised outputs are compared with ``assert_q8_close`` (codes within one
step, scales within one fp16 ulp, and only at rounding boundaries); float
outputs with the op tolerances; the embedding and every cache byte the step
must not touch are bit-exact.
"""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import glue as oglue
from oracle import kv as okv
from oracle import q8_0 as oq
from oracle import rope as orope
from oracle import step as ostep
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import ROPE_ATOL, ROPE_RTOL, assert_close, assert_q8_close, to_dev, to_host

pytestmark = pytest.mark.gpu

DT = {"f16": 0, "bf16": 1}


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _bits_dev(bits):
    import torch
    return to_dev(bits.view(np.int16)).view(torch.int16)


@pytest.mark.parametrize("n_tok,hidden", [(8, 768), (3, 5120), (16, 8192), (1, 256), (33, 1024)])
def test_rmsnorm_q8_0(cuda_device, n_tok, hidden):
    x = synth.normal_rows(3, synth.stream_id(synth.STREAM_X, 20), n_tok, hidden, 1.0)
    x *= np.float32(0.05) * (1 + np.arange(n_tok, dtype=np.float32))[:, None]   # rows of different scale
    w = (0.5 + synth.normal_rows(3, synth.stream_id(synth.STREAM_X, 21), 1, hidden, 0.1)[0]).astype(np.float32)
    got = to_host(_dsb().rmsnorm_q8_0(to_dev(x), to_dev(w), 1e-6))
    want = ostep.quant(oglue.rmsnorm(x, w, 1e-6))
    assert_q8_close(got, want, f"rmsnorm {n_tok}x{hidden}")


def test_rmsnorm_q8_0_zero_row(cuda_device):
    """An all-zero row normalises to zeros: scale 0, codes 0, exactly."""
    x = np.zeros((2, 512), np.float32)
    x[1] = 1.0
    got = to_host(_dsb().rmsnorm_q8_0(to_dev(x), to_dev(np.ones(512, np.float32)), 1e-6))
    assert got.tobytes() == ostep.quant(oglue.rmsnorm(x, np.ones(512), 1e-6)).tobytes()
    assert not got[0].any()


@pytest.mark.parametrize("n_tok,ffn", [(8, 3072), (3, 17408), (1, 32), (17, 768)])
def test_silu_mul_q8_0(cuda_device, n_tok, ffn):
    gu = synth.normal_rows(4, synth.stream_id(synth.STREAM_X, 22), n_tok, 2 * ffn, 2.0)
    got = to_host(_dsb().silu_mul_q8_0(to_dev(gu)))
    want = ostep.quant(oglue.silu_mul(gu[:, :ffn], gu[:, ffn:]))
    assert_q8_close(got, want, f"silu_mul {n_tok}x{ffn}")


def test_embed_q8_0_exact(cuda_device):
    d = _dsb()
    vocab, hidden = 1000, 768
    table32 = synth.normal_rows(5, synth.stream_id(synth.STREAM_EMBED, 3), vocab, hidden, 0.02)
    table = oq.quantize_rows(table32)
    toks = np.array([0, vocab - 1, 17, 17, 500, 999, 3], np.int32)
    ws = d.Workspace(len(toks), 1, 64, 16)
    got = to_host(d.embed_q8_0(to_dev(table), vocab, hidden, toks, ws))
    want = oglue.embedding(table, toks)
    assert np.array_equal(got.astype(np.float64), want)   # fp16 scale x int8 code is exact in float32
    with pytest.raises(d.DsbError) as e:
        d.embed_q8_0(to_dev(table), vocab, hidden, np.array([vocab], np.int32), ws)
    assert e.value.status == 1


def _head_weights(seed, d, n):
    return [(1.0 + synth.normal_rows(seed, synth.stream_id(synth.STREAM_W, 60 + i), 1, d, 0.1)[0]).astype(np.float32)
            for i in range(n)]


YARNS = {"": None, "y4": (4.0, 4096), "y16": (16.0, 2048), "y8": (8.0, 32768)}


@pytest.mark.parametrize("hq,hkv,d,norms,yarn", [(12, 12, 64, "qk", ""), (40, 8, 128, "qk", ""), (8, 2, 128, "k", ""),
                                                 (4, 0, 256, "q", ""), (5, 3, 1024, "qk", ""), (3, 1, 2, "qk", ""),
                                                 (6, 2, 64, "", ""), (40, 8, 128, "qk", "y4"), (8, 2, 64, "", "y16"),
                                                 (5, 3, 1024, "q", "y8")])
def test_head_rmsnorm_rope(cuda_device, hq, hkv, d, norms, yarn):
    """Per-head RMS norm then RoPE (plain or YaRN) against the oracle; heads of
    very different scales (1e-3 .. 1e3) and an all-zero head, which stays
    zero."""
    dd = _dsb()
    oy = orope.Yarn(*YARNS[yarn]) if YARNS[yarn] else None
    dy = dd.Yarn(*YARNS[yarn]) if YARNS[yarn] else None
    n_tok = 7
    pos = np.array([0, 1, 5, 127, 2047, 4095, 100000], np.int32)
    q = synth.normal(8, synth.stream_id(synth.STREAM_Q, 32), (n_tok, hq, d))
    q *= np.float32(10.0) ** np.linspace(-3, 3, hq, dtype=np.float32)[None, :, None]
    q[2, 0] = 0.0
    k = synth.normal(8, synth.stream_id(synth.STREAM_K, 32), (n_tok, hkv, d)) * np.float32(30.0) if hkv else None
    qw, kw = _head_weights(8, d, 2)
    qn = qw if "q" in norms else None
    kn = kw if "k" in norms and hkv else None
    eps = 1e-6
    qd = to_dev(q)
    kd = to_dev(k) if hkv else None
    dd.head_rmsnorm_rope(qd, kd, pos, 10000.0, None if qn is None else to_dev(qn), None if kn is None else to_dev(kn),
                         eps, dd.Workspace(n_tok, hq, d, 16), yarn=dy)
    got_q = to_host(qd)
    _assert_heads_close(got_q, orope.head_rmsnorm_rope(q, pos, 10000.0, qn, eps, oy), "q")
    if qn is not None:
        assert not got_q[2, 0].any()
    if hkv:
        _assert_heads_close(to_host(kd), orope.head_rmsnorm_rope(k, pos, 10000.0, kn, eps, oy), "k")


def _assert_heads_close(got, ref, what):
    """Every element within ROPE_RTOL of its head vector's RMS (heads here span
    six orders of magnitude; an all-zero head must come back exactly zero)."""
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= ROPE_RTOL * rms), (what, float(np.max(err / np.maximum(rms, 1e-300))))


@pytest.mark.parametrize("hq,hkv,d,dtype,T,norm,yarn", [(12, 12, 64, "f16", 1, False, ""),
                                                        (40, 8, 128, "bf16", 1, False, ""),
                                                        (12, 12, 64, "f16", 8, False, ""),
                                                        (8, 2, 128, "bf16", 4, False, ""),
                                                        (40, 8, 128, "bf16", 2, True, ""),
                                                        (12, 12, 64, "f16", 3, True, ""),
                                                        (40, 8, 128, "bf16", 2, True, "y4"),
                                                        (12, 12, 64, "f16", 1, False, "y16")])
def test_rope_kv_write(cuda_device, hq, hkv, d, dtype, T, norm, yarn):
    dd = _dsb()
    oy = orope.Yarn(*YARNS[yarn]) if YARNS[yarn] else None
    dy = dd.Yarn(*YARNS[yarn]) if YARNS[yarn] else None
    F, C = 6, 4096
    bi = np.array([5, 0, 2], np.int32)
    lens = np.array([C, T, 1777], np.int32)
    pos = ostep.positions(lens, T).astype(np.int32)
    n_tok = len(pos)
    cols = (hq + 2 * hkv) * d
    qkv = synth.normal_rows(6, synth.stream_id(synth.STREAM_Q, 30), n_tok, cols, 1.5)
    kc = synth.cache_bits(6, synth.stream_id(synth.STREAM_KCACHE, 30), (F, hkv, C, d), dtype)
    vc = synth.cache_bits(6, synth.stream_id(synth.STREAM_VCACHE, 30), (F, hkv, C, d), dtype)
    kd, vd = _bits_dev(kc), _bits_dev(vc)
    kv = dd.kv_cache(kd, vd, DT[dtype])
    qkv_d = to_dev(qkv)
    qw, kw = _head_weights(6, d, 2) if norm else (None, None)
    eps = 1e-6
    dd.rope_kv_write(qkv_d, hq, kv, bi, T, pos, 10000.0, dd.Workspace(n_tok, hq, d, C),
                     q_norm=None if qw is None else to_dev(qw), k_norm=None if kw is None else to_dev(kw), eps=eps,
                     yarn=dy)
    got = to_host(qkv_d)
    q = qkv[:, :hq * d].reshape(n_tok, hq, d)
    k = qkv[:, hq * d:(hq + hkv) * d].reshape(n_tok, hkv, d)
    v = qkv[:, (hq + hkv) * d:].reshape(n_tok, hkv, d)
    assert_close(got[:, :hq * d].reshape(n_tok, hq, d), orope.head_rmsnorm_rope(q, pos, 10000.0, qw, eps, oy),
                 ROPE_RTOL, ROPE_ATOL, "q")
    assert np.array_equal(got[:, hq * d:].view(np.uint32), qkv[:, hq * d:].view(np.uint32))  # k, v untouched
    kr = orope.head_rmsnorm_rope(k, pos, 10000.0, kw, eps, oy).astype(np.float32)
    want_k, want_v = okv.kv_scatter(kc, vc, bi, T, pos, kr, v, dtype)
    gk, gv = to_host(kd).view(np.uint16), to_host(vd).view(np.uint16)
    assert np.array_equal(gv, want_v)                       # v: one conversion of the same float32 values
    # k: the float32 rotation may land on the other side of a cache-dtype
    # rounding boundary than the rounded float64 one -- one ulp, rarely
    diff = np.abs(gk.astype(np.int32) - want_k.astype(np.int32))
    assert diff.max() <= 1
    assert np.sum(diff != 0) <= max(2, n_tok * hkv * d // 100)
    written = np.zeros(kc.shape[:3], bool)
    for s, slot in enumerate(bi):
        written[slot, :, lens[s] - T:lens[s]] = True
    assert np.array_equal(gk[~written], kc[~written])         # nothing else is written


@pytest.mark.parametrize("hq,hkv,d,dtype,T,C", [(12, 12, 64, "f16", 1, 2048), (40, 8, 128, "bf16", 1, 4096),
                                                (12, 12, 64, "f16", 8, 2048), (8, 2, 128, "bf16", 4, 300)])
def test_attention_q8_0(cuda_device, hq, hkv, d, dtype, T, C):
    dd = _dsb()
    F = 5
    bi = np.array([3, 0, 4], np.int32)
    lens = np.array([C, T, C // 2 + 7], np.int32)
    n_tok = len(bi) * T
    q = synth.normal(7, synth.stream_id(synth.STREAM_Q, 31), (n_tok, hq, d))
    kc = synth.cache_bits(7, synth.stream_id(synth.STREAM_KCACHE, 31), (F, hkv, C, d), dtype)
    vc = synth.cache_bits(7, synth.stream_id(synth.STREAM_VCACHE, 31), (F, hkv, C, d), dtype)
    kv = dd.kv_cache(_bits_dev(kc), _bits_dev(vc), DT[dtype])
    got = to_host(dd.attention_decode_multi_q8_0(to_dev(q), kv, bi, T, lens, dd.Workspace(n_tok, hq, d, C)))
    a = oatt.attention_decode_multi(q, okv.bits_to_f64(kc, dtype), okv.bits_to_f64(vc, dtype), bi, T, lens)
    assert_q8_close(got, ostep.quant(a.reshape(n_tok, hq * d)), f"attention q8 {hq}/{hkv} D={d} T={T}")
