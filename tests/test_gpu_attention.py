"""GPU parity of the pos-vector RoPE, the batch_index KV write and the
multi-sequence GQA decode attention, through the C ABI."""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import kv as okv
from oracle import rope as orope
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import ATTN_ATOL, ATTN_RTOL, ROPE_ATOL, ROPE_RTOL, assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu

DT = {"f16": 0, "bf16": 1}


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _ws(max_tokens, hq, d, ctx):
    return _dsb().Workspace(max_tokens, hq, d, ctx)


def _cache(seed, F, hkv, C, D, dtype, which):
    kind = synth.STREAM_KCACHE if which == "k" else synth.STREAM_VCACHE
    return synth.cache_bits(seed, synth.stream_id(kind, 0), (F, hkv, C, D), dtype)


def _bits_dev(bits):
    import torch
    return to_dev(bits.view(np.int16)).view(torch.int16)


# ---------------------------------------------------------------- RoPE
@pytest.mark.parametrize("n_tok,hq,hkv,d", [(2, 8, 2, 64), (16, 40, 8, 128), (33, 12, 12, 64), (3, 128, 128, 128)])
def test_rope_matches_oracle(cuda_device, n_tok, hq, hkv, d):
    q = synth.normal(1, synth.stream_id(synth.STREAM_Q, 0), (n_tok, hq, d))
    k = synth.normal(1, synth.stream_id(synth.STREAM_K, 0), (n_tok, hkv, d))
    pos = synth.uniform_int(1, synth.stream_id(synth.STREAM_META, 9), 0, 65535, n_tok)
    pos[0] = 0
    ws = _ws(n_tok, hq, d, 16)
    qd, kd = to_dev(q), to_dev(k)
    _dsb().rope_posvec(qd, kd, pos, 10000.0, ws)
    qg, kg = to_host(qd), to_host(kd)
    assert_close(qg, orope.rope_posvec(q, pos, 10000.0), ROPE_RTOL, ROPE_ATOL, "rope q")
    assert_close(kg, orope.rope_posvec(k, pos, 10000.0), ROPE_RTOL, ROPE_ATOL, "rope k")
    assert np.array_equal(qg[0], q[0]) and np.array_equal(kg[0], k[0])  # position 0 is the identity
    # row t of the batched call equals an n_tok = 1 call
    for t in (1, n_tok - 1):
        q1, k1 = to_dev(q[t:t + 1]), to_dev(k[t:t + 1])
        _dsb().rope_posvec(q1, k1, pos[t:t + 1], 10000.0, ws)
        assert np.array_equal(to_host(q1)[0].view(np.uint32), qg[t].view(np.uint32))
        assert np.array_equal(to_host(k1)[0].view(np.uint32), kg[t].view(np.uint32))


# ---------------------------------------------------------------- KV write
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T", [1, 4])
def test_kv_scatter_bit_exact(cuda_device, dtype, T):
    F, hkv, C, D = 6, 3, 200, 64
    kc = _cache(2, F, hkv, C, D, dtype, "k")
    vc = _cache(2, F, hkv, C, D, dtype, "v")
    bi = np.array([4, 1, 5], np.int32)
    lens = np.array([10, T, 200], np.int32)
    pos = np.array([L - T + j for L in lens for j in range(T)], np.int32)
    n_tok = len(pos)
    k = synth.normal(2, synth.stream_id(synth.STREAM_K, 1), (n_tok, hkv, D)) * np.float32(300.0)
    v = synth.normal(2, synth.stream_id(synth.STREAM_V, 1), (n_tok, hkv, D))
    kd, vd = _bits_dev(kc), _bits_dev(vc)
    kv = _dsb().kv_cache(kd, vd, DT[dtype])
    _dsb().kv_scatter(kv, bi, T, pos, to_dev(k), to_dev(v), _ws(n_tok, hkv, D, C))
    want_k, want_v = okv.kv_scatter(kc, vc, bi, T, pos, k, v, dtype)
    assert np.array_equal(to_host(kd).view(np.uint16), want_k)
    assert np.array_equal(to_host(vd).view(np.uint16), want_v)


# ---------------------------------------------------------------- attention
def _attn_case(seed, F, hq, hkv, C, D, dtype, bi, lens, T):
    kc = _cache(seed, F, hkv, C, D, dtype, "k")
    vc = _cache(seed, F, hkv, C, D, dtype, "v")
    n_tok = len(bi) * T
    q = synth.normal(seed, synth.stream_id(synth.STREAM_Q, 2), (n_tok, hq, D))
    kv = _dsb().kv_cache(_bits_dev(kc), _bits_dev(vc), DT[dtype])
    return kc, vc, q, kv


def _attn_oracle(q, kc, vc, dtype, bi, T, lens, heads=None):
    return oatt.attention_decode_multi(q, okv.bits_to_f64(kc, dtype), okv.bits_to_f64(vc, dtype), bi, T, lens, heads)


ATTN_CASES = [
    # F, hq, hkv, C, D, dtype, batch_index, seq_lens, T
    (4, 8, 2, 256, 64, "f16", [2, 0], [200, 37], 1),                       # tiny step shapes
    (8, 12, 12, 2048, 64, "f16", [5, 1, 7, 0], [128, 2048, 1000, 129], 1),  # llama-68m shapes
    (16, 40, 8, 4096, 128, "bf16", [3, 9, 15], [1, 4096, 2500], 1),         # Qwen3-14B shapes (GQA 5:1)
    (128, 12, 12, 2048, 64, "f16", [100, 3], [300, 2048], 8),               # speculative drafts (K=7)
    (8, 4, 4, 700, 128, "f16", [1], [700], 16),                             # ragged ctx, T=16
    (5, 8, 2, 384, 128, "bf16", [0, 1, 2, 3, 4], [1, 127, 128, 129, 384], 1),  # chunk edges
    # 64-key copy-box edges; slot 5 is the last of the cache tensor and C = 200
    # is not a multiple of 64, so its last box reaches past the tensor's end
    (6, 8, 2, 200, 64, "f16", [5, 0, 3, 1, 2, 4], [200, 63, 64, 65, 191, 192], 1),
    (6, 10, 2, 200, 128, "bf16", [5, 2], [200, 65], 2),                    # G*T = 10: two query row groups
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"F{c[0]}_hq{c[1]}_hkv{c[2]}_C{c[3]}_D{c[4]}_{c[5]}_T{c[8]}")
def test_attention_matches_oracle(cuda_device, case):
    F, hq, hkv, C, D, dtype, bi, lens, T = case
    bi, lens = np.array(bi, np.int32), np.array(lens, np.int32)
    kc, vc, q, kv = _attn_case(3, F, hq, hkv, C, D, dtype, bi, lens, T)
    ws = _ws(len(bi) * T, hq, D, C)
    out = to_host(_dsb().attention_decode_multi(to_dev(q), kv, bi, T, lens, ws))
    assert_close(out, _attn_oracle(q, kc, vc, dtype, bi, T, lens), ATTN_RTOL, ATTN_ATOL, "attention")
    _dsb().device_error()


@pytest.mark.parametrize("case", ATTN_CASES[1:4], ids=["llama", "qwen", "spec"])
def test_attention_batched_rows_equal_single_runs(cuda_device, case):
    F, hq, hkv, C, D, dtype, bi, lens, T = case
    bi, lens = np.array(bi, np.int32), np.array(lens, np.int32)
    kc, vc, q, kv = _attn_case(4, F, hq, hkv, C, D, dtype, bi, lens, T)
    ws = _ws(len(bi) * T, hq, D, C)
    out = to_host(_dsb().attention_decode_multi(to_dev(q), kv, bi, T, lens, ws))
    for s in range(len(bi)):
        one = to_host(_dsb().attention_decode_multi(to_dev(q[s * T:(s + 1) * T]), kv, bi[s:s + 1], T, lens[s:s + 1], ws))
        assert np.array_equal(one.view(np.uint32), out[s * T:(s + 1) * T].view(np.uint32)), s


def test_attention_one_key_returns_v_exactly(cuda_device):
    F, hq, hkv, C, D = 3, 4, 2, 64, 128
    kc, vc, q, kv = _attn_case(5, F, hq, hkv, C, D, "f16", np.array([1]), np.array([1]), 1)
    out = to_host(_dsb().attention_decode_multi(to_dev(q), kv, np.array([1], np.int32), 1, np.array([1], np.int32),
                                                _ws(1, hq, D, C)))
    v = okv.bits_to_f64(vc, "f16")
    for h in range(hq):
        assert np.array_equal(out[0, h].astype(np.float64), v[1, h // 2, 0])


def test_attention_draft_tokens_causal(cuda_device):
    F, hq, hkv, C, D, T = 4, 4, 4, 512, 64, 4
    bi, lens = np.array([3, 0], np.int32), np.array([300, 129], np.int32)
    kc, vc, q, kv = _attn_case(6, F, hq, hkv, C, D, "f16", bi, lens, T)
    ws = _ws(len(bi) * T, hq, D, C)
    out = to_host(_dsb().attention_decode_multi(to_dev(q), kv, bi, T, lens, ws))
    for s in range(2):
        for j in range(T):
            t = s * T + j
            one = to_host(_dsb().attention_decode_multi(to_dev(q[t:t + 1]), kv, bi[s:s + 1], 1,
                                                        np.array([lens[s] - T + j + 1], np.int32), ws))
            assert_close(one[0], out[t], 1e-6, 1e-7, f"draft token {j}")


def test_untouched_slots_after_scatter_and_attention(cuda_device):
    F, hkv, C, D, T = 8, 2, 128, 64, 2
    kc = _cache(7, F, hkv, C, D, "f16", "k")
    vc = _cache(7, F, hkv, C, D, "f16", "v")
    kd, vd = _bits_dev(kc), _bits_dev(vc)
    kv = _dsb().kv_cache(kd, vd, 0)
    bi, lens = np.array([6, 2], np.int32), np.array([50, 128], np.int32)
    pos = np.array([L - T + j for L in lens for j in range(T)], np.int32)
    k = synth.normal(7, synth.stream_id(synth.STREAM_K, 3), (4, hkv, D))
    ws = _ws(4, 4, D, C)
    _dsb().kv_scatter(kv, bi, T, pos, to_dev(k), to_dev(k), ws)
    q = synth.normal(7, synth.stream_id(synth.STREAM_Q, 3), (4, 4, D))
    _dsb().attention_decode_multi(to_dev(q), kv, bi, T, lens, ws)
    kh = to_host(kd).view(np.uint16)
    vh = to_host(vd).view(np.uint16)
    others = [s for s in range(F) if s not in bi]
    assert np.array_equal(kh[others], kc[others]) and np.array_equal(vh[others], vc[others])
    for s, slot in enumerate(bi):
        mask = np.ones(C, bool)
        mask[pos[s * T:(s + 1) * T]] = False
        assert np.array_equal(kh[slot][:, mask], kc[slot][:, mask])


@pytest.mark.slow
@pytest.mark.parametrize("C", [32768, 65536])
def test_long_context_sampled_heads(cuda_device, C):
    """MHA-shaped long-context attention (128 heads, D 128, fp16 cache of
    full_batch_size 8) past the ~31k rows where the ds4 page's multi-sequence
    kernel stops.  Every head of every sequence's slot holds its own rows: head
    h is synthetic block h mod 4 rotated by 37 h rows, so no two heads of a
    slot agree and a head or slot read from the wrong place changes the
    output.  Five heads (neighbours included) are checked against the oracle
    on the same rows."""
    import torch
    F, H, D = 8, 128, 128
    b, P = 4, 4
    bi = synth.distinct_slots(8, 1, b, F)
    lens = synth.uniform_int(8, 2, 16384, C, b)
    lens[0] = C
    pools = {}
    for name, stream in (("k", synth.STREAM_KCACHE), ("v", synth.STREAM_VCACHE)):
        pools[name] = [synth.cache_bits_rows(8, synth.stream_id(stream, 300 + p), (C, D), "f16", 0, C) for p in range(P)]

    def rows(name, h):
        return np.roll(pools[name][h % P], 37 * h, axis=0)

    kd = torch.zeros((F, H, C, D), dtype=torch.float16, device="cuda")
    vd = torch.zeros((F, H, C, D), dtype=torch.float16, device="cuda")
    for name, dst in (("k", kd), ("v", vd)):
        dev_pools = [to_dev(x.view(np.int16)).view(torch.float16) for x in pools[name]]
        for s in range(b):
            for h in range(H):
                dst[int(bi[s]), h, :lens[s]] = torch.roll(dev_pools[h % P], 37 * h, dims=0)[:lens[s]]
        del dev_pools
    heads = [0, 1, 64, 77, 127]
    kc_small = np.zeros((b, len(heads), C, D), np.uint16)   # oracle copy, one slot per sequence
    vc_small = np.zeros((b, len(heads), C, D), np.uint16)
    for s in range(b):
        for hi, h in enumerate(heads):
            kc_small[s, hi, :lens[s]] = rows("k", h)[:lens[s]]
            vc_small[s, hi, :lens[s]] = rows("v", h)[:lens[s]]
    q = synth.normal(8, synth.stream_id(synth.STREAM_Q, 4), (b, H, D))
    kv = _dsb().kv_cache(kd, vd, 0)
    out = to_host(_dsb().attention_decode_multi(to_dev(q), kv, bi, 1, lens, _ws(b, H, D, C)))
    q_small = q[:, heads, :]
    want = oatt.attention_decode_multi(q_small, okv.bits_to_f64(kc_small, "f16"), okv.bits_to_f64(vc_small, "f16"),
                                       np.arange(b), 1, lens)
    assert_close(out[:, heads, :], want, ATTN_RTOL, ATTN_ATOL, f"long context C={C}")
