"""Stage-by-stage parity of the GPU decode step (teacher-forced).

dsb_decode_step_trace runs the step's own kernels and copies every stage's
result out.  Each stage is then held to its own operation's tolerance against
the oracle, fed the GPU's own inputs to that stage (the q8_0 codes the GPU
quantised, the h it carried, the caches it wrote), so no rounding difference
of an earlier stage can amplify into a later one:

  * q8_0 stages (RMSNorm, attention output, SiLU-gate): the flip-tolerant
    codec comparison (codes within one step, scales within one fp16 ulp, only
    at rounding boundaries);
  * matmuls and the residual adds in their epilogues: 1e-3 relative, 1e-4
    absolute;
  * the rope: 1e-5 of each head vector's RMS; the new cache rows: V bit-exact,
    K within one ulp of the cache dtype;
  * the embedding: exact.

A batched step must agree with its parts (ds4 PR #530, "Correctness").  The
traced step's logits are also bitwise those of the untraced step, so the
copies change nothing; the oracle's own composition is pinned by closed forms
in the CPU tests.
"""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import glue as oglue
from oracle import kv as okv
from oracle import matmul as omm
from oracle import q8_0 as oq
from oracle import rope as orope
from oracle import step as ostep
from tests import _shapes
from tests.gpu_util import MATMUL_ATOL, MATMUL_RTOL, ROPE_RTOL, assert_close, assert_q8_close, to_host
from tests.test_gpu_step import _build, _oshape

pytestmark = pytest.mark.gpu


def _q8(x):
    return oq.quantize_rows(np.asarray(x, dtype=np.float64).astype(np.float32))


def _heads_close(got, ref, what):
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= ROPE_RTOL * rms + 1e-30), (what, float(np.max(err / np.maximum(rms, 1e-300))))


CASES = [(_shapes.TINY, 3, 1), (_shapes.TINY, 2, 4), (_shapes.TINY_BF16_QKN, 4, 2), (_shapes.TINY_YARN, 3, 2),
         (_shapes.LLAMA68M, 4, 1), (_shapes.LLAMA68M, 8, 1), (_shapes.LLAMA68M, 2, 32),
         pytest.param(_shapes.QWEN3_14B_LAYER, 16, 1, marks=pytest.mark.slow)]


@pytest.mark.parametrize("ms,b,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_step_stages_match_oracle_ops(cuda_device, ms, b, T):
    model, orc, kc, vc = _build(ms)
    bi, lens, toks = _shapes.step_meta(4, ms, b, T)
    ws = model.workspace(b * T)
    logits_t, tr = model.step_trace(toks, bi, T, lens, ws)
    logits_t = to_host(logits_t)
    # the same step again without the copies (it rewrites the same cache rows)
    plain = to_host(model.step(toks, bi, T, lens, ws))
    assert np.array_equal(plain.view(np.uint32), logits_t.view(np.uint32)), "trace copies changed the step"

    osh = _oshape(ms)
    pos = ostep.positions(lens, T)
    n_tok = len(pos)
    hq, hkv, d, ffn = ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn
    g = lambda t: to_host(t)  # noqa: E731

    h_in = g(tr["h_embed"]).astype(np.float64)
    assert np.array_equal(h_in, oglue.embedding(orc["embed"], toks)), "embedding"
    for l, L in enumerate(tr["layers"]):
        tag = f"layer {l}"
        x_attn = g(L["x_attn"])
        assert_q8_close(x_attn, _q8(oglue.rmsnorm(h_in, orc["attn_norm"][l], ms.eps)), f"{tag} attn rmsnorm q8")
        qkv = g(L["qkv"])
        assert_close(qkv, omm.matmul_q8_0(orc["wqkv"][l], x_attn), MATMUL_RTOL, MATMUL_ATOL, f"{tag} qkv matmul")
        qkv_r = g(L["qkv_rope"])
        q_pre = qkv[:, :hq * d].reshape(n_tok, hq, d)
        k_pre = qkv[:, hq * d:(hq + hkv) * d].reshape(n_tok, hkv, d)
        v_pre = qkv[:, (hq + hkv) * d:].reshape(n_tok, hkv, d)
        qn = orc["q_norm"][l] if "q_norm" in orc else None
        kn = orc["k_norm"][l] if "k_norm" in orc else None
        q_rot = qkv_r[:, :hq * d].reshape(n_tok, hq, d)
        _heads_close(q_rot, orope.head_rmsnorm_rope(q_pre, pos, osh.theta, qn, ms.eps, osh.yarn), f"{tag} q rope")
        assert np.array_equal(qkv_r[:, hq * d:].view(np.uint32), qkv[:, hq * d:].view(np.uint32)), f"{tag} k|v kept"
        # the rows this step wrote into layer l's cache
        kg = to_host(model.k_caches[l]).view(np.uint16)
        vg = to_host(model.v_caches[l]).view(np.uint16)
        k_rot = orope.head_rmsnorm_rope(k_pre, pos, osh.theta, kn, ms.eps, osh.yarn).astype(np.float32)
        want_k, want_v = okv.kv_scatter(kc[l], vc[l], bi, T, pos, k_rot, v_pre, ms.cache_dtype)
        assert np.array_equal(vg, want_v), f"{tag} V rows"
        dk = np.abs(kg.astype(np.int32) - want_k.astype(np.int32))
        assert dk.max() <= 1 and np.sum(dk != 0) <= max(2, n_tok * hkv * d // 100), f"{tag} K rows"
        att = oatt.attention_decode_multi(q_rot.astype(np.float64), okv.bits_to_f64(kg, ms.cache_dtype),
                                          okv.bits_to_f64(vg, ms.cache_dtype), bi, T, lens)
        att_q8 = g(L["att_q8"])
        assert_q8_close(att_q8, _q8(att.reshape(n_tok, hq * d)), f"{tag} attention q8")
        h_attn = g(L["h_attn"])
        assert_close(h_attn, h_in + omm.matmul_q8_0(orc["wo"][l], att_q8), MATMUL_RTOL, MATMUL_ATOL,
                     f"{tag} O matmul + residual")
        x_ffn = g(L["x_ffn"])
        assert_q8_close(x_ffn, _q8(oglue.rmsnorm(h_attn, orc["ffn_norm"][l], ms.eps)), f"{tag} ffn rmsnorm q8")
        gu = g(L["gu"])
        assert_close(gu, omm.matmul_q8_0(orc["wgu"][l], x_ffn), MATMUL_RTOL, MATMUL_ATOL, f"{tag} gate|up matmul")
        act_q8 = g(L["act_q8"])
        assert_q8_close(act_q8, _q8(oglue.silu_mul(gu[:, :ffn], gu[:, ffn:])), f"{tag} silu*up q8")
        h_out = g(L["h_out"])
        assert_close(h_out, h_attn + omm.matmul_q8_0(orc["wdown"][l], act_q8), MATMUL_RTOL, MATMUL_ATOL,
                     f"{tag} down matmul + residual")
        h_in = h_out.astype(np.float64)
    x_final = g(tr["x_final"])
    assert_q8_close(x_final, _q8(oglue.rmsnorm(h_in, orc["final_norm"], ms.eps)), "final rmsnorm q8")
    assert_close(logits_t, omm.matmul_q8_0(orc["head"], x_final), MATMUL_RTOL, MATMUL_ATOL, "head matmul")
    _build.__globals__["_dsb"]().device_error()
