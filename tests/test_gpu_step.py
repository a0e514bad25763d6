"""GPU parity of the whole batched decode step (C ABI dsb_decode_step and the
captured step graph) against the oracle's composed step.

Each side builds its own model from the same seeded float32 draws: the GPU
quantises its weights with its own kernel, the oracle with its own codec, and
the bytes must agree.  No page prints an end-to-end value: the oracle's
composition is pinned by closed forms (CPU tests) and every stage of the GPU
step is held to its own operation's tolerance in test_gpu_step_chain.py; this
end-to-end comparison, with the tolerance derived in the comment above
``STEP_TOL_RMS``, catches the wiring of the step and its captured graph.  The
per-sequence and per-slot invariants are exact.
"""
import numpy as np
import pytest

from oracle import q8_0 as oq
from oracle import step as ostep
from tests import _shapes
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

# Logit tolerances, relative to the RMS of the reference logits.  Both sides
# round every activation to q8_0 codes before each matmul; where the float32
# GPU value and the float64 oracle value fall on opposite sides of a rounding
# boundary, that code differs by one step d = max|x|/127 (about 3/127 of the
# block's RMS).  A relative activation difference eps flips a fraction
# p ~ eps * |x| / d ~ 42 eps of the codes, and the flips move the next matmul's
# output by sigma_w * d * sqrt(p K), i.e. by ~ (3/127) sqrt(42 eps) ~
# 0.15 sqrt(eps) of its RMS.  The step re-quantises five times per layer, and
# the map eps -> 0.15 sqrt(eps) has its fixed point at eps ~ 2.3e-2: one early
# flip (a float32 rounding of the RMS-norm sum crossing an fp16 scale boundary
# suffices) grows toward a few percent of the RMS, while a wiring error (head,
# position, slot, scale) is O(1).  So the logits are held to an RMS error of
# 3e-2 and a maximum error of 0.2 of the logit RMS, and the stages before the
# first attention are pinned tightly below (new layer-0 cache rows), with each
# fused kernel's own parity checked in its op test.
STEP_TOL_RMS = 3e-2
STEP_TOL_MAX = 2e-1
# The new layer-0 K/V rows pass one q8_0 rounding (of the RMS-normed
# embedding) before they are written: within one ulp of the cache dtype plus
# 1e-3 of their RMS.
CACHE_ULP = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}

DT = {"f16": 0, "bf16": 1}


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _build(ms, seed=0):
    import torch
    d = _dsb()
    wf = _shapes.weight_f32(seed, ms)
    dev, orc = {}, {}
    for k in ("wqkv", "wo", "wgu", "wdown"):
        dev[k] = [d.quantize_q8_0(to_dev(m)) for m in wf[k]]
        orc[k] = [oq.quantize_rows(m) for m in wf[k]]
        for a, b in zip(dev[k], orc[k]):
            assert to_host(a).tobytes() == b.tobytes()
    for k in ("head", "embed"):
        dev[k] = d.quantize_q8_0(to_dev(wf[k]))
        orc[k] = oq.quantize_rows(wf[k])
        assert to_host(dev[k]).tobytes() == orc[k].tobytes()
    for k in ("attn_norm", "ffn_norm", "q_norm", "k_norm"):
        if k not in wf:
            continue
        dev[k] = [to_dev(v) for v in wf[k]]
        orc[k] = wf[k]
    dev["final_norm"], orc["final_norm"] = to_dev(wf["final_norm"]), wf["final_norm"]
    kc = [_shapes.cache_bits(seed, ms, l, "k") for l in range(ms.n_layers)]
    vc = [_shapes.cache_bits(seed, ms, l, "v") for l in range(ms.n_layers)]
    kd = [to_dev(c.view(np.int16)) for c in kc]
    vd = [to_dev(c.view(np.int16)) for c in vc]
    yarn = d.Yarn(ms.yarn_factor, ms.yarn_orig_ctx) if ms.yarn_factor > 1 else None
    model = d.DecodeModel(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, dev,
                          kd, vd, DT[ms.cache_dtype], ms.eps, ms.theta, yarn)
    return model, orc, kc, vc


def _oshape(ms):
    from oracle import rope as orope
    yarn = orope.Yarn(ms.yarn_factor, ms.yarn_orig_ctx) if ms.yarn_factor > 1 else None
    return ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, ms.eps,
                       ms.theta, yarn)


def _rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref * ref)))


def _rms_err(got, ref):
    return float(np.sqrt(np.mean((got - ref) ** 2)) / np.sqrt(np.mean(ref * ref)))


# Speculative decode on the llama shapes: T = K + 1 in {8, 32} puts n_tok = 24,
# 32 and 64 tokens through every matmul (beyond the narrow kernel's 16: up to
# 32 as 16-token narrow launches, the last one ragged at 24; 64 on the tensor
# cores), and the causal mask inside the drafts through the attention.
# The qk-norm shapes add the per-head q / k RMS norm before the rope; the
# yarn shapes use the YaRN RoPE with sequences past the original context.
CASES = [(_shapes.TINY, 3, 1), (_shapes.TINY, 2, 4), (_shapes.TINY_BF16, 5, 1), (_shapes.TINY_QKN, 3, 1),
         (_shapes.TINY_QKN, 2, 4), (_shapes.TINY_BF16_QKN, 4, 2), (_shapes.TINY_YARN, 3, 2),
         (_shapes.TINY_BF16_YARN, 4, 1), (_shapes.LLAMA68M, 4, 1),
         (_shapes.LLAMA68M, 1, 1), (_shapes.LLAMA68M, 3, 8), (_shapes.LLAMA68M, 4, 8), (_shapes.LLAMA68M, 2, 32),
         pytest.param(_shapes.QWEN3_14B_LAYER, 3, 1, marks=pytest.mark.slow),
         pytest.param(_shapes.QWEN3_14B_LAYER, 16, 1, marks=pytest.mark.slow)]


@pytest.mark.parametrize("ms,b,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_step_matches_oracle(cuda_device, ms, b, T):
    model, orc, kc, vc = _build(ms)
    bi, lens, toks = _shapes.step_meta(1, ms, b, T)
    ws = model.workspace(b * T)
    logits = to_host(model.step(toks, bi, T, lens, ws))
    ref, nk, nv = ostep.decode_step(_oshape(ms), orc, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    err_rms, err_max = _rms_err(logits, ref), _rel_err(logits, ref)
    assert err_rms < STEP_TOL_RMS, f"rms |g - r| / rms(r) = {err_rms:.3e}"
    assert err_max < STEP_TOL_MAX, f"max |g - r| / rms(r) = {err_max:.3e}"
    # the argmax of every row agrees unless the top two logits are within tolerance
    top = np.argmax(ref, axis=1)
    for t in range(len(toks)):
        g = int(np.argmax(logits[t]))
        assert g == top[t] or abs(ref[t, g] - ref[t, top[t]]) < STEP_TOL_MAX * np.sqrt(np.mean(ref * ref))
    # the new layer-0 rows, before any attention: tight
    from oracle import kv as okv
    for cache_g, cache_o in ((model.k_caches[0], nk[0]), (model.v_caches[0], nv[0])):
        bits = to_host(cache_g).view(np.uint16)
        g_rows = np.stack([bits[slot][:, lens[s] - T + j] for s, slot in enumerate(bi) for j in range(T)])
        o_rows = np.stack([cache_o[slot][:, lens[s] - T + j] for s, slot in enumerate(bi) for j in range(T)])
        gv, ov = okv.bits_to_f64(g_rows, ms.cache_dtype), okv.bits_to_f64(o_rows, ms.cache_dtype)
        bound = CACHE_ULP[ms.cache_dtype] * np.abs(ov) + 1e-3 * np.sqrt(np.mean(ov * ov))
        assert np.all(np.abs(gv - ov) <= bound), float(np.max(np.abs(gv - ov) / bound))
    # slots the step does not name are untouched; named slots change only at pos
    untouched = np.ones(ms.full_batch_size, bool)
    untouched[bi] = False
    for l in range(ms.n_layers):
        kg = to_host(model.k_caches[l]).view(np.uint16)
        vg = to_host(model.v_caches[l]).view(np.uint16)
        assert np.array_equal(kg[untouched], kc[l][untouched])
        assert np.array_equal(vg[untouched], vc[l][untouched])
        for s, slot in enumerate(bi):
            keep = np.ones(ms.ctx, bool)
            keep[lens[s] - T:lens[s]] = False
            assert np.array_equal(kg[slot][:, keep], kc[l][slot][:, keep])


# (8 sequences x 2 tokens: the batched step's matmuls take 16 tokens on the
# tensor-core block dots and its glue the wide launch shapes, each single
# sequence's 2 tokens the dp4a block dots and the narrow shapes)
@pytest.mark.parametrize("ms,b,T", [(_shapes.TINY, 3, 2), (_shapes.LLAMA68M, 4, 1), (_shapes.LLAMA68M, 8, 2)],
                         ids=["tiny", "llama", "llama-16-tokens"])
def test_batched_step_rows_equal_single_sequence_steps(cuda_device, ms, b, T):
    model, _, _, _ = _build(ms)
    bi, lens, toks = _shapes.step_meta(2, ms, b, T)
    ws = model.workspace(b * T)
    batched = to_host(model.step(toks, bi, T, lens, ws))
    for s in range(b):
        one = to_host(model.step(toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1], ws))
        assert np.array_equal(one.view(np.uint32), batched[s * T:(s + 1) * T].view(np.uint32)), s


def test_graph_replay_mapped_metadata_equals_eager_step(cuda_device):
    """A step whose metadata exceeds the parameter block (n_tok = 2048): the
    graph reads it from mapped pinned memory; replays with new metadata equal
    the eager step bitwise."""
    import torch
    ms = _shapes.TINY_WIDE
    b, T = 64, 32
    model, _, _, _ = _build(ms)
    ws = model.workspace(b * T)
    logits = torch.empty((b * T, ms.vocab), dtype=torch.float32, device="cuda")
    g = model.graph(b, T, logits, ws)
    for seed in (6, 7):
        bi, lens, toks = _shapes.step_meta(seed, ms, b, T)
        eager = to_host(model.step(toks, bi, T, lens, ws))
        replay = to_host(g.launch(toks, bi, lens))
        assert np.array_equal(eager.view(np.uint32), replay.view(np.uint32)), seed
    g.close()
    _dsb().device_error()


@pytest.mark.parametrize("b,T", [(4, 1), (2, 32)])
def test_graph_replay_equals_eager_step(cuda_device, b, T):
    import torch
    ms = _shapes.LLAMA68M
    model, _, _, _ = _build(ms)
    ws = model.workspace(b * T)
    logits = torch.empty((b * T, ms.vocab), dtype=torch.float32, device="cuda")
    g = model.graph(b, T, logits, ws)
    for seed in (3, 4, 5):   # new tokens, slots and lengths on every replay
        bi, lens, toks = _shapes.step_meta(seed, ms, b, T)
        eager = to_host(model.step(toks, bi, T, lens, ws))
        replay = to_host(g.launch(toks, bi, lens))
        assert np.array_equal(eager.view(np.uint32), replay.view(np.uint32)), seed
    g.close()
    _dsb().device_error()
