"""GPU parity of the whole batched decode step (C ABI dsb_decode_step and the
captured step graph) against the oracle's composed step.

Each side builds its own model from the same seeded float32 draws: the GPU
quantises its weights with its own kernel, the oracle with its own codec, and
the bytes must agree.  The composed step is "parity unpinned" as a whole (no
page prints an end-to-end value); its tolerance is derived in
``STEP_TOL``'s comment.  The per-sequence and per-slot invariants are exact.
"""
import numpy as np
import pytest

from oracle import q8_0 as oq
from oracle import step as ostep
from tests import _shapes
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

# Logit tolerance, relative to the RMS of the reference logits.  The GPU
# accumulates in float32 where the oracle uses float64, so the activations
# entering each re-quantisation differ by ~1e-6 relative; when that moves a
# value across a rounding boundary of its q8_0 code (rare), that one code
# changes by 1, i.e. by d = max|x|/127 of its block.  Through the following
# matmul such a flip perturbs an output by ~|w| * d, about 1e-3 of the output
# RMS, and a step has 4 re-quantisations per layer plus the head's.  2e-2 of
# the logit RMS bounds a handful of flips per row with margin; errors from
# wrong wiring (head mapping, positions, slots) are O(1) of the RMS.
STEP_TOL = 2e-2

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
    for k in ("attn_norm", "ffn_norm"):
        dev[k] = [to_dev(v) for v in wf[k]]
        orc[k] = wf[k]
    dev["final_norm"], orc["final_norm"] = to_dev(wf["final_norm"]), wf["final_norm"]
    kc = [_shapes.cache_bits(seed, ms, l, "k") for l in range(ms.n_layers)]
    vc = [_shapes.cache_bits(seed, ms, l, "v") for l in range(ms.n_layers)]
    kd = [to_dev(c.view(np.int16)) for c in kc]
    vd = [to_dev(c.view(np.int16)) for c in vc]
    model = d.DecodeModel(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, dev,
                          kd, vd, DT[ms.cache_dtype], ms.eps, ms.theta)
    return model, orc, kc, vc


def _oshape(ms):
    return ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, ms.eps,
                       ms.theta)


def _rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref * ref)))


CASES = [(_shapes.TINY, 3, 1), (_shapes.TINY, 2, 4), (_shapes.TINY_BF16, 5, 1), (_shapes.LLAMA68M, 4, 1),
         (_shapes.LLAMA68M, 1, 1)]


@pytest.mark.parametrize("ms,b,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_step_matches_oracle(cuda_device, ms, b, T):
    model, orc, kc, vc = _build(ms)
    bi, lens, toks = _shapes.step_meta(1, ms, b, T)
    ws = model.workspace(b * T)
    logits = to_host(model.step(toks, bi, T, lens, ws))
    ref, nk, nv = ostep.decode_step(_oshape(ms), orc, kc, vc, ms.cache_dtype, toks, bi, T, lens)
    err = _rel_err(logits, ref)
    assert err < STEP_TOL, f"max |g - r| / rms(r) = {err:.3e}"
    # the argmax of every row agrees unless the top two logits are within tolerance
    top = np.argmax(ref, axis=1)
    for t in range(len(toks)):
        g = int(np.argmax(logits[t]))
        assert g == top[t] or abs(ref[t, g] - ref[t, top[t]]) < STEP_TOL * np.sqrt(np.mean(ref * ref))
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


@pytest.mark.parametrize("ms,b,T", [(_shapes.TINY, 3, 2), (_shapes.LLAMA68M, 4, 1)], ids=["tiny", "llama"])
def test_batched_step_rows_equal_single_sequence_steps(cuda_device, ms, b, T):
    model, _, _, _ = _build(ms)
    bi, lens, toks = _shapes.step_meta(2, ms, b, T)
    ws = model.workspace(b * T)
    batched = to_host(model.step(toks, bi, T, lens, ws))
    for s in range(b):
        one = to_host(model.step(toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1], ws))
        assert np.array_equal(one.view(np.uint32), batched[s * T:(s + 1) * T].view(np.uint32)), s


def test_graph_replay_equals_eager_step(cuda_device):
    import torch
    ms = _shapes.LLAMA68M
    model, _, _, _ = _build(ms)
    b, T = 4, 1
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
