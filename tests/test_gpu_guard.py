"""Guard bands around the buffers the library writes.

A device-side memory checker is not available on this machine, so this file
stands in for it for writes: each output buffer is a view into a larger device
allocation whose leading and trailing GUARD bytes hold a fixed byte pattern,
and after the call both bands must still hold it.  The shapes are ragged (row
counts that are no multiple of a warp's 32 rows or of a CTA tile, token counts
that are no multiple of 8, contexts that are no multiple of the 128-key chunk
or the 64-key copy box), so the kernels' edge handling is what runs.  Each
result is also compared bitwise with the same call on a plain allocation: the
placement of a buffer changes nothing.
"""
import ctypes

import numpy as np
import pytest

from session_decode_step_dsb_gb300 import synth
from tests import _shapes
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

GUARD = 8192
PATTERN = 0xA5
DT = {"f16": 0, "bf16": 1}


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


class Guarded:
    """nbytes of device memory between two GUARD-byte bands of PATTERN."""

    def __init__(self, nbytes):
        import torch
        self.n = int(nbytes)
        self.buf = torch.full((2 * GUARD + self.n,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(*shape)

    def check(self, what):
        import torch
        torch.cuda.synchronize()
        h = self.buf.cpu().numpy()
        lo, hi = h[:GUARD], h[GUARD + self.n:]
        assert np.all(lo == PATTERN), f"{what}: {int(np.sum(lo != PATTERN))} guard bytes before the buffer changed"
        assert np.all(hi == PATTERN), f"{what}: {int(np.sum(hi != PATTERN))} guard bytes after the buffer changed"


def _q8_weights(rows, cols, seed=3):
    w = synth.normal_rows(seed, synth.stream_id(synth.STREAM_W, 40), rows, cols, 0.02)
    return _dsb().quantize_q8_0(to_dev(w))


def _acts(n_tok, cols, seed=3):
    return to_dev(synth.normal_rows(seed, synth.stream_id(synth.STREAM_X, 40), n_tok, cols, 1.0))


@pytest.mark.parametrize("rows,cols,n_tok", [(1000, 1024, 1), (4099, 768, 3), (45, 256, 8), (1000, 2048, 13),
                                             (300, 1024, 16)])
def test_narrow_and_staged_matmul_write_only_their_outputs(cuda_device, rows, cols, n_tok):
    import torch
    d = _dsb()
    w = _q8_weights(rows, cols)
    x = _acts(n_tok, cols)
    gq = Guarded(n_tok * d.q8_rows_bytes(cols))
    xq = gq.view(torch.uint8, (n_tok, d.q8_rows_bytes(cols)))
    d.quantize_q8_0(x, xq=xq)
    gq.check("quantize")
    assert torch.equal(xq, d.quantize_q8_0(x))

    gy = Guarded(4 * n_tok * rows)
    y = gy.view(torch.float32, (n_tok, rows))
    d.matmul_q8_0_narrow(w, rows, cols, xq, n_tok, y=y)
    gy.check("narrow matmul")
    assert torch.equal(y, d.matmul_q8_0_narrow(w, rows, cols, xq, n_tok))

    nbytes = d.lib().dsb_matmul_q8_0_staged_bytes(n_tok, cols)
    gs = Guarded(nbytes)
    staged = gs.view(torch.uint8, (nbytes,))
    d.stage_q8_0(w, rows, cols, xq, n_tok, staged=staged)
    gs.check("staged layout")
    gy2 = Guarded(4 * n_tok * rows)
    y2 = gy2.view(torch.float32, (n_tok, rows))
    d.matmul_q8_0_staged(w, rows, cols, staged, n_tok, y=y2)
    gy2.check("staged matmul")
    assert torch.equal(y2, y)
    d.device_error()


@pytest.mark.parametrize("rows,cols,n_tok", [(1000, 1024, 37), (300, 768, 130)])
def test_wide_matmuls_write_only_their_outputs(cuda_device, rows, cols, n_tok):
    import torch
    d = _dsb()
    w = _q8_weights(rows, cols)
    xq = d.quantize_q8_0(_acts(n_tok, cols))
    gy = Guarded(4 * n_tok * rows)
    y = gy.view(torch.float32, (n_tok, rows))
    d.matmul_q8_0(w, rows, cols, xq, n_tok, y=y)
    gy.check("16-token chunked matmul")
    assert torch.equal(y, d.matmul_q8_0(w, rows, cols, xq, n_tok))

    sbytes = d.lib().dsb_matmul_q8_0_wide_scratch_bytes(n_tok, cols)
    gsc = Guarded(sbytes)
    gy2 = Guarded(4 * n_tok * rows)
    y2 = gy2.view(torch.float32, (n_tok, rows))
    d.matmul_q8_0_wide(w, rows, cols, xq, n_tok, y=y2, scratch=gsc.view(torch.uint8, (sbytes,)))
    gsc.check("tensor-core matmul scratch")
    gy2.check("tensor-core matmul")
    assert torch.equal(y2, d.matmul_q8_0_wide(w, rows, cols, xq, n_tok))
    d.device_error()


@pytest.mark.parametrize("n_tok,hidden,ffn", [(3, 5120, 17408), (9, 768, 3072), (1, 256, 512)])
def test_glue_kernels_write_only_their_outputs(cuda_device, n_tok, hidden, ffn):
    import torch
    d = _dsb()
    lib = d.lib()
    x = _acts(n_tok, hidden)
    nw = to_dev((1.0 + 0.1 * synth.normal(3, synth.stream_id(synth.STREAM_W, 41), (hidden,))).astype(np.float32))
    gq = Guarded(n_tok * d.q8_rows_bytes(hidden))
    xq = gq.view(torch.uint8, (n_tok, d.q8_rows_bytes(hidden)))
    assert lib.dsb_rmsnorm_q8_0(d._ptr(x), d._ptr(nw), n_tok, hidden, 1e-6, d._ptr(xq), None) == 0
    gq.check("RMSNorm + q8_0")
    assert torch.equal(xq, d.rmsnorm_q8_0(x, nw, 1e-6))

    gu = _acts(n_tok, 2 * ffn, seed=4)
    ga = Guarded(n_tok * d.q8_rows_bytes(ffn))
    aq = ga.view(torch.uint8, (n_tok, d.q8_rows_bytes(ffn)))
    assert lib.dsb_silu_mul_q8_0(d._ptr(gu), n_tok, ffn, d._ptr(aq), None) == 0
    ga.check("SiLU-gate + q8_0")
    assert torch.equal(aq, d.silu_mul_q8_0(gu))

    vocab = 700
    table = _q8_weights(vocab, hidden, seed=5)
    toks = synth.uniform_int(3, synth.stream_id(synth.STREAM_TOKENS, 9), 0, vocab - 1, n_tok)
    ws = d.Workspace(n_tok, 4, 64, 256)
    _, ptk = d._i32(toks)
    gh = Guarded(4 * n_tok * hidden)
    h = gh.view(torch.float32, (n_tok, hidden))
    assert lib.dsb_embed_q8_0(d._ptr(table), vocab, hidden, ptk, n_tok, d._ptr(h), ws.handle, None) == 0
    gh.check("embedding")
    assert torch.equal(h, d.embed_q8_0(table, vocab, hidden, toks, ws))
    d.device_error()


# F, hq, hkv, C, D, dtype, batch_index, seq_lens, T: contexts that are no
# multiple of the 64-key box, the last slot of the cache tensor in use, drafts
ATTN_CASES = [
    (6, 8, 2, 200, 64, "f16", [5, 0, 3], [200, 63, 129], 1),
    (5, 10, 2, 300, 128, "bf16", [4, 1], [300, 70], 3),
    (16, 40, 8, 4096, 128, "bf16", [15, 2, 7], [4096, 1, 2500], 1),
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=["f16-ragged", "bf16-drafts", "qwen3-shaped"])
def test_kv_write_and_attention_write_only_their_outputs(cuda_device, case):
    import torch
    d = _dsb()
    lib = d.lib()
    F, hq, hkv, C, D, dtype, bi, lens, T = case
    bi, lens = np.array(bi, np.int32), np.array(lens, np.int32)
    n_tok = len(bi) * T
    pos = np.array([L - T + j for L in lens for j in range(T)], np.int32)
    cache_bytes = 2 * F * hkv * C * D
    caches = []
    for which, kind in (("k", synth.STREAM_KCACHE), ("v", synth.STREAM_VCACHE)):
        g = Guarded(cache_bytes)
        bits = synth.cache_bits(6, synth.stream_id(kind, 3), (F, hkv, C, D), dtype)
        g.view(torch.int16, (F, hkv, C, D)).copy_(to_dev(bits.view(np.int16)))
        caches.append(g)
    kd = caches[0].view(torch.int16, (F, hkv, C, D))
    vd = caches[1].view(torch.int16, (F, hkv, C, D))
    kv = d.kv_cache(kd, vd, DT[dtype])
    ws = d.Workspace(n_tok, hq, D, C)

    # the fused RoPE + KV write, q rotated in place inside its own band
    qkv_cols = (hq + 2 * hkv) * D
    gqkv = Guarded(4 * n_tok * qkv_cols)
    qkv = gqkv.view(torch.float32, (n_tok, qkv_cols))
    qkv.copy_(to_dev(synth.normal(6, synth.stream_id(synth.STREAM_Q, 7), (n_tok, qkv_cols))))
    d.rope_kv_write(qkv, hq, kv, bi, T, pos, 10000.0, ws)
    gqkv.check("RoPE + KV write (qkv)")
    for g, what in zip(caches, ("K cache", "V cache")):
        g.check(f"RoPE + KV write ({what})")

    # the plain KV write of separate k / v rows
    k = _acts(n_tok * hkv, D, seed=7).view(n_tok, hkv, D)
    v = _acts(n_tok * hkv, D, seed=8).view(n_tok, hkv, D)
    d.kv_scatter(kv, bi, T, pos, k, v, ws)
    for g, what in zip(caches, ("K cache", "V cache")):
        g.check(f"KV write ({what})")

    # the attention, float32 rows and q8_0 rows
    q = qkv[:, :hq * D].contiguous().view(n_tok, hq, D)
    go = Guarded(4 * n_tok * hq * D)
    out = go.view(torch.float32, (n_tok, hq, D))
    d.attention_decode_multi(q, kv, bi, T, lens, ws, out=out)
    go.check("attention")
    assert torch.equal(out, d.attention_decode_multi(q, kv, bi, T, lens, ws))
    gx = Guarded(n_tok * d.q8_rows_bytes(hq * D))
    xq = gx.view(torch.uint8, (n_tok, d.q8_rows_bytes(hq * D)))
    _, pbi = d._i32(bi)
    _, psl = d._i32(lens)
    assert lib.dsb_attention_decode_multi_q8_0(d._ptr(q), hq, ctypes.byref(kv), pbi, len(bi), T, psl, d._ptr(xq),
                                               ws.handle, None) == 0
    gx.check("attention + q8_0")
    assert torch.equal(xq, d.attention_decode_multi_q8_0(q, kv, bi, T, lens, ws))
    for g, what in zip(caches, ("K cache", "V cache")):
        g.check(f"attention ({what}, read only)")
    d.device_error()


@pytest.mark.parametrize("ms,b,T", [(_shapes.TINY, 3, 2), (_shapes.LLAMA68M, 5, 1)], ids=["tiny", "llama-68m-shaped"])
def test_decode_step_writes_only_its_outputs(cuda_device, ms, b, T):
    """The whole step, eager and as a replayed graph: the logits and every
    layer's caches sit in their own bands."""
    import torch
    from tests.test_gpu_step import _build
    d = _dsb()
    base, _, kc, vc = _build(ms)
    guards, kd, vd = [], [], []
    shape = (ms.full_batch_size, ms.n_kv_heads, ms.ctx, ms.head_dim)
    for l in range(ms.n_layers):
        for bits, dst in ((kc[l], kd), (vc[l], vd)):
            g = Guarded(2 * int(np.prod(shape)))
            g.view(torch.int16, shape).copy_(to_dev(bits.view(np.int16)))
            guards.append(g)
            dst.append(g.view(torch.int16, shape))
    yarn = d.Yarn(ms.yarn_factor, ms.yarn_orig_ctx) if ms.yarn_factor > 1 else None
    model = d.DecodeModel(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, base.w,
                          kd, vd, DT[ms.cache_dtype], ms.eps, ms.theta, yarn)
    bi, lens, toks = _shapes.step_meta(9, ms, b, T)
    n_tok = b * T
    ws = model.workspace(n_tok)
    gl = Guarded(4 * n_tok * ms.vocab)
    logits = gl.view(torch.float32, (n_tok, ms.vocab))
    model.step(toks, bi, T, lens, ws, logits=logits)
    gl.check("decode step logits")
    for g in guards:
        g.check("decode step caches")
    eager = to_host(logits).copy()

    # the next step, as a captured graph replay, into the same banded buffers
    lens2 = np.minimum(np.asarray(lens) + T, ms.ctx).astype(np.int32)
    graph = model.graph(b, T, logits, ws)
    graph.launch(toks, bi, lens2)
    gl.check("step graph logits")
    for g in guards:
        g.check("step graph caches")
    graph.close()
    assert np.all(np.isfinite(eager)) and np.all(np.isfinite(to_host(logits)))
    d.device_error()
