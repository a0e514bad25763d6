"""The decode step on paged and ring KV (dsb_decode_step_paged) on the GPU.

* Linear block tables over the pages of a contiguous cache (permuted): the
  paged step is bitwise the contiguous step (same kernels, same keys), logits
  and every written page row.
* A two-page ring per sequence under a window W (W + T - 1 <= 256), with
  sequences long enough to wrap: bitwise the step on linear pages holding the
  whole history under the same window (the attention visits the same keys in
  the same chunks), and within the composed-step tolerance of the oracle's
  paged step, whose ring and window arithmetic the CPU tests pin.
"""
import numpy as np
import pytest

from oracle import kv as okv
from oracle import paged as opg
from oracle import step as ostep
from tests import _shapes
from tests.gpu_util import to_dev, to_host
from tests.test_gpu_step import DT, STEP_TOL_MAX, STEP_TOL_RMS, _build, _oshape, _rel_err, _rms_err

pytestmark = pytest.mark.gpu

P = opg.PAGE
SHAPES = [_shapes.ModelShape("tiny-paged", 256, 4, 2, 64, 512, 1000, 2, 4, 3 * P, "f16"),
          _shapes.ModelShape("tiny-paged-bf16-qkn", 512, 8, 2, 128, 768, 700, 1, 5, 3 * P, "bf16", qk_norm=True)]


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _pools(caches, perm, ms):
    """Host page pools holding every slot's blocks: block i of slot f at page perm[f * nb + i]."""
    nb = ms.ctx // P
    out = []
    for c in caches:
        pool = np.zeros((ms.full_batch_size * nb, ms.n_kv_heads, P, ms.head_dim), c.dtype)
        for f in range(ms.full_batch_size):
            for i in range(nb):
                pool[perm[f * nb + i]] = c[f, :, i * P:(i + 1) * P]
        out.append(pool)
    return out


def _dev_pages(kpools, vpools, ms):
    d = _dsb()
    return [d.kv_pages(to_dev(k.view(np.int16)), to_dev(v.view(np.int16)), DT[ms.cache_dtype])
            for k, v in zip(kpools, vpools)]


@pytest.mark.parametrize("ms,b,T", [(SHAPES[0], 3, 2), (SHAPES[0], 4, 4), (SHAPES[1], 2, 3)],
                         ids=["f16-b3-T2", "f16-b4-T4", "bf16-qkn-b2-T3"])
def test_linear_pages_equal_the_contiguous_step(cuda_device, ms, b, T):
    model, orc, kc, vc = _build(ms, seed=21)
    bi, lens, toks = _shapes.step_meta(21, ms, b, T)
    nb = ms.ctx // P
    perm = np.random.default_rng(3).permutation(ms.full_batch_size * nb)
    kp, vp = _pools(kc, perm, ms), _pools(vc, perm, ms)
    pages = _dev_pages(kp, vp, ms)
    ws = model.workspace(b * T)
    want = to_host(model.step(toks, bi, T, lens, ws))
    bt = np.array([[perm[int(f) * nb + i] for i in range(nb)] for f in bi], np.int32)
    got = to_host(model.step_paged(pages, toks, T, lens, bt, np.full(b, nb), np.zeros(b), ws))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for l in range(ms.n_layers):
        kc_after = to_host(model.k_caches[l]).view(np.uint16)
        vc_after = to_host(model.v_caches[l]).view(np.uint16)
        assert np.array_equal(to_host(pages[l]._tensors[0]).view(np.uint16), _pools([kc_after], perm, ms)[0])
        assert np.array_equal(to_host(pages[l]._tensors[1]).view(np.uint16), _pools([vc_after], perm, ms)[0])
    _dsb().device_error()


@pytest.mark.parametrize("ms,b,T", [(SHAPES[0], 3, 2), (SHAPES[1], 2, 1)], ids=["f16-b3-T2", "bf16-qkn-b2-T1"])
def test_ring_step_equals_linear_pages_and_matches_the_oracle(cuda_device, ms, b, T):
    model, orc, kc, vc = _build(ms, seed=22)
    bi, lens, toks = _shapes.step_meta(22, ms, b, T, 2 * P + 20)
    nb, W = ms.ctx // P, 200
    win = np.full(b, W)
    perm = np.arange(ms.full_batch_size * nb)
    lin_bt = np.array([[perm[int(f) * nb + i] for i in range(nb)] for f in bi], np.int32)
    ws = model.workspace(b * T)
    lin = _dev_pages(_pools(kc, perm, ms), _pools(vc, perm, ms), ms)
    want = to_host(model.step_paged(lin, toks, T, lens, lin_bt, np.full(b, nb), win, ws))
    # two pages per sequence, in swapped order; the old history of the last
    # 256 positions placed at (p / 128) mod 2
    ring_bt = np.array([[2 * s + 1, 2 * s] for s in range(b)], np.int32)
    rk, rv = [], []
    for caches, out in ((kc, rk), (vc, rv)):
        for l in range(ms.n_layers):
            pool = np.zeros((2 * b, ms.n_kv_heads, P, ms.head_dim), np.uint16)
            for s, f in enumerate(bi):
                for p in range(max(0, int(lens[s]) - 2 * P), int(lens[s]) - T):
                    page, row = opg.locate(p, ring_bt[s], 2, W)
                    pool[page, :, row] = caches[l][f, :, p]
            out.append(pool)
    ring = _dev_pages(rk, rv, ms)
    got = to_host(model.step_paged(ring, toks, T, lens, ring_bt, np.full(b, 2), win, ws))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    ref, nk, nv = ostep.decode_step(_oshape(ms), orc, rk, rv, ms.cache_dtype, toks, None, T, lens,
                                    geometry=(ring_bt, np.full(b, 2), win))
    assert _rms_err(got, ref) <= STEP_TOL_RMS
    assert _rel_err(got, ref) <= STEP_TOL_MAX
    # the step's rows landed where the ring puts them (values within one
    # cache ulp: the oracle rounds float64 activations, the GPU float32)
    for s in range(b):
        for j in range(T):
            page, row = opg.locate(int(lens[s]) - T + j, ring_bt[s], 2, W)
            g = okv.bits_to_f64(to_host(ring[0]._tensors[1]).view(np.uint16)[page, :, row], ms.cache_dtype)
            r = okv.bits_to_f64(nv[0][page, :, row], ms.cache_dtype)
            assert np.max(np.abs(g - r)) <= 4 * 2.0 ** -7 * max(1.0, float(np.max(np.abs(r))))
    _dsb().device_error()


def test_paged_step_rejects_bad_geometry(cuda_device):
    ms = SHAPES[0]
    model, orc, kc, vc = _build(ms, seed=23)
    d = _dsb()
    b, T = 2, 1
    bi, lens, toks = _shapes.step_meta(23, ms, b, T)
    nb = ms.ctx // P
    perm = np.arange(ms.full_batch_size * nb)
    pages = _dev_pages(_pools(kc, perm, ms), _pools(vc, perm, ms), ms)
    ws = model.workspace(b * T)
    bt = np.array([[perm[int(f) * nb + i] for i in range(nb)] for f in bi], np.int32)
    bad = bt.copy()
    bad[0, 0] = len(perm)  # page out of range
    with pytest.raises(d.DsbError):
        model.step_paged(pages, toks, T, lens, bad, np.full(b, nb), np.zeros(b), ws)
    same = bt.copy()
    same[1] = same[0]  # both sequences write the same page rows... only if their positions coincide
    lens_same = np.array([lens[0], lens[0]], np.int32)
    with pytest.raises(d.DsbError):
        model.step_paged(pages, toks, T, lens_same, same, np.full(b, nb), np.zeros(b), ws)
    with pytest.raises(ValueError):
        model.step_paged(pages[:-1] if ms.n_layers > 1 else [], toks, T, lens, bt, np.full(b, nb), np.zeros(b), ws)


def _geometry_steps(ms, b, T, max_blocks, seed):
    """Three steps' metadata for one captured graph: linear tables with no
    window; the next positions under a window W = 200 (each sequence's nb
    blocks used as a ring, which the longer sequences wrap); then the first
    step's lengths again with the sequences' page rows handed round (another
    block table).  Tables are max_blocks wide, the columns past nb padding."""
    bi, lens, toks = _shapes.step_meta(seed, ms, b, T)
    nb = ms.ctx // P
    perm = np.random.default_rng(seed).permutation(ms.full_batch_size * nb)
    bt = np.zeros((b, max_blocks), np.int32)
    for s, f in enumerate(bi):
        bt[s, :nb] = [perm[int(f) * nb + i] for i in range(nb)]
    rng = np.random.default_rng(seed + 1)
    toks2 = rng.integers(0, ms.vocab, size=b * T).astype(np.int32)
    toks3 = rng.integers(0, ms.vocab, size=b * T).astype(np.int32)
    zero, full = np.zeros(b, np.int32), np.full(b, nb, np.int32)
    return perm, [(toks, lens, bt, full, zero),
                  (toks2, lens + T, bt, full, np.full(b, 200, np.int32)),
                  (toks3, lens, np.roll(bt, 1, axis=0), full, zero)]


@pytest.mark.parametrize("ms,b,T,wide", [(SHAPES[0], 3, 2, False), (SHAPES[1], 2, 3, False), (SHAPES[0], 4, 2, True)],
                         ids=["f16-b3-T2-params", "bf16-qkn-b2-T3-params", "f16-b4-T2-mapped"])
def test_paged_graph_replay_equals_the_eager_paged_step(cuda_device, ms, b, T, wide):
    """The paged step captured once (dsb_step_graph_create_paged) and replayed
    with a new geometry each time is bitwise the eager paged step on a second
    copy of the pools: logits of every replay and the pools afterwards.  With
    1100-wide tables the metadata passes the first kernel's parameter block
    and the graph reads it from mapped memory."""
    import torch
    d = _dsb()
    model, orc, kc, vc = _build(ms, seed=24)
    nb = ms.ctx // P
    max_blocks = 1100 if wide else nb
    perm, steps = _geometry_steps(ms, b, T, max_blocks, seed=24 + b)
    kp, vp = _pools(kc, perm, ms), _pools(vc, perm, ms)
    for_graph, for_eager = _dev_pages(kp, vp, ms), _dev_pages(kp, vp, ms)
    ws = d.StepWorkspace(model.shape, b * T, P * (max_blocks + 1))
    logits = torch.empty((b * T, ms.vocab), dtype=torch.float32, device="cuda")
    g = model.graph_paged(for_graph, max_blocks, b, T, logits, ws)
    for i, (toks, lens, bt, nbk, win) in enumerate(steps):
        eager = to_host(model.step_paged(for_eager, toks, T, lens, bt, nbk, win, ws))
        replay = to_host(g.launch_paged(toks, lens, bt, nbk, win))
        assert np.array_equal(eager.view(np.uint32), replay.view(np.uint32)), i
    for l in range(ms.n_layers):
        for j in range(2):
            assert np.array_equal(to_host(for_graph[l]._tensors[j]).view(np.uint16),
                                  to_host(for_eager[l]._tensors[j]).view(np.uint16)), (l, j)
    g.close()
    d.device_error()


def test_paged_graph_rejects_the_other_kind_and_bad_geometry(cuda_device):
    import torch
    d = _dsb()
    ms = SHAPES[0]
    model, orc, kc, vc = _build(ms, seed=25)
    b, T = 2, 1
    nb = ms.ctx // P
    perm, steps = _geometry_steps(ms, b, T, nb, seed=25)
    pages = _dev_pages(_pools(kc, perm, ms), _pools(vc, perm, ms), ms)
    ws = d.StepWorkspace(model.shape, b * T, P * (nb + 1))
    logits = torch.empty((b * T, ms.vocab), dtype=torch.float32, device="cuda")
    toks, lens, bt, nbk, win = steps[0]
    g = model.graph_paged(pages, nb, b, T, logits, ws)
    bi = np.arange(b, dtype=np.int32)
    with pytest.raises(d.DsbError):   # a paged graph takes no contiguous launch
        g.launch(toks, bi, lens)
    bad = bt.copy()
    bad[0, 0] = len(perm)             # page out of range
    with pytest.raises(d.DsbError):
        g.launch_paged(toks, lens, bad, nbk, win)
    with pytest.raises(ValueError):   # a table of another width
        g.launch_paged(toks, lens, bt[:, :1], nbk, win)
    g.launch_paged(toks, lens, bt, nbk, win)
    torch.cuda.synchronize()
    g.close()
    c = model.graph(b, T, logits, model.workspace(b * T))
    st = d.lib().dsb_step_graph_launch_paged(c.handle, *[None] * 6)
    assert st == d.DSB_ERR_INVALID_ARG   # a contiguous graph takes no paged launch
    c.close()
    with pytest.raises(d.DsbError):   # block tables beyond the staging slot
        model.graph_paged(pages, 6000, b, T, logits, ws)
    d.device_error()
