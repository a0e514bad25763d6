"""Host-only checks of the C ABI (no GPU needed): the library builds, loads,
exports every function include/dsb.h declares, and rejects invalid arguments
before making any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from session_decode_step_dsb_gb300 import build, dsb
    if not os.path.exists(dsb.LIB_PATH):
        build.build()
    return dsb.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "dsb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsb_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "dsb_matmul_q8_0_narrow" in names and "dsb_attention_decode_multi" in names
    for n in names:
        assert hasattr(lib, n), n
    from session_decode_step_dsb_gb300 import dsb
    assert set(dsb.SIGNATURES) == set(names)


def test_version(lib):
    assert b"sm_103a" in lib.dsb_version()


def _err(lib):
    return lib.dsb_last_error().decode()


def test_matmul_rejects_bad_arguments(lib):
    from session_decode_step_dsb_gb300 import dsb
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    m = dsb.Q8Mat(fake, 64, 256)
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m), fake, 0, fake, None) == 1
    assert "n_tok" in _err(lib)
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m), fake, 17, fake, None) == 1
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m), None, 1, fake, None) == 1
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m), ctypes.c_void_p((1 << 20) + 4), 1, fake, None) == 1
    assert "aligned" in _err(lib)
    m2 = dsb.Q8Mat(fake, 64, 100)
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m2), fake, 1, fake, None) == 1
    m3 = dsb.Q8Mat(fake, 64, 96)
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m3), fake, 1, fake, None) == 2  # valid q8_0, unsupported width
    m4 = dsb.Q8Mat(fake, 0, 256)
    assert lib.dsb_matmul_q8_0_narrow(ctypes.byref(m4), fake, 1, fake, None) == 1
    assert lib.dsb_matmul_q8_0(ctypes.byref(m), fake, 0, fake, None) == 1
    assert lib.dsb_matmul_q8_0_block_dots(ctypes.byref(m), fake, 1, None, None) == 1


def test_fused_matmul_rejects_bad_arguments(lib):
    """The norm / SiLU-gate + matmul entry points validate on the host before
    any device work."""
    from session_decode_step_dsb_gb300 import dsb
    fake = ctypes.c_void_p(1 << 20)
    m = dsb.Q8Mat(fake, 64, 256)
    eps = ctypes.c_float(1e-6)
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), fake, fake, eps, 0, fake, None) == 1
    assert "n_tok" in _err(lib)
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), fake, fake, eps, 17, fake, None) == 1
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), fake, fake, ctypes.c_float(0.0), 2, fake, None) == 1
    assert "eps" in _err(lib)
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), fake, None, eps, 2, fake, None) == 1
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), None, fake, eps, 2, fake, None) == 1
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), ctypes.c_void_p((1 << 20) + 4), fake, eps, 2, fake,
                                       None) == 1
    wide = dsb.Q8Mat(fake, 64, 8448)
    assert lib.dsb_rmsnorm_matmul_q8_0(ctypes.byref(wide), fake, fake, eps, 2, fake, None) == 2
    assert lib.dsb_silu_matmul_q8_0(ctypes.byref(m), fake, 17, fake, None) == 1
    assert lib.dsb_silu_matmul_q8_0(ctypes.byref(m), fake, 2, None, None) == 1
    m96 = dsb.Q8Mat(fake, 64, 96)
    assert lib.dsb_silu_matmul_q8_0(ctypes.byref(m96), fake, 2, fake, None) == 2  # cols % 256


def test_staged_matmul_rejects_bad_arguments(lib):
    """The staged-layout entry points (the step's matmul path as an op) check
    the matrix, the token count and the staged buffer's size and alignment on
    the host before any device work."""
    from session_decode_step_dsb_gb300 import dsb
    fake = ctypes.c_void_p(1 << 20)
    m = dsb.Q8Mat(fake, 64, 1024)
    need = lib.dsb_matmul_q8_0_staged_bytes(16, 1024)
    assert need == 1024 // 32 * 36 * 16  # 32 blocks x (8 code words + 1 scale word) x 16 token slots
    assert lib.dsb_matmul_q8_0_staged_bytes(3, 1024) == 1024 // 32 * 36 * 4
    assert lib.dsb_matmul_q8_0_staged_bytes(9, 1024) == 1024 // 32 * 36 * 16
    for nt, cols in [(0, 1024), (17, 1024), (16, 100), (16, 0)]:
        assert lib.dsb_matmul_q8_0_staged_bytes(nt, cols) == 0
    assert lib.dsb_stage_q8_0(ctypes.byref(m), fake, 0, fake, need, None) == 1
    assert "n_tok" in _err(lib)
    assert lib.dsb_stage_q8_0(ctypes.byref(m), fake, 17, fake, need, None) == 1
    assert lib.dsb_stage_q8_0(ctypes.byref(m), None, 16, fake, need, None) == 1
    assert lib.dsb_stage_q8_0(ctypes.byref(m), fake, 16, None, need, None) == 3
    assert lib.dsb_stage_q8_0(ctypes.byref(m), fake, 16, fake, need - 16, None) == 3
    assert "staged" in _err(lib)
    assert lib.dsb_stage_q8_0(ctypes.byref(m), fake, 16, ctypes.c_void_p((1 << 20) + 8), need, None) == 3
    assert lib.dsb_matmul_q8_0_staged(ctypes.byref(m), fake, need, 16, None, None) == 1
    assert lib.dsb_matmul_q8_0_staged(ctypes.byref(m), fake, need - 16, 16, fake, None) == 3
    assert lib.dsb_matmul_q8_0_staged(ctypes.byref(m), fake, need, 0, fake, None) == 1
    m96 = dsb.Q8Mat(fake, 64, 96)
    assert lib.dsb_matmul_q8_0_staged(ctypes.byref(m96), fake, need, 16, fake, None) == 2  # cols % 256


def test_quantize_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(1 << 20)
    assert lib.dsb_quantize_q8_0(fake, 4, 33, fake, None) == 1
    assert lib.dsb_quantize_q8_0(fake, -1, 32, fake, None) == 1
    assert lib.dsb_quantize_q8_0(None, 4, 32, fake, None) == 1
    assert lib.dsb_quantize_q8_0(None, 0, 32, None, None) == 0  # nothing to do


def _kv(fake, **kw):
    from session_decode_step_dsb_gb300 import dsb
    args = dict(k=fake, v=fake, dtype=0, full_batch_size=4, n_kv_heads=2, ctx=256, head_dim=64)
    args.update(kw)
    return dsb.KVCache(**args)


def _i32(a):
    arr = np.ascontiguousarray(np.asarray(a, np.int32))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def test_scatter_rejects_bad_metadata(lib):
    fake = ctypes.c_void_p(1 << 20)
    ws = fake  # never reached
    kv = _kv(fake)
    cases = [
        ([2, 0], [10, 20], 1, "ok-shape-but-ws-fake"),
    ]
    bi, pbi = _i32([2, 2])
    pos, ppos = _i32([10, 20])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 1, ppos, fake, fake, ws, None) == 1
    assert "duplicated" in _err(lib)
    bi, pbi = _i32([4, 0])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 1, ppos, fake, fake, ws, None) == 1
    bi, pbi = _i32([1, 0])
    pos, ppos = _i32([10, 256])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 1, ppos, fake, fake, ws, None) == 1
    assert "pos" in _err(lib)
    pos, ppos = _i32([5, 5, 7, 8])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 2, ppos, fake, fake, ws, None) == 1
    assert "twice" in _err(lib)
    bi5, pbi5 = _i32([0, 1, 2, 3, 0])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi5, 5, 1, ppos, fake, fake, ws, None) == 1
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 0, ppos, fake, fake, ws, None) == 1
    bad = _kv(fake, dtype=7)
    assert lib.dsb_kv_scatter(ctypes.byref(bad), pbi, 2, 1, ppos, fake, fake, ws, None) == 1
    pos, ppos = _i32([3, 4])
    assert lib.dsb_kv_scatter(ctypes.byref(kv), pbi, 2, 1, ppos, fake, fake, None, None) == 3


def test_attention_rejects_bad_metadata(lib):
    fake = ctypes.c_void_p(1 << 20)
    kv = _kv(fake)
    bi, pbi = _i32([2, 0])
    lens, plens = _i32([0, 10])
    assert lib.dsb_attention_decode_multi(fake, 8, ctypes.byref(kv), pbi, 2, 1, plens, fake, fake, None) == 1
    assert "seq_lens" in _err(lib)
    lens, plens = _i32([257, 10])
    assert lib.dsb_attention_decode_multi(fake, 8, ctypes.byref(kv), pbi, 2, 1, plens, fake, fake, None) == 1
    lens, plens = _i32([3, 10])
    assert lib.dsb_attention_decode_multi(fake, 8, ctypes.byref(kv), pbi, 2, 4, plens, fake, fake, None) == 1
    assert lib.dsb_attention_decode_multi(fake, 7, ctypes.byref(kv), pbi, 2, 1, plens, fake, fake, None) == 1
    kv96 = _kv(fake, head_dim=96)
    lens, plens = _i32([3, 10])
    assert lib.dsb_attention_decode_multi(fake, 8, ctypes.byref(kv96), pbi, 2, 1, plens, fake, fake, None) == 2
    assert lib.dsb_attention_decode_multi(fake, 2 * 40, ctypes.byref(kv), pbi, 2, 2, plens, fake, fake, None) == 2
    assert lib.dsb_attention_decode_multi(fake, 8, ctypes.byref(kv), pbi, 2, 1, plens, fake, None, None) == 3
    # full_batch_size * n_kv_heads * ctx beyond the 32-bit row coordinate
    huge = _kv(fake, full_batch_size=256, n_kv_heads=128, ctx=65536)
    assert lib.dsb_attention_decode_multi(fake, 128, ctypes.byref(huge), pbi, 2, 1, plens, fake, fake, None) == 2
    assert "2^31" in _err(lib)
    assert lib.dsb_kv_scatter(ctypes.byref(huge), pbi, 2, 1, plens, fake, fake, fake, None) == 2


def test_paged_rejects_pools_beyond_the_row_coordinate(lib):
    from session_decode_step_dsb_gb300 import dsb
    fake = ctypes.c_void_p(1 << 20)
    pages = dsb.KVPages(fake, fake, 0, 1 << 20, 16, 64)   # 2^20 pages x 16 heads x 128 rows = 2^31 rows
    bt, pbt = _i32([[0, 1]])
    nb, pnb = _i32([2])
    win, pwin = _i32([0])
    lens, plens = _i32([200])
    assert lib.dsb_attention_decode_paged(fake, 16, ctypes.byref(pages), pbt, 2, pnb, pwin, 1, 1, plens, fake,
                                          fake, None) == 2
    assert "2^31" in _err(lib)


def test_rope_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(1 << 20)
    pos, ppos = _i32([0, -1])
    assert lib.dsb_rope_posvec(fake, 4, fake, 2, 64, 2, ppos, ctypes.c_float(10000.0), fake, None) == 1
    pos, ppos = _i32([0, 1])
    assert lib.dsb_rope_posvec(fake, 4, fake, 2, 63, 2, ppos, ctypes.c_float(10000.0), fake, None) == 1
    assert lib.dsb_rope_posvec(fake, 4, None, 2, 64, 2, ppos, ctypes.c_float(10000.0), fake, None) == 1
    assert lib.dsb_rope_posvec(fake, 4, fake, 2, 64, 2, ppos, ctypes.c_float(-1.0), fake, None) == 1
    assert lib.dsb_rope_posvec(fake, 4, fake, 2, 64, 2, ppos, ctypes.c_float(10000.0), None, None) == 3
    from session_decode_step_dsb_gb300 import dsb
    th, eps = ctypes.byref(dsb.rope_params(10000.0)), ctypes.c_float(1e-6)
    assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, th, fake, fake, ctypes.c_float(-1.0), fake,
                                     None) == 1
    assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, th, fake, fake, ctypes.c_float(float("nan")),
                                     fake, None) == 1
    assert "eps" in _err(lib)
    assert lib.dsb_head_rmsnorm_rope(fake, 4, None, 0, 64, 2, ppos, th, fake, fake, eps, fake, None) == 1
    assert "k_norm" in _err(lib)
    assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, th, fake, None, eps, None, None) == 3
    assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, None, fake, None, eps, fake, None) == 1
    for bad in (dsb.Yarn(4.0, 0), dsb.Yarn(4.0, 4096, 1.0, 32.0), dsb.Yarn(4.0, 4096, 32.0, 0.0),
                dsb.Yarn(float("inf"), 4096)):
        r = ctypes.byref(dsb.rope_params(10000.0, bad))
        assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, r, fake, None, eps, fake, None) == 1, bad
    ok = ctypes.byref(dsb.rope_params(10000.0, dsb.Yarn(4.0, 4096)))
    assert lib.dsb_head_rmsnorm_rope(fake, 4, fake, 2, 64, 2, ppos, ok, fake, None, eps, None, None) == 3


def test_workspace_sizes(lib):
    assert lib.dsb_workspace_bytes(-1, 8, 64, 256) == 0
    a = lib.dsb_workspace_bytes(2, 8, 64, 256)
    b = lib.dsb_workspace_bytes(16, 40, 128, 4096)
    assert 0 < a < b
    # partials: n_tok * Hq * ceil(ctx/128) * (D+2) floats beyond the fixed metadata area
    assert b - lib.dsb_workspace_bytes(0, 40, 128, 4096) >= 16 * 40 * 32 * 130 * 4
    out = ctypes.c_void_p()
    assert lib.dsb_workspace_create(None, 1 << 20, ctypes.byref(out)) == 1
    assert lib.dsb_workspace_create(ctypes.c_void_p((1 << 20) + 8), 1 << 20, ctypes.byref(out)) == 1
    assert lib.dsb_workspace_create(ctypes.c_void_p(1 << 20), 100, ctypes.byref(out)) == 3


def test_step_graph_entry_points_reject_null_handles(lib):
    """The captured-step entry points, both kinds, refuse missing handles on
    the host before any CUDA call."""
    out = ctypes.c_void_p()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.dsb_step_graph_create_paged(None, None, 2, 1, 1, fake, fake, None, ctypes.byref(out)) == 1
    assert lib.dsb_step_graph_create_paged(None, None, 2, 1, 1, fake, fake, None, None) == 1
    assert "out" in _err(lib)
    assert lib.dsb_step_graph_launch_paged(None, None, None, None, None, None, None) == 1
    assert "graph" in _err(lib)
    assert lib.dsb_step_graph_launch(None, None, None, None, None) == 1
    assert lib.dsb_step_graph_create(None, 1, 1, fake, fake, None, ctypes.byref(out)) == 1
    assert not out.value
