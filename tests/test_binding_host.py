"""Host-only checks of the Python binding (no GPU): a buffer too small for the
call, a wrong element type, or a host index array of the wrong length is
rejected in Python, before any pointer reaches the library (which sees bare
pointers and could not tell)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _u8(n):
    return torch.zeros(n, dtype=torch.uint8)


def test_matmul_buffers_are_sized_before_the_call():
    d = _dsb()
    rows, cols, n_tok = 64, 256, 4
    w = _u8(rows * cols // 32 * 34)
    xq = _u8(n_tok * cols // 32 * 34)
    with pytest.raises(ValueError, match="w_blocks holds"):
        d.matmul_q8_0_narrow(w[:-1], rows, cols, xq, n_tok)
    with pytest.raises(ValueError, match="xq holds"):
        d.matmul_q8_0_narrow(w, rows, cols, xq[:-34], n_tok)
    with pytest.raises(ValueError, match="y holds"):
        d.matmul_q8_0_narrow(w, rows, cols, xq, n_tok, y=torch.zeros((n_tok, rows - 1)))
    with pytest.raises(ValueError, match="y must be float32"):
        d.matmul_q8_0(w, rows, cols, xq, n_tok, y=torch.zeros((n_tok, rows), dtype=torch.float64))
    with pytest.raises(ValueError, match="w_blocks must be uint8"):
        d.matmul_q8_0_narrow(torch.zeros(rows * cols // 32 * 34, dtype=torch.int8), rows, cols, xq, n_tok)
    with pytest.raises(ValueError, match="x holds"):
        d.rmsnorm_matmul_q8_0(w, rows, cols, torch.zeros((n_tok, cols - 32)), torch.ones(cols), 1e-6)
    with pytest.raises(ValueError, match="norm_w holds"):
        d.rmsnorm_matmul_q8_0(w, rows, cols, torch.zeros((n_tok, cols)), torch.ones(cols - 1), 1e-6)
    with pytest.raises(ValueError, match="gu holds"):
        d.silu_matmul_q8_0(w, rows, cols, torch.zeros((n_tok, cols)))


def test_quantize_and_glue_buffers():
    d = _dsb()
    with pytest.raises(ValueError, match="x must be float32"):
        d.quantize_q8_0(torch.zeros((2, 64), dtype=torch.float16))
    with pytest.raises(ValueError, match="xq holds"):
        d.quantize_q8_0(torch.zeros((2, 64)), _u8(2 * 68 - 1))
    with pytest.raises(ValueError, match="w holds"):
        d.rmsnorm_q8_0(torch.zeros((2, 256)), torch.ones(255), 1e-6)
    with pytest.raises(ValueError, match="table holds"):
        d.embed_q8_0(_u8(10 * 24 * 34 - 1), 10, 768, [1, 2], ws=None)


def test_cache_descriptions_check_their_tensors():
    d = _dsb()
    k = torch.zeros((2, 2, 128, 64), dtype=torch.int16)
    with pytest.raises(ValueError, match="shapes differ"):
        d.kv_cache(k, torch.zeros((2, 2, 127, 64), dtype=torch.int16), 0)
    with pytest.raises(ValueError, match="16-bit"):
        d.kv_cache(k, torch.zeros((2, 2, 128, 64), dtype=torch.float32), 0)
    with pytest.raises(ValueError, match="16-bit"):
        d.kv_pages(torch.zeros((3, 2, 128, 64)), torch.zeros((3, 2, 128, 64)), 0)


class _FakeKV:
    n_kv_heads, head_dim = 2, 64


def test_host_arrays_have_the_call_length():
    d = _dsb()
    kv = _FakeKV()
    q = torch.zeros((4, 4, 64))
    with pytest.raises(ValueError, match="pos has 3 entries, needs 4"):
        d.kv_scatter(kv, [0, 1], 2, [1, 2, 3], torch.zeros((4, 2, 64)), torch.zeros((4, 2, 64)), ws=None)
    with pytest.raises(ValueError, match="k holds"):
        d.kv_scatter(kv, [0, 1], 2, [1, 2, 3, 4], torch.zeros((3, 2, 64)), torch.zeros((4, 2, 64)), ws=None)
    with pytest.raises(ValueError, match="seq_lens has 1 entries, needs 2"):
        d.attention_decode_multi(q, kv, [0, 1], 2, [9], ws=None)
    with pytest.raises(ValueError, match="q must be"):
        d.attention_decode_multi(q, kv, [0, 1], 1, [9, 9], ws=None)   # 2 token rows, q holds 4
    with pytest.raises(ValueError, match="out holds"):
        d.attention_decode_multi(q, kv, [0, 1], 2, [9, 9], ws=None, out=torch.zeros((4, 4, 63)))
    with pytest.raises(ValueError, match="pos has 1 entries"):
        d.rope_posvec(q, None, [0], 10000.0, ws=None)
    with pytest.raises(ValueError, match="qkv holds"):
        d.rope_kv_write(torch.zeros((2, 4 * 64)), 4, kv, [0, 1], 1, [3, 4], 10000.0, ws=None)
    with pytest.raises(ValueError, match="n_blocks has 1 entries, needs 2"):
        d.attention_decode_paged(q, kv, np.zeros((2, 3)), [1], [0, 0], 2, [5, 5], ws=None)
