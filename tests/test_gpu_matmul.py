"""GPU parity of the q8_0 quantiser and the narrow-batch q8_0 matmul.

Both sides start from the same seeded float32 draws: the GPU quantises with its
own kernel, the oracle with its own codec, and the bytes must be identical;
then each side runs its matmul on its own blocks.  All GPU calls go through the
C ABI (libdsb.so).
"""
import numpy as np
import pytest

from oracle import matmul as omm
from oracle import q8_0 as oq
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import MATMUL_ATOL, MATMUL_RTOL, assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _weights(seed, rows, cols, stream=7, row_lo=0, row_hi=None):
    return synth.normal_rows(seed, synth.stream_id(synth.STREAM_W, stream), rows, cols, 0.02, row_lo, row_hi)


def _acts(seed, n_tok, cols, stream=7):
    return synth.normal_rows(seed, synth.stream_id(synth.STREAM_X, stream), n_tok, cols, 1.0)


def _gpu_quant(x):
    import torch
    return _dsb().quantize_q8_0(to_dev(x))


@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 96), (300, 768), (33, 4096)])
def test_quantize_bit_exact(cuda_device, rows, cols):
    rng = np.random.default_rng(rows * 131 + cols)
    x = (rng.standard_normal((rows, cols)) * rng.uniform(1e-3, 1e3, (rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                       # all-zero block
    if cols >= 64:
        x[0, 32:64] = np.linspace(-127, 127, 32).astype(np.float32)  # exact scale 1.0, many ties
        x[0, 33] = 2.5
        x[0, 34] = -0.5
    got = to_host(_gpu_quant(x))
    want = oq.quantize_rows(x)
    assert got.tobytes() == want.tobytes()


def test_quantize_hand_blocks(cuda_device):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "q8_0_hand_blocks.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        _, vals, hexes = (p.strip() for p in line.split("|"))
        x = np.array([float(v) for v in vals.split()], dtype=np.float32)[None, :]
        want = bytes(int(h, 16) for h in hexes.split())
        assert to_host(_gpu_quant(x)).tobytes() == want


def _case(seed, rows, cols, n_tok):
    w32 = _weights(seed, rows, cols)
    x32 = _acts(seed, n_tok, cols)
    w_dev = _gpu_quant(w32)
    x_dev = _gpu_quant(x32)
    w_or = oq.quantize_rows(w32)
    x_or = oq.quantize_rows(x32)
    assert to_host(w_dev).tobytes() == w_or.tobytes()
    assert to_host(x_dev).tobytes() == x_or.tobytes()
    return w_dev, x_dev, w_or, x_or


@pytest.mark.parametrize("rows,cols,n_tok", [(1024, 1024, 2), (1000, 2048, 16), (45, 256, 5), (768, 3072, 3)])
def test_block_dots_bit_exact(cuda_device, rows, cols, n_tok):
    w_dev, x_dev, w_or, x_or = _case(0, rows, cols, n_tok)
    got = to_host(_dsb().matmul_q8_0_block_dots(w_dev, rows, cols, x_dev, n_tok))
    want = omm.block_dots(w_or, x_or)
    assert got.dtype == np.int32 and np.array_equal(got.astype(np.int64), want)


@pytest.mark.parametrize("rows,cols", [(1024, 1024), (1000, 2048), (4099, 768), (64, 5120), (37, 256)])
@pytest.mark.parametrize("n_tok", [1, 2, 3, 4, 8, 16])
def test_matmul_matches_oracle(cuda_device, rows, cols, n_tok):
    w_dev, x_dev, w_or, x_or = _case(1, rows, cols, n_tok)
    y = to_host(_dsb().matmul_q8_0_narrow(w_dev, rows, cols, x_dev, n_tok))
    assert_close(y, omm.matmul_q8_0(w_or, x_or), MATMUL_RTOL, MATMUL_ATOL, f"y {rows}x{cols} n_tok={n_tok}")


@pytest.mark.parametrize("rows,cols", [(1024, 1024), (1000, 7168), (300, 17408)])
def test_columns_bitwise_equal_single_runs(cuda_device, rows, cols):
    """Column t of an n_tok = k call equals the n_tok = 1 call on row t."""
    w_dev, x_dev, _, _ = _case(2, rows, cols, 16)
    d = _dsb()
    singles = [to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev[t:t + 1].contiguous(), 1))[0] for t in range(16)]
    for k in (2, 3, 7, 16):
        yk = to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev[:k].contiguous(), k))
        for t in range(k):
            assert np.array_equal(yk[t].view(np.uint32), singles[t].view(np.uint32)), (k, t)


def test_wide_path_matches_narrow_columns(cuda_device):
    rows, cols, n_tok = 500, 768, 37
    w_dev, x_dev, w_or, x_or = _case(3, rows, cols, n_tok)
    d = _dsb()
    y = to_host(d.matmul_q8_0(w_dev, rows, cols, x_dev, n_tok))
    assert_close(y, omm.matmul_q8_0(w_or, x_or), MATMUL_RTOL, MATMUL_ATOL, "wide")
    y1 = to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev[20:21].contiguous(), 1))
    assert np.array_equal(y[20].view(np.uint32), y1[0].view(np.uint32))


def test_repeat_calls_identical(cuda_device):
    rows, cols = 2048, 1024
    w_dev, x_dev, _, _ = _case(4, rows, cols, 8)
    d = _dsb()
    a = to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev, 8))
    b = to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev, 8))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    d.device_error()


@pytest.mark.slow
@pytest.mark.parametrize("rows,cols", [(7168, 7168), (18432, 7168), (129280, 7168), (34816, 5120), (5120, 17408)])
def test_full_size_sampled_rows(cuda_device, rows, cols):
    """Full-size matrices of the workloads, every n_tok the bench times,
    checked on sampled rows (first, last, random) that the oracle computes
    one by one."""
    import torch
    d = _dsb()
    w32 = _weights(5, rows, cols)
    w_dev = d.quantize_q8_0(torch.from_numpy(w32).cuda())
    del w32
    x32 = _acts(5, 16, cols)
    x_dev = d.quantize_q8_0(to_dev(x32))
    x_or = oq.quantize_rows(x32)
    assert to_host(x_dev).tobytes() == x_or.tobytes()
    rng = np.random.default_rng(rows)
    sample = np.unique(np.concatenate([[0, 1, 31, 32, rows - 1], rng.integers(0, rows, 59)]))
    w_or = np.stack([oq.quantize_rows(_weights(5, rows, cols, row_lo=int(r), row_hi=int(r) + 1))[0] for r in sample])
    w_dev_rows = to_host(w_dev[torch.from_numpy(sample).cuda()])
    assert w_dev_rows.tobytes() == w_or.tobytes()
    for n_tok in (1, 2, 3, 4, 8, 16):
        y = to_host(d.matmul_q8_0_narrow(w_dev, rows, cols, x_dev[:n_tok].contiguous(), n_tok))
        want = omm.matmul_q8_0(w_or, x_or[:n_tok])
        assert_close(y[:, sample], want, MATMUL_RTOL, MATMUL_ATOL, f"{rows}x{cols} n_tok={n_tok}")
