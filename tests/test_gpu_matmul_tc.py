"""GPU parity of the wide-batch q8_0 matmul on the tensor cores
(dsb_matmul_q8_0_wide) against the oracle.

The kernel splits every dequantised value d*q exactly into two f16 parts and
accumulates hi*hi + hi*lo + lo*hi in float32 over the whole row.  Pins:
integer-valued inputs (every scale 1, every partial sum an integer below
2^24) give the oracle's result bit for bit, so operand layout, descriptors and
accumulation are exact; on ordinary inputs the error stays below 1e-5 of the
output RMS, far inside the matmul tolerance, which a missing lo term (~3e-4)
would break.  Token counts cover one and several 128-row token tiles with
ragged tails, and row counts ragged against the 128-row weight tile.
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


def _case(seed, rows, cols, n_tok):
    d = _dsb()
    w32 = synth.normal_rows(seed, synth.stream_id(synth.STREAM_W, 11), rows, cols, 0.02)
    x32 = synth.normal_rows(seed, synth.stream_id(synth.STREAM_X, 11), n_tok, cols, 1.0)
    w_dev, x_dev = d.quantize_q8_0(to_dev(w32)), d.quantize_q8_0(to_dev(x32))
    w_or, x_or = oq.quantize_rows(w32), oq.quantize_rows(x32)
    assert to_host(w_dev).tobytes() == w_or.tobytes()
    assert to_host(x_dev).tobytes() == x_or.tobytes()
    return w_dev, x_dev, w_or, x_or


def _integer_rows(rng, n, cols):
    """Integer values in [-127, 127] with a +-127 in every 32-block: the q8_0
    scale is exactly 1 and the codes are the values."""
    x = rng.integers(-127, 128, (n, cols)).astype(np.float32)
    x[:, ::32] = np.where(rng.random((n, cols // 32)) < 0.5, -127.0, 127.0)
    return x


@pytest.mark.parametrize("rows,cols,n_tok", [(128, 256, 17), (1000, 1024, 130), (300, 768, 1), (2304, 768, 64)])
def test_wide_exact_on_integer_inputs(cuda_device, rows, cols, n_tok):
    rng = np.random.default_rng(rows + cols + n_tok)
    w32, x32 = _integer_rows(rng, rows, cols), _integer_rows(rng, n_tok, cols)
    d = _dsb()
    w_dev, x_dev = d.quantize_q8_0(to_dev(w32)), d.quantize_q8_0(to_dev(x32))
    w_or, x_or = oq.quantize_rows(w32), oq.quantize_rows(x32)
    assert to_host(w_dev).tobytes() == w_or.tobytes() and to_host(x_dev).tobytes() == x_or.tobytes()
    want = omm.matmul_q8_0(w_or, x_or)
    assert np.all(np.abs(want) < 2 ** 24) and np.array_equal(want, np.round(want))
    got = to_host(d.matmul_q8_0_wide(w_dev, rows, cols, x_dev, n_tok))
    assert np.array_equal(got.astype(np.float64), want)


def test_wide_extreme_codes_exact(cuda_device):
    """Codes +-127 everywhere with unit scales: |y| reaches cols * 127^2."""
    rows, cols, n_tok = 256, 1024, 32
    rng = np.random.default_rng(7)
    w32 = np.where(rng.random((rows, cols)) < 0.5, -127.0, 127.0).astype(np.float32)
    x32 = np.where(rng.random((n_tok, cols)) < 0.5, -127.0, 127.0).astype(np.float32)
    w32[0] = 127.0
    x32[0], x32[1] = 127.0, -127.0
    d = _dsb()
    w_or, x_or = oq.quantize_rows(w32), oq.quantize_rows(x32)
    want = omm.matmul_q8_0(w_or, x_or)
    assert want[0, 0] == cols * 127 * 127 and want[1, 0] == -cols * 127 * 127
    got = to_host(d.matmul_q8_0_wide(d.quantize_q8_0(to_dev(w32)), rows, cols, d.quantize_q8_0(to_dev(x32)), n_tok))
    assert np.array_equal(got.astype(np.float64), want)


@pytest.mark.parametrize("rows,cols,n_tok", [(1000, 1024, 37), (640, 7168, 200), (256, 17408, 20)])
def test_wide_error_far_below_tolerance(cuda_device, rows, cols, n_tok):
    """The split is exact and only the float32 accumulation rounds: the error
    stays below 1e-5 of the output RMS (dropping the lo parts would cost
    ~3e-4)."""
    w_dev, x_dev, w_or, x_or = _case(4, rows, cols, n_tok)
    got = to_host(_dsb().matmul_q8_0_wide(w_dev, rows, cols, x_dev, n_tok)).astype(np.float64)
    want = omm.matmul_q8_0(w_or, x_or)
    err = np.max(np.abs(got - want)) / np.sqrt(np.mean(want * want))
    assert err < 1e-5, err


def test_wide_flags_scales_beyond_f16_range(cuda_device):
    """A scale above 65504/127 (values beyond the f16 range) is reported."""
    d = _dsb()
    d.device_error()
    w32 = np.full((128, 256), 0.01, np.float32)
    w32[5, :32] = 127.0 * 600.0   # scale 600
    x32 = np.ones((20, 256), np.float32)
    d.matmul_q8_0_wide(d.quantize_q8_0(to_dev(w32)), 128, 256, d.quantize_q8_0(to_dev(x32)), 20)
    with pytest.raises(d.DsbError) as e:
        d.device_error()
    assert e.value.status == 6  # DSB_ERR_DEVICE
    d.device_error()  # cleared


@pytest.mark.parametrize("rows,cols,n_tok", [(1000, 1024, 37), (2304, 768, 64), (768, 3072, 200), (4099, 768, 129),
                                             (6144, 768, 256), (128, 5120, 17)])
def test_wide_matmul_matches_oracle(cuda_device, rows, cols, n_tok):
    w_dev, x_dev, w_or, x_or = _case(1, rows, cols, n_tok)
    y = to_host(_dsb().matmul_q8_0_wide(w_dev, rows, cols, x_dev, n_tok))
    assert_close(y, omm.matmul_q8_0(w_or, x_or), MATMUL_RTOL, MATMUL_ATOL, f"wide {rows}x{cols} n_tok={n_tok}")


def test_wide_rows_independent_of_token_count(cuda_device):
    """Token row t of a call equals the same row in a call with other rows
    around it (each output accumulates over K in the same order)."""
    rows, cols = 640, 1024
    w_dev, x_dev, _, _ = _case(2, rows, cols, 300)
    d = _dsb()
    full = to_host(d.matmul_q8_0_wide(w_dev, rows, cols, x_dev, 300))
    for lo, n in ((0, 1), (5, 17), (128, 128), (250, 50)):
        part = to_host(d.matmul_q8_0_wide(w_dev, rows, cols, x_dev[lo:lo + n].contiguous(), n))
        assert np.array_equal(part.view(np.uint32), full[lo:lo + n].view(np.uint32)), (lo, n)
    d.device_error()


def test_wide_rejects_bad_arguments(cuda_device):
    import torch
    d = _dsb()
    w_dev, x_dev, _, _ = _case(3, 128, 256, 20)
    y = torch.empty((20, 128), device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(d.DsbError) as e:
        d.matmul_q8_0_wide(w_dev, 128, 256, x_dev, 20, y=y, scratch=small)
    assert e.value.status == 3  # DSB_ERR_WORKSPACE
    w96 = d.quantize_q8_0(to_dev(np.ones((128, 96), np.float32)))
    with pytest.raises(d.DsbError) as e:
        d.matmul_q8_0_wide(w96, 128, 96, d.quantize_q8_0(to_dev(np.ones((20, 96), np.float32))), 20)
    assert e.value.status == 2  # DSB_ERR_UNSUPPORTED
    assert d.lib().dsb_matmul_q8_0_wide_scratch_bytes(0, 256) == 0


@pytest.mark.slow
@pytest.mark.parametrize("rows,cols,n_tok", [(32000, 768, 4096), (34816, 5120, 256)])
def test_wide_full_size_sampled_rows(cuda_device, rows, cols, n_tok):
    """Workload-sized matrices at the largest token counts, checked on
    sampled weight rows that the oracle computes one by one."""
    import torch
    d = _dsb()
    w32 = synth.normal_rows(5, synth.stream_id(synth.STREAM_W, 12), rows, cols, 0.02)
    w_dev = d.quantize_q8_0(torch.from_numpy(w32).cuda())
    del w32
    x32 = synth.normal_rows(5, synth.stream_id(synth.STREAM_X, 12), n_tok, cols, 1.0)
    x_dev = d.quantize_q8_0(to_dev(x32))
    x_or = oq.quantize_rows(x32)
    rng = np.random.default_rng(rows)
    sample = np.unique(np.concatenate([[0, 1, 127, 128, rows - 1], rng.integers(0, rows, 27)]))
    w_or = np.stack([oq.quantize_rows(synth.normal_rows(5, synth.stream_id(synth.STREAM_W, 12), rows, cols, 0.02,
                                                        int(r), int(r) + 1))[0] for r in sample])
    assert to_host(w_dev[torch.from_numpy(sample).cuda()]).tobytes() == w_or.tobytes()
    y = to_host(d.matmul_q8_0_wide(w_dev, rows, cols, x_dev, n_tok))
    assert_close(y[:, sample], omm.matmul_q8_0(w_or, x_or), MATMUL_RTOL, MATMUL_ATOL, f"{rows}x{cols} n_tok={n_tok}")
