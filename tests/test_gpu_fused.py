"""GPU checks of the matmul with its activation quantisation fused in front
(dsb_rmsnorm_matmul_q8_0, dsb_silu_matmul_q8_0): bitwise equal to the
two-call sequence (the standalone quantising kernel, then the narrow matmul),
which the glue and matmul tests hold to the oracle.  Shapes cover the step's
matrices (one and several k-split ranks, ragged rows, k-split and rows-mode
tilings) and every token count class."""
import numpy as np
import pytest

from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _weights(seed, rows, cols):
    d = _dsb()
    return d.quantize_q8_0(to_dev(synth.normal_rows(seed, synth.stream_id(synth.STREAM_W, 50), rows, cols, 0.02)))


@pytest.mark.parametrize("rows,cols,n_tok", [(2304, 768, 8), (32000, 768, 8), (6144, 768, 1), (300, 1024, 16),
                                             (1000, 5120, 3), (128, 8192, 5), (7168, 5120, 16), (640, 768, 11)])
def test_rmsnorm_matmul_bitwise_two_calls(cuda_device, rows, cols, n_tok):
    d = _dsb()
    w = _weights(rows + cols, rows, cols)
    x = synth.normal_rows(1, synth.stream_id(synth.STREAM_X, 51), n_tok, cols, 1.0)
    x *= (0.1 + np.arange(n_tok, dtype=np.float32))[:, None]
    nw = (1.0 + synth.normal_rows(1, synth.stream_id(synth.STREAM_X, 52), 1, cols, 0.1)[0]).astype(np.float32)
    xd, nwd = to_dev(x), to_dev(nw)
    fused = to_host(d.rmsnorm_matmul_q8_0(w, rows, cols, xd, nwd, 1e-6))
    two = to_host(d.matmul_q8_0_narrow(w, rows, cols, d.rmsnorm_q8_0(xd, nwd, 1e-6), n_tok))
    assert np.array_equal(fused.view(np.uint32), two.view(np.uint32))
    d.device_error()


@pytest.mark.parametrize("rows,cols,n_tok", [(768, 3072, 8), (5120, 17408, 2), (640, 768, 16), (300, 256, 7),
                                             (5120, 17408, 16), (768, 3072, 1)])
def test_silu_matmul_bitwise_two_calls(cuda_device, rows, cols, n_tok):
    d = _dsb()
    w = _weights(rows * 3 + cols, rows, cols)
    gu = synth.normal_rows(2, synth.stream_id(synth.STREAM_X, 53), n_tok, 2 * cols, 2.0)
    gud = to_dev(gu)
    fused = to_host(d.silu_matmul_q8_0(w, rows, cols, gud))
    two = to_host(d.matmul_q8_0_narrow(w, rows, cols, d.silu_mul_q8_0(gud), n_tok))
    assert np.array_equal(fused.view(np.uint32), two.view(np.uint32))
    d.device_error()


def test_fused_matmul_rejects_bad_arguments(cuda_device):
    import torch
    d = _dsb()
    w = _weights(3, 256, 768)
    x = torch.zeros((17, 768), device="cuda")
    nw = torch.ones(768, device="cuda")
    with pytest.raises(d.DsbError) as e:
        d.rmsnorm_matmul_q8_0(w, 256, 768, x, nw, 1e-6)
    assert e.value.status == 1  # n_tok above 16
    with pytest.raises(d.DsbError) as e:
        d.rmsnorm_matmul_q8_0(w, 256, 768, x[:4], nw, 0.0)
    assert e.value.status == 1  # eps must be > 0
    wide = _weights(4, 64, 8448)
    with pytest.raises(d.DsbError) as e:
        d.rmsnorm_matmul_q8_0(wide, 64, 8448, torch.zeros((2, 8448), device="cuda"), torch.ones(8448, device="cuda"),
                              1e-6)
    assert e.value.status == 2  # RMSNorm rows above 8192
