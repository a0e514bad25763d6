"""GPU parity of the staged narrow matmul: the decode step's matmul path.

dsb_stage_q8_0 writes the staged activation layout of q8_0 rows (what the
step's RMSNorm, SiLU-gate and attention-merge kernels write next to their q8_0
rows), and dsb_matmul_q8_0_staged must return bitwise what
dsb_matmul_q8_0_narrow returns on the same rows: the same kernel, plan, codes
and scales, only the activations' way into shared memory differs (antirez/ds4
PR #530, "Correctness": a batched result equals the independent runs;
test_gpu_matmul.py holds the narrow kernel to the oracle).  Two shapes are
also checked against the oracle directly, on sampled rows.
"""
import numpy as np
import pytest

from oracle import matmul as omm
from tests.gpu_util import MATMUL_ATOL, MATMUL_RTOL, assert_close, to_host

pytestmark = pytest.mark.gpu


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _weights(rows, cols, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w = torch.empty((rows, cols // 32 * 34), dtype=torch.uint8, device="cuda")
    step = max(1, (1 << 24) // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        _dsb().quantize_q8_0(torch.randn((r1 - r0, cols), generator=g, device="cuda") * 0.02, w[r0:r1])
    return w


def _acts(n_tok, cols, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1)
    x = torch.randn((n_tok, cols), generator=g, device="cuda")
    x[0, :32] = 0.0  # an all-zero block (scale 0)
    return _dsb().quantize_q8_0(x)


# Qwen3-14B-shaped O / QKV projections and the DeepSeek-class dense shape
# (several cluster splits), a ragged last tile, a tall matrix whose clusters
# take many tiles each, the gate|up matrix (one CTA per tile, no cluster), and
# a small matrix (row groups of fewer than 8 warps).
SHAPES = [(5120, 5120), (7168, 5120), (18432, 7168), (5000, 2048), (40000, 1024), (34816, 5120), (768, 768)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_staged_bitwise_narrow(cuda_device, rows, cols):
    import torch
    dsb = _dsb()
    w = _weights(rows, cols, seed=rows + cols)
    x = _acts(16, cols, seed=rows)
    for nt in (1, 3, 7, 8, 9, 12, 15, 16):
        xs = x[:nt].contiguous()
        want = dsb.matmul_q8_0_narrow(w, rows, cols, xs, nt)
        staged = dsb.stage_q8_0(w, rows, cols, xs, nt)
        got = dsb.matmul_q8_0_staged(w, rows, cols, staged, nt)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), (rows, cols, nt)
    dsb.device_error()


@pytest.mark.parametrize("rows,cols,nt", [(5000, 2048, 16), (5000, 2048, 11), (768, 768, 16)])
def test_staged_matches_oracle(cuda_device, rows, cols, nt):
    dsb = _dsb()
    w = _weights(rows, cols, seed=3 * rows + cols)
    x = _acts(nt, cols, seed=cols)
    staged = dsb.stage_q8_0(w, rows, cols, x, nt)
    got = to_host(dsb.matmul_q8_0_staged(w, rows, cols, staged, nt))
    pick = np.unique(np.concatenate([np.arange(0, rows, max(1, rows // 97)), [rows - 1]]))
    want = omm.matmul_q8_0(to_host(w), to_host(x), rows=pick)
    assert_close(got[:, pick], want, MATMUL_RTOL, MATMUL_ATOL, f"staged {rows}x{cols} n_tok {nt}")
    dsb.device_error()


def test_staged_bad_arguments(cuda_device):
    import torch
    dsb = _dsb()
    rows, cols = 512, 1024
    w = _weights(rows, cols, seed=5)
    x = _acts(16, cols, seed=5)
    with pytest.raises(dsb.DsbError):
        dsb.stage_q8_0(w, rows, cols, x, 17)
    short = torch.empty(dsb.lib().dsb_matmul_q8_0_staged_bytes(16, cols) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):  # the binding's size check
        dsb.stage_q8_0(w, rows, cols, x, 16, staged=short)
    assert dsb.lib().dsb_matmul_q8_0_staged_bytes(0, cols) == 0
    assert dsb.lib().dsb_matmul_q8_0_staged_bytes(16, 1000) == 0
