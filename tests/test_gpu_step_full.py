"""The Qwen3-14B-shaped decode step at its full size on the GPU: 40 layers,
the 151936-row head, a bf16 cache of [16, 8, 4096, 128] per layer and the live
batch b = 16 (the pypto page's dynamic public batch 1..16), the configuration
the benchmark times.

The oracle cannot run 40 such layers, so the full-size step is held to what
holds at any size:

  * the traced step (every stage copied out) gives bitwise the untraced
    step's logits, and a captured-graph replay gives them too;
  * a batched step's rows equal each sequence's step run alone, bitwise
    (antirez/ds4 PR #530, "Correctness");
  * teacher-forced at the last stage: logits of sampled vocabulary rows equal
    the oracle's q8_0 matmul of those head rows and the step's own final
    q8_0 rows, within the matmul tolerance.  The sampled head rows are drawn
    on the host and quantised by the oracle, then written over the device
    head, so no oracle input comes from a device kernel but the final rows
    the chained stage comparison feeds it by design.
"""
import numpy as np
import pytest

from oracle import matmul as omm
from oracle import q8_0 as oq
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import MATMUL_ATOL, MATMUL_RTOL, assert_close, to_host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def test_full_size_qwen3_step(cuda_device):
    import torch
    import bench
    d = _dsb()
    ms = bench._shape("qwen3-14b")
    assert (ms.n_layers, ms.vocab, ms.hidden, ms.full_batch_size) == (40, 151936, 5120, 16)
    model = bench._make_model(ms, seed=1000)
    b, T = 16, 1
    bi, lens, toks = bench._meta(ms, b, T, seed=7)
    # head rows the oracle checks: drawn on the host, quantised by the oracle
    rng = np.random.default_rng(3)
    sample = np.unique(np.concatenate([[0, 1, ms.vocab - 1], rng.integers(0, ms.vocab, 21)]))
    stream = synth.stream_id(synth.STREAM_W, 40)
    head_rows = np.stack([oq.quantize_rows(synth.normal_rows(9, stream, ms.vocab, ms.hidden, 0.02, int(r),
                                                             int(r) + 1))[0] for r in sample])
    head = model.w["head"]
    head[torch.from_numpy(sample).cuda()] = torch.from_numpy(head_rows).cuda()
    ws = model.workspace(b * T)

    plain = to_host(model.step(toks, bi, T, lens, ws))
    traced, trace = model.step_trace(toks, bi, T, lens, ws)
    traced = to_host(traced)
    assert np.array_equal(traced.view(np.uint32), plain.view(np.uint32))
    assert np.all(np.isfinite(plain))

    x_final = to_host(trace["x_final"])
    want = omm.matmul_q8_0(head_rows, x_final)
    assert_close(plain[:, sample], want, MATMUL_RTOL, MATMUL_ATOL, "full-size step: sampled logits")

    for s in (0, 7, 15):
        one = to_host(model.step(toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1], ws))
        assert np.array_equal(one.view(np.uint32), plain[s * T:(s + 1) * T].view(np.uint32)), s

    logits = torch.empty((b * T, ms.vocab), dtype=torch.float32, device="cuda")
    g = model.graph(b, T, logits, ws)
    replay = to_host(g.launch(toks, bi, lens))
    g.close()
    assert np.array_equal(replay.view(np.uint32), plain.view(np.uint32))
    d.device_error()
