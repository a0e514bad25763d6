"""Several host threads driving the library at once, each with its own stream
and workspace, give the bits a serial run gives.

Each thread uses matrix shapes no earlier call has seen, so the threads fill
the library's launch-plan, occupancy and tensor-map memos concurrently; the
plans depend on the shape and the device only, so the results must be bitwise
equal to the serial ones computed afterwards."""
import threading

import numpy as np
import pytest

from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

# (rows, cols, n_tok) of the matmul and (F, Hq, Hkv, C, D, dtype) of the attention, per thread
CASES = [((1312, 2304, 3), (3, 8, 2, 384, 64, 0)),
         ((2080, 1280, 7), (2, 16, 4, 256, 128, 1)),
         ((544, 3328, 16), (4, 12, 12, 512, 64, 0)),
         ((3104, 1792, 1), (2, 40, 8, 640, 128, 1))]


def _inputs(i, case):
    import torch
    from session_decode_step_dsb_gb300 import dsb
    (rows, cols, n_tok), (F, hq, hkv, C, D, dt) = case
    w = dsb.quantize_q8_0(to_dev(synth.normal_rows(i, synth.stream_id(synth.STREAM_W, 90), rows, cols, 0.02)))
    xq = dsb.quantize_q8_0(to_dev(synth.normal_rows(i, synth.stream_id(synth.STREAM_X, 90), n_tok, cols, 1.0)))
    name = "f16" if dt == 0 else "bf16"
    kc = to_dev(synth.cache_bits(i, synth.stream_id(synth.STREAM_KCACHE, 90), (F, hkv, C, D), name).view(np.int16))
    vc = to_dev(synth.cache_bits(i, synth.stream_id(synth.STREAM_VCACHE, 90), (F, hkv, C, D), name).view(np.int16))
    bi = np.arange(F, dtype=np.int32)[::-1].copy()
    lens = np.array([C - 3 * s for s in range(F)], np.int32)
    q = to_dev(synth.normal(i, synth.stream_id(synth.STREAM_Q, 90), (F, hq, D)))
    torch.cuda.synchronize()
    return w, xq, kc, vc, bi, lens, q


def _run(inputs, case, ws, stream):
    from session_decode_step_dsb_gb300 import dsb
    (rows, cols, n_tok), (F, hq, hkv, C, D, dt) = case
    w, xq, kc, vc, bi, lens, q = inputs
    y = dsb.matmul_q8_0_narrow(w, rows, cols, xq, n_tok, stream=stream)
    out = dsb.attention_decode_multi(q, dsb.kv_cache(kc, vc, dt), bi, 1, lens, ws, stream=stream)
    return y, out


def test_threads_match_serial(cuda_device):
    import torch
    from session_decode_step_dsb_gb300 import dsb
    inputs = [_inputs(i, c) for i, c in enumerate(CASES)]
    results = [None] * len(CASES)
    errors = []
    start = threading.Barrier(len(CASES))

    def worker(i):
        try:
            (_, _, _), (F, hq, _, C, D, _) = CASES[i]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                ws = dsb.Workspace(F, hq, D, C)
                start.wait(timeout=60)
                for _ in range(3):
                    y, out = _run(inputs[i], CASES[i], ws, stream)
                stream.synchronize()
                results[i] = (to_host(y), to_host(out))
        except Exception as e:  # reported on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    dsb.device_error()
    for i, case in enumerate(CASES):
        (_, _, _), (F, hq, _, C, D, _) = case
        y, out = _run(inputs[i], case, dsb.Workspace(F, hq, D, C), None)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(y).view(np.uint32), results[i][0].view(np.uint32)), i
        assert np.array_equal(to_host(out).view(np.uint32), results[i][1].view(np.uint32)), i
