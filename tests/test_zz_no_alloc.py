"""The attention entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (allocator hooks, pools owned by another
framework, loops that must not take allocator locks); for them
dsb_attention_decode_multi_noalloc keeps its scratch in a static device array
instead of a caller workspace.  These tests call it through the C ABI and
check it against dsb_attention_decode_multi (same tolerance as the other
attention tests), on two calls in a row with different batches, so that
leftovers of the first call in the shared array cannot leak into the second.
This file is collected last so a stop-at-first-failure run has already run
everything else; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import kv as okv
from session_decode_step_dsb_gb300 import synth
from tests.gpu_util import ATTN_ATOL, ATTN_RTOL, assert_close, to_dev, to_host


def _dsb():
    from session_decode_step_dsb_gb300 import dsb
    return dsb


def _case(seed, F, hq, hkv, C, D, dtype, bi, lens, T):
    import torch
    kind_k = synth.stream_id(synth.STREAM_KCACHE, 50 + seed)
    kind_v = synth.stream_id(synth.STREAM_VCACHE, 50 + seed)
    kc = synth.cache_bits(seed, kind_k, (F, hkv, C, D), dtype)
    vc = synth.cache_bits(seed, kind_v, (F, hkv, C, D), dtype)
    q = synth.normal(seed, synth.stream_id(synth.STREAM_Q, 60 + seed), (len(bi) * T, hq, D))
    kd = to_dev(kc.view(np.int16))
    vd = to_dev(vc.view(np.int16))
    kv = _dsb().kv_cache(kd, vd, 0 if dtype == "f16" else 1)
    return kc, vc, q, kv


@pytest.mark.gpu
def test_no_alloc_matches_workspace_entry_on_two_calls(cuda_device):
    d = _dsb()
    cases = [
        # F, hq, hkv, C, D, dtype, batch_index, seq_lens, T
        (16, 40, 8, 4096, 128, "bf16", [3, 9, 15, 0], [1, 4096, 2500, 130], 1),
        (8, 12, 12, 2048, 64, "f16", [5, 1], [700, 129], 4),
    ]
    for n, (F, hq, hkv, C, D, dtype, bi, lens, T) in enumerate(cases):
        bi, lens = np.array(bi, np.int32), np.array(lens, np.int32)
        kc, vc, q, kv = _case(n, F, hq, hkv, C, D, dtype, bi, lens, T)
        qd = to_dev(q)
        ws = d.Workspace(len(bi) * T, hq, D, C)
        ref = to_host(d.attention_decode_multi(qd, kv, bi, T, lens, ws))
        got = to_host(d.attention_decode_multi_noalloc(qd, kv, bi, T, lens))
        assert_close(got, ref, ATTN_RTOL, ATTN_ATOL, f"no-alloc call {n + 1} vs workspace entry")
        oracle = oatt.attention_decode_multi(q, okv.bits_to_f64(kc, dtype), okv.bits_to_f64(vc, dtype), bi, T, lens)
        assert_close(got, oracle, ATTN_RTOL, ATTN_ATOL, f"no-alloc call {n + 1} vs oracle")
    d.device_error()


@pytest.mark.gpu
def test_no_alloc_at_its_limits_and_allocates_nothing(cuda_device):
    """The largest sequence table (256 sequences) and partials that fill the
    scratch exactly, each against the workspace entry and the oracle; after a
    first call (which may load kernels), a second call leaves the device's free
    memory unchanged."""
    import torch
    d = _dsb()
    rng = np.random.default_rng(7)
    n_max = 256
    lens256 = rng.integers(1, 257, n_max).astype(np.int32)
    # 18 tokens x 56 heads x 32 chunks x (128 + 2) x 4 bytes = 16 MiB - 4 KiB
    cap_lens = rng.integers(1, 4097, 18).astype(np.int32)
    cases = [
        (n_max, 8, 2, 256, 64, "f16", rng.permutation(n_max).astype(np.int32), lens256, 1),
        (18, 56, 8, 4096, 128, "bf16", rng.permutation(18).astype(np.int32), cap_lens, 1),
    ]
    for n, (F, hq, hkv, C, D, dtype, bi, lens, T) in enumerate(cases):
        kc, vc, q, kv = _case(10 + n, F, hq, hkv, C, D, dtype, bi, lens, T)
        qd = to_dev(q)
        ws = d.Workspace(len(bi) * T, hq, D, C)
        ref = to_host(d.attention_decode_multi(qd, kv, bi, T, lens, ws))
        out = torch.empty_like(qd)
        # torch's own fill kernel runs inside the measured window below; with
        # lazy module loading its first launch loads it into device memory,
        # so it runs once here first
        out.zero_()
        d.attention_decode_multi_noalloc(qd, kv, bi, T, lens, out=out)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        out.zero_()
        d.attention_decode_multi_noalloc(qd, kv, bi, T, lens, out=out)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, f"case {n}: free device memory moved by {free0 - free1} bytes across a call"
        got = to_host(out)
        assert_close(got, ref, ATTN_RTOL, ATTN_ATOL, f"no-alloc limit case {n} vs workspace entry")
        oracle = oatt.attention_decode_multi(q, okv.bits_to_f64(kc, dtype), okv.bits_to_f64(vc, dtype), bi, T, lens)
        assert_close(got, oracle, ATTN_RTOL, ATTN_ATOL, f"no-alloc limit case {n} vs oracle")
    d.device_error()


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    from session_decode_step_dsb_gb300 import build, dsb
    import os
    if not os.path.exists(dsb.LIB_PATH):
        build.build()
    lib = dsb.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    kv = dsb.KVCache(fake, fake, 0, 512, 1, 1 << 20, 128)
    bi = np.arange(300, dtype=np.int32)
    lens = np.full(300, 10, np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    st = lib.dsb_attention_decode_multi_noalloc(fake, 1, ctypes.byref(kv), bi.ctypes.data_as(p32), 300, 1,
                                                lens.ctypes.data_as(p32), fake, None)
    assert st == 2 and b"256" in lib.dsb_last_error()
    bi, lens = np.arange(8, dtype=np.int32), np.full(8, 1 << 20, np.int32)
    st = lib.dsb_attention_decode_multi_noalloc(fake, 64, ctypes.byref(kv), bi.ctypes.data_as(p32), 8, 1,
                                                lens.ctypes.data_as(p32), fake, None)
    assert st == 2 and b"scratch" in lib.dsb_last_error()
