"""Helpers for the GPU parity tests: tolerance checks and small wrappers.

The tolerances are the ones the method's acceptance states: matmul outputs
within 1e-3 relative with a 1e-4 absolute floor, attention outputs within
2e-3 relative (same floor); integer, byte and index results bit-exact.
"""
from __future__ import annotations

import numpy as np

MATMUL_RTOL, MATMUL_ATOL = 1e-3, 1e-4
ATTN_RTOL, ATTN_ATOL = 2e-3, 1e-4
# RoPE: float32 rotation of float32 inputs against a float64 reference; the
# error is a few float32 ulps of the pair's magnitude.
ROPE_RTOL, ROPE_ATOL = 1e-5, 1e-5


def assert_close(got, ref, rtol, atol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = np.maximum(rtol * np.abs(ref), atol)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (rtol={rtol}, atol={atol})")


def to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    return t.detach().cpu().numpy()


def assert_q8_close(got, want, what="", code_frac=2e-3, scale_frac=1e-2):
    """q8_0 rows from a float32 GPU stage against the oracle's float64 stage,
    both quantised by the same codec from the same float32 inputs.

    The two values entering the codec differ by a few float32 ulps (relative
    delta ~ 1e-6), so a code can only differ where x/d lies within ~127*delta
    of a rounding boundary (a fraction ~1e-4), and then by exactly one step;
    an fp16 scale can only differ at an fp16 rounding boundary (a fraction
    ~2^11 * delta ~ 2e-3), and then by one fp16 ulp.  A wrong computation
    (eps, weight, row, head) moves nearly every code.  Checked: every code
    within one step, every scale within one fp16 ulp, and the fractions that
    differ at all below code_frac / scale_frac."""
    from oracle import q8_0 as oq
    got = np.ascontiguousarray(got, dtype=np.uint8)
    want = np.ascontiguousarray(want, dtype=np.uint8)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    cg, sg = oq.unpack(got)
    cw, sw = oq.unpack(want)
    dc = np.abs(cg.astype(np.int32) - cw.astype(np.int32))
    ds = np.abs(sg.view(np.uint16).astype(np.int32) - sw.view(np.uint16).astype(np.int32))
    assert dc.max() <= 1, f"{what}: a code differs by {dc.max()} steps"
    assert ds.max() <= 1, f"{what}: a scale differs by {ds.max()} fp16 ulps"
    assert np.mean(dc != 0) <= code_frac, f"{what}: {np.mean(dc != 0):.2e} of the codes differ"
    assert np.mean(ds != 0) <= scale_frac, f"{what}: {np.mean(ds != 0):.2e} of the scales differ"
