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
