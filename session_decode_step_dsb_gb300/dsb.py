"""ctypes binding of libdsb.so (C ABI in include/dsb.h).

Argument marshalling only: tensors become device pointers, host index arrays
become int32 buffers, the current torch stream becomes the cudaStream_t.  Every
step of the computation runs in the library's CUDA kernels; if the library has
not been built the first call raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libdsb.so")

DSB_OK = 0
STATUS_NAMES = {0: "DSB_OK", 1: "DSB_ERR_INVALID_ARG", 2: "DSB_ERR_UNSUPPORTED", 3: "DSB_ERR_WORKSPACE",
                4: "DSB_ERR_CUDA", 5: "DSB_ERR_TIMEOUT", 6: "DSB_ERR_DEVICE"}
DSB_F16, DSB_BF16 = 0, 1
NARROW_MAX = 16
ATTN_CHUNK = 128
MAX_SEQS = 1024
MAX_TOKENS = 8192


class DsbError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Q8Mat(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class KVCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("full_batch_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("ctx", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_PI32 = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes); the names are exactly the exported C symbols.
SIGNATURES = {
    "dsb_last_error": (ctypes.c_char_p, []),
    "dsb_version": (ctypes.c_char_p, []),
    "dsb_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "dsb_workspace_create": (_I, [_P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "dsb_workspace_destroy": (_I, [_P]),
    "dsb_device_error": (_I, []),
    "dsb_quantize_q8_0": (_I, [_P, _I64, _I64, _P, _P]),
    "dsb_matmul_q8_0_narrow": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, _P]),
    "dsb_matmul_q8_0": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, _P]),
    "dsb_matmul_q8_0_block_dots": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, _P]),
    "dsb_rope_posvec": (_I, [_P, _I, _P, _I, _I, _I, _PI32, _F, _P, _P]),
    "dsb_kv_scatter": (_I, [ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P, _P]),
    "dsb_attention_decode_multi": (_I, [_P, _I, ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """Load libdsb.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdsb.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int):
    if status != DSB_OK:
        raise DsbError(status, lib().dsb_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _i32(a: Sequence[int]):
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(_PI32)


def version() -> str:
    return lib().dsb_version().decode()


def device_error():
    _check(lib().dsb_device_error())


class Workspace:
    """Caller-owned device scratch (a torch uint8 tensor) wrapped for the library."""

    def __init__(self, max_tokens: int, n_q_heads: int, head_dim: int, ctx: int, device=None):
        import torch
        nbytes = lib().dsb_workspace_bytes(max_tokens, n_q_heads, head_dim, ctx)
        if nbytes == 0:
            raise ValueError("workspace size arguments out of range")
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buffer.data_ptr()
        aligned = (base + 255) // 256 * 256
        handle = _P()
        _check(lib().dsb_workspace_create(_P(aligned), nbytes, ctypes.byref(handle)))
        self.handle = handle
        self.nbytes = nbytes

    def close(self):
        if getattr(self, "handle", None):
            lib().dsb_workspace_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q8_rows_bytes(cols: int) -> int:
    return cols // 32 * 34


def quantize_q8_0(x, xq=None, stream=None):
    """q8_0 bytes ``[n_rows, cols/32*34]`` (uint8, device) of float32 rows ``x``."""
    import torch
    n_rows, cols = x.shape
    if xq is None:
        xq = torch.empty((n_rows, q8_rows_bytes(cols)), dtype=torch.uint8, device=x.device)
    _check(lib().dsb_quantize_q8_0(_ptr(x), n_rows, cols, _ptr(xq), _stream(stream)))
    return xq


def _mat(w_blocks, rows: int, cols: int) -> Q8Mat:
    return Q8Mat(_ptr(w_blocks), rows, cols)


def matmul_q8_0_narrow(w_blocks, rows: int, cols: int, xq, n_tok: int, y=None, stream=None):
    """``y[n_tok, rows]`` float32 = q8_0 weights times q8_0 activations (n_tok <= 16)."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_narrow(ctypes.byref(m), _ptr(xq), n_tok, _ptr(y), _stream(stream)))
    return y


def matmul_q8_0(w_blocks, rows: int, cols: int, xq, n_tok: int, y=None, stream=None):
    """Same product for any n_tok (chunks of 16 through the narrow kernel)."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0(ctypes.byref(m), _ptr(xq), n_tok, _ptr(y), _stream(stream)))
    return y


def matmul_q8_0_block_dots(w_blocks, rows: int, cols: int, xq, n_tok: int, stream=None):
    """int32 ``isum[n_tok, rows, cols/32]`` through the narrow kernel's dp4a chain."""
    import torch
    isum = torch.empty((n_tok, rows, cols // 32), dtype=torch.int32, device=w_blocks.device)
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_block_dots(ctypes.byref(m), _ptr(xq), n_tok, _ptr(isum), _stream(stream)))
    return isum


def rope_posvec(q, k, pos, theta: float, ws: Workspace, stream=None):
    """In-place RoPE on ``q[n_tok, Hq, D]`` and ``k[n_tok, Hkv, D]`` (k may be None)."""
    n_tok, hq, d = q.shape
    hkv = 0 if k is None else k.shape[1]
    arr, p = _i32(pos)
    _check(lib().dsb_rope_posvec(_ptr(q), hq, _ptr(k), hkv, d, n_tok, p, float(theta), ws.handle, _stream(stream)))


def kv_cache(k_cache, v_cache, dtype: int) -> KVCache:
    f, hkv, ctx, d = k_cache.shape
    return KVCache(_ptr(k_cache), _ptr(v_cache), dtype, f, hkv, ctx, d)


def kv_scatter(kv: KVCache, batch_index, tokens_per_seq: int, pos, k, v, ws: Workspace, stream=None):
    bi, pbi = _i32(batch_index)
    ps, pp = _i32(pos)
    _check(lib().dsb_kv_scatter(ctypes.byref(kv), pbi, len(bi), tokens_per_seq, pp, _ptr(k), _ptr(v), ws.handle,
                                _stream(stream)))


def attention_decode_multi(q, kv: KVCache, batch_index, tokens_per_seq: int, seq_lens, ws: Workspace, out=None,
                           stream=None):
    import torch
    n_tok, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    bi, pbi = _i32(batch_index)
    sl, psl = _i32(seq_lens)
    _check(lib().dsb_attention_decode_multi(_ptr(q), hq, ctypes.byref(kv), pbi, len(bi), tokens_per_seq, psl,
                                            _ptr(out), ws.handle, _stream(stream)))
    return out
