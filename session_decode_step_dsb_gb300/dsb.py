"""ctypes binding of libdsb.so (C ABI in include/dsb.h).

Argument marshalling only: tensors become device pointers, host index arrays
become int32 buffers, the current torch stream becomes the cudaStream_t.  Since
the C ABI sees bare pointers, the binding first checks that every tensor holds
the bytes and element type the call will touch and that every host array has
the call's length (ValueError otherwise).  Every step of the computation runs
in the library's CUDA kernels; if the library has not been built the first call
raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional, Sequence

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libdsb.so")

DSB_OK = 0
DSB_ERR_INVALID_ARG = 1
DSB_ERR_UNSUPPORTED = 2
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


class KVPages(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int), ("n_pages", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class RopeC(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_float), ("yarn_factor", ctypes.c_float), ("yarn_orig_ctx", ctypes.c_int32),
                ("yarn_beta_fast", ctypes.c_float), ("yarn_beta_slow", ctypes.c_float)]


class Yarn(NamedTuple):
    """YaRN RoPE parameters: scale ``factor`` > 1 over the original context
    ``orig_ctx``, ramp bounds ``beta_fast`` / ``beta_slow`` (rotation counts)."""
    factor: float
    orig_ctx: int
    beta_fast: float = 32.0
    beta_slow: float = 1.0


def rope_params(theta: float, yarn=None) -> RopeC:
    """``dsb_rope`` for the plain RoPE (``yarn`` None) or YaRN (any object with
    ``factor, orig_ctx, beta_fast, beta_slow``)."""
    if yarn is None:
        return RopeC(float(theta), 0.0, 0, 0.0, 0.0)
    return RopeC(float(theta), float(yarn.factor), int(yarn.orig_ctx), float(yarn.beta_fast), float(yarn.beta_slow))


KV_PAGE = 128

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
    "dsb_matmul_q8_0_staged_bytes": (ctypes.c_size_t, [_I, _I64]),
    "dsb_stage_q8_0": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, ctypes.c_size_t, _P]),
    "dsb_matmul_q8_0_staged": (_I, [ctypes.POINTER(Q8Mat), _P, ctypes.c_size_t, _I, _P, _P]),
    "dsb_matmul_q8_0_wide_scratch_bytes": (ctypes.c_size_t, [_I, _I64]),
    "dsb_matmul_q8_0_wide": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, _P, ctypes.c_size_t, _P]),
    "dsb_rope_posvec": (_I, [_P, _I, _P, _I, _I, _I, _PI32, _F, _P, _P]),
    "dsb_head_rmsnorm_rope": (_I, [_P, _I, _P, _I, _I, _I, _PI32, _P, _P, _P, _F, _P, _P]),
    "dsb_rmsnorm_matmul_q8_0": (_I, [ctypes.POINTER(Q8Mat), _P, _P, _F, _I, _P, _P]),
    "dsb_silu_matmul_q8_0": (_I, [ctypes.POINTER(Q8Mat), _P, _I, _P, _P]),
    "dsb_kv_scatter": (_I, [ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P, _P]),
    "dsb_attention_decode_multi": (_I, [_P, _I, ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P]),
    "dsb_attention_decode_multi_noalloc": (_I, [_P, _I, ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P]),
    "dsb_attention_decode_multi_q8_0": (_I, [_P, _I, ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P]),
    "dsb_rmsnorm_q8_0": (_I, [_P, _P, _I, _I, _F, _P, _P]),
    "dsb_kv_scatter_paged": (_I, [ctypes.POINTER(KVPages), _PI32, _I, _PI32, _PI32, _I, _I, _PI32, _P, _P, _P, _P]),
    "dsb_attention_decode_paged": (_I, [_P, _I, ctypes.POINTER(KVPages), _PI32, _I, _PI32, _PI32, _I, _I, _PI32, _P,
                                        _P, _P]),
    "dsb_silu_mul_q8_0": (_I, [_P, _I, _I, _P, _P]),
    "dsb_embed_q8_0": (_I, [_P, _I, _I, _PI32, _I, _P, _P, _P]),
    "dsb_rope_kv_write": (_I, [_P, _I, ctypes.POINTER(KVCache), _PI32, _I, _I, _PI32, _P, _P, _P, _F, _P, _P]),
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


def _i32(a: Sequence[int], n: Optional[int] = None, name: str = "array"):
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32)).reshape(-1)
    if n is not None and arr.size != n:
        raise ValueError(f"{name} has {arr.size} entries, needs {n}")
    return arr, arr.ctypes.data_as(_PI32)


def _need(t, nbytes: int, name: str, kind: Optional[str] = None):
    """Checks, before any pointer reaches the library, that tensor ``t`` holds
    at least ``nbytes`` bytes of the expected kind ("f32", "u8" or "16": any
    16-bit type): the C ABI sees bare pointers, so a short buffer would be read
    or written past its end on the device."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if kind == "f32" and t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32, got {t.dtype}")
    if kind == "u8" and t.dtype != torch.uint8:
        raise ValueError(f"{name} must be uint8 (q8_0 bytes), got {t.dtype}")
    if kind == "16" and t.element_size() != 2:
        raise ValueError(f"{name} must have a 16-bit element type, got {t.dtype}")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, needs {nbytes}")


def _need_opt(t, nbytes: int, name: str, kind: Optional[str] = None):
    if t is not None:
        _need(t, nbytes, name, kind)


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
    _need(x, 4 * n_rows * cols, "x", "f32")
    if xq is None:
        xq = torch.empty((n_rows, q8_rows_bytes(cols)), dtype=torch.uint8, device=x.device)
    _need(xq, n_rows * q8_rows_bytes(cols), "xq", "u8")
    _check(lib().dsb_quantize_q8_0(_ptr(x), n_rows, cols, _ptr(xq), _stream(stream)))
    return xq


def _mat(w_blocks, rows: int, cols: int, name: str = "w_blocks") -> Q8Mat:
    _need(w_blocks, rows * q8_rows_bytes(cols), name, "u8")
    return Q8Mat(_ptr(w_blocks), rows, cols)


def _mm_io(rows: int, cols: int, xq, n_tok: int, y):
    _need(xq, n_tok * q8_rows_bytes(cols), "xq", "u8")
    _need(y, 4 * n_tok * rows, "y", "f32")


def matmul_q8_0_narrow(w_blocks, rows: int, cols: int, xq, n_tok: int, y=None, stream=None):
    """``y[n_tok, rows]`` float32 = q8_0 weights times q8_0 activations (n_tok <= 16)."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    _mm_io(rows, cols, xq, n_tok, y)
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_narrow(ctypes.byref(m), _ptr(xq), n_tok, _ptr(y), _stream(stream)))
    return y


def matmul_q8_0(w_blocks, rows: int, cols: int, xq, n_tok: int, y=None, stream=None):
    """Same product for any n_tok (chunks of 16 through the narrow kernel)."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    _mm_io(rows, cols, xq, n_tok, y)
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0(ctypes.byref(m), _ptr(xq), n_tok, _ptr(y), _stream(stream)))
    return y


def matmul_q8_0_block_dots(w_blocks, rows: int, cols: int, xq, n_tok: int, stream=None):
    """int32 ``isum[n_tok, rows, cols/32]`` through the narrow kernel's dp4a chain."""
    import torch
    isum = torch.empty((n_tok, rows, cols // 32), dtype=torch.int32, device=w_blocks.device)
    _need(xq, n_tok * q8_rows_bytes(cols), "xq", "u8")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_block_dots(ctypes.byref(m), _ptr(xq), n_tok, _ptr(isum), _stream(stream)))
    return isum


def stage_q8_0(w_blocks, rows: int, cols: int, xq, n_tok: int, staged=None, stream=None):
    """The staged activation layout of ``xq`` that the narrow kernel reads at
    ``n_tok`` tokens (uint8 device tensor, allocated when not given)."""
    import torch
    nbytes = lib().dsb_matmul_q8_0_staged_bytes(n_tok, cols)
    if nbytes == 0:
        raise DsbError(DSB_ERR_INVALID_ARG, f"no staged layout for n_tok={n_tok}, cols={cols}")
    if staged is None:
        staged = torch.empty(nbytes, dtype=torch.uint8, device=w_blocks.device)
    _need(xq, n_tok * q8_rows_bytes(cols), "xq", "u8")
    _need(staged, nbytes, "staged", "u8")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_stage_q8_0(ctypes.byref(m), _ptr(xq), n_tok, _ptr(staged), staged.numel(), _stream(stream)))
    return staged


def matmul_q8_0_staged(w_blocks, rows: int, cols: int, staged, n_tok: int, y=None, stream=None):
    """``y[n_tok, rows]`` from activations staged by :func:`stage_q8_0` (the
    decode step's matmul path); bitwise :func:`matmul_q8_0_narrow`."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    _need(y, 4 * n_tok * rows, "y", "f32")
    _need(staged, 0, "staged", "u8")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_staged(ctypes.byref(m), _ptr(staged), staged.numel(), n_tok, _ptr(y),
                                        _stream(stream)))
    return y


def _wide_scratch(n_tok: int, cols: int, device):
    import torch
    nbytes = lib().dsb_matmul_q8_0_wide_scratch_bytes(n_tok, cols)
    if nbytes == 0:
        raise DsbError(DSB_ERR_UNSUPPORTED, f"no wide-matmul scratch size for n_tok={n_tok}, cols={cols}")
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def matmul_q8_0_wide(w_blocks, rows: int, cols: int, xq, n_tok: int, y=None, scratch=None, stream=None):
    """Same product on the tensor cores (any n_tok; cols % 256 == 0).  ``scratch``
    (uint8 device tensor) is allocated when not given."""
    import torch
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=w_blocks.device)
    if scratch is None:
        scratch, _ = _wide_scratch(n_tok, cols, w_blocks.device)
    _mm_io(rows, cols, xq, n_tok, y)
    _need(scratch, 0, "scratch", "u8")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_matmul_q8_0_wide(ctypes.byref(m), _ptr(xq), n_tok, _ptr(y), _ptr(scratch), scratch.numel(),
                                      _stream(stream)))
    return y


def rmsnorm_matmul_q8_0(w_blocks, rows: int, cols: int, x, norm_w, eps: float, y=None, stream=None):
    """``y[n_tok, rows] = W q8(rmsnorm(x) * norm_w)`` in one kernel (x float32 ``[n_tok, cols]``)."""
    import torch
    n_tok = x.shape[0]
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=x.device)
    _need(x, 4 * n_tok * cols, "x", "f32")
    _need_opt(norm_w, 4 * cols, "norm_w", "f32")
    _need(y, 4 * n_tok * rows, "y", "f32")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_rmsnorm_matmul_q8_0(ctypes.byref(m), _ptr(x), _ptr(norm_w), float(eps), n_tok, _ptr(y),
                                         _stream(stream)))
    return y


def silu_matmul_q8_0(w_blocks, rows: int, cols: int, gu, y=None, stream=None):
    """``y[n_tok, rows] = W q8(silu(gate) * up)`` in one kernel (gu float32 ``[n_tok, 2 cols]``)."""
    import torch
    n_tok = gu.shape[0]
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=gu.device)
    _need(gu, 8 * n_tok * cols, "gu", "f32")
    _need(y, 4 * n_tok * rows, "y", "f32")
    m = _mat(w_blocks, rows, cols)
    _check(lib().dsb_silu_matmul_q8_0(ctypes.byref(m), _ptr(gu), n_tok, _ptr(y), _stream(stream)))
    return y


def rope_posvec(q, k, pos, theta: float, ws: Workspace, stream=None):
    """In-place RoPE on ``q[n_tok, Hq, D]`` and ``k[n_tok, Hkv, D]`` (k may be None)."""
    n_tok, hq, d = q.shape
    hkv = 0 if k is None else k.shape[1]
    _need(q, 4 * n_tok * hq * d, "q", "f32")
    _need_opt(k, 4 * n_tok * hkv * d, "k", "f32")
    arr, p = _i32(pos, n_tok, "pos")
    _check(lib().dsb_rope_posvec(_ptr(q), hq, _ptr(k), hkv, d, n_tok, p, float(theta), ws.handle, _stream(stream)))


def head_rmsnorm_rope(q, k, pos, theta: float, q_norm, k_norm, eps: float, ws: Workspace, stream=None, yarn=None):
    """In place: per-head RMS norm (weights ``q_norm, k_norm`` float32 ``[D]``,
    either may be None) then RoPE (plain, or YaRN with ``yarn``) on
    ``q[n_tok, Hq, D]`` and ``k[n_tok, Hkv, D]``."""
    n_tok, hq, d = q.shape
    hkv = 0 if k is None else k.shape[1]
    _need(q, 4 * n_tok * hq * d, "q", "f32")
    _need_opt(k, 4 * n_tok * hkv * d, "k", "f32")
    _need_opt(q_norm, 4 * d, "q_norm", "f32")
    _need_opt(k_norm, 4 * d, "k_norm", "f32")
    arr, p = _i32(pos, n_tok, "pos")
    r = rope_params(theta, yarn)
    _check(lib().dsb_head_rmsnorm_rope(_ptr(q), hq, _ptr(k), hkv, d, n_tok, p, ctypes.byref(r), _ptr(q_norm),
                                       _ptr(k_norm), float(eps), ws.handle, _stream(stream)))


def attention_decode_multi_noalloc(q, kv: KVCache, batch_index, tokens_per_seq: int, seq_lens, out=None,
                                   stream=None):
    """Same as :func:`attention_decode_multi` without a workspace: for callers
    that cannot allocate device memory (the library's static scratch is used;
    calls that overlap on the GPU must be serialised)."""
    import torch
    if out is None:
        out = torch.empty_like(q)
    bi, pbi = _i32(batch_index)
    sl, psl = _i32(seq_lens, bi.size, "seq_lens")
    _attn_io(q, kv.head_dim, bi.size * tokens_per_seq, out)
    _check(lib().dsb_attention_decode_multi_noalloc(_ptr(q), q.shape[1], ctypes.byref(kv), pbi, len(bi),
                                                    tokens_per_seq, psl, _ptr(out), _stream(stream)))
    return out


def kv_cache(k_cache, v_cache, dtype: int) -> KVCache:
    """Describe device caches ``[F, Hkv, ctx, D]``; the returned struct keeps
    the two tensors alive for as long as it lives."""
    f, hkv, ctx, d = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache shapes differ")
    _need(k_cache, 2 * f * hkv * ctx * d, "k_cache", "16")
    _need(v_cache, 2 * f * hkv * ctx * d, "v_cache", "16")
    kv = KVCache(_ptr(k_cache), _ptr(v_cache), dtype, f, hkv, ctx, d)
    kv._tensors = (k_cache, v_cache)
    return kv


def _attn_io(q, head_dim: int, n_tok: int, out, out_kind: str = "f32"):
    """q float32 [n_tok, Hq, head_dim]; out the same size."""
    if q.dim() != 3 or q.shape[0] != n_tok or q.shape[2] != head_dim:
        raise ValueError(f"q must be [n_seq*T={n_tok}, Hq, head_dim={head_dim}], got {tuple(q.shape)}")
    _need(q, 4 * q.numel(), "q", "f32")
    if out_kind == "f32":
        _need(out, 4 * q.numel(), "out", "f32")


def kv_scatter(kv: KVCache, batch_index, tokens_per_seq: int, pos, k, v, ws: Workspace, stream=None):
    bi, pbi = _i32(batch_index)
    n_tok = bi.size * tokens_per_seq
    ps, pp = _i32(pos, n_tok, "pos")
    _need(k, 4 * n_tok * kv.n_kv_heads * kv.head_dim, "k", "f32")
    _need(v, 4 * n_tok * kv.n_kv_heads * kv.head_dim, "v", "f32")
    _check(lib().dsb_kv_scatter(ctypes.byref(kv), pbi, len(bi), tokens_per_seq, pp, _ptr(k), _ptr(v), ws.handle,
                                _stream(stream)))


def attention_decode_multi(q, kv: KVCache, batch_index, tokens_per_seq: int, seq_lens, ws: Workspace, out=None,
                           stream=None):
    import torch
    n_tok, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    bi, pbi = _i32(batch_index)
    sl, psl = _i32(seq_lens, bi.size, "seq_lens")
    _attn_io(q, kv.head_dim, bi.size * tokens_per_seq, out)
    _check(lib().dsb_attention_decode_multi(_ptr(q), hq, ctypes.byref(kv), pbi, len(bi), tokens_per_seq, psl,
                                            _ptr(out), ws.handle, _stream(stream)))
    return out


def attention_decode_multi_q8_0(q, kv: KVCache, batch_index, tokens_per_seq: int, seq_lens, ws: Workspace,
                                stream=None):
    """The attention with its rows q8_0-quantised: uint8 ``[n_tok, Hq*D/32*34]``."""
    import torch
    n_tok, hq, d = q.shape
    xq = torch.empty((n_tok, hq * d // 32 * 34), dtype=torch.uint8, device=q.device)
    bi, pbi = _i32(batch_index)
    sl, psl = _i32(seq_lens, bi.size, "seq_lens")
    _attn_io(q, kv.head_dim, bi.size * tokens_per_seq, None, out_kind="none")
    _check(lib().dsb_attention_decode_multi_q8_0(_ptr(q), hq, ctypes.byref(kv), pbi, len(bi), tokens_per_seq, psl,
                                                 _ptr(xq), ws.handle, _stream(stream)))
    return xq


def kv_pages(k_pool, v_pool, dtype: int) -> KVPages:
    """Describe device page pools ``[n_pages, Hkv, 128, D]``; the returned struct
    keeps the two tensors alive for as long as it lives."""
    n_pages, hkv, page, d = k_pool.shape
    if page != KV_PAGE:
        raise ValueError("pages hold 128 keys")
    if tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("k_pool and v_pool shapes differ")
    _need(k_pool, 2 * k_pool.numel(), "k_pool", "16")
    _need(v_pool, 2 * v_pool.numel(), "v_pool", "16")
    kv = KVPages(_ptr(k_pool), _ptr(v_pool), dtype, n_pages, hkv, d)
    kv._tensors = (k_pool, v_pool)
    return kv


def _geometry(block_table, n_blocks, window):
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2:
        raise ValueError("block_table is [n_seq, max_blocks]")
    nb, pnb = _i32(n_blocks, bt.shape[0], "n_blocks")
    win, pwin = _i32(window, bt.shape[0], "window")
    return bt, bt.ctypes.data_as(_PI32), nb, pnb, win, pwin


def kv_scatter_paged(kv: KVPages, block_table, n_blocks, window, tokens_per_seq: int, pos, k, v, ws: Workspace,
                     stream=None):
    bt, pbt, nb, pnb, win, pwin = _geometry(block_table, n_blocks, window)
    n_tok = bt.shape[0] * tokens_per_seq
    ps, pp = _i32(pos, n_tok, "pos")
    _need(k, 4 * n_tok * kv.n_kv_heads * kv.head_dim, "k", "f32")
    _need(v, 4 * n_tok * kv.n_kv_heads * kv.head_dim, "v", "f32")
    _check(lib().dsb_kv_scatter_paged(ctypes.byref(kv), pbt, bt.shape[1], pnb, pwin, bt.shape[0], tokens_per_seq, pp,
                                      _ptr(k), _ptr(v), ws.handle, _stream(stream)))


def attention_decode_paged(q, kv: KVPages, block_table, n_blocks, window, tokens_per_seq: int, seq_lens,
                           ws: Workspace, out=None, stream=None):
    import torch
    n_tok, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    bt, pbt, nb, pnb, win, pwin = _geometry(block_table, n_blocks, window)
    sl, psl = _i32(seq_lens, bt.shape[0], "seq_lens")
    _attn_io(q, kv.head_dim, bt.shape[0] * tokens_per_seq, out)
    _check(lib().dsb_attention_decode_paged(_ptr(q), hq, ctypes.byref(kv), pbt, bt.shape[1], pnb, pwin, bt.shape[0],
                                            tokens_per_seq, psl, _ptr(out), ws.handle, _stream(stream)))
    return out


def rmsnorm_q8_0(x, w, eps: float, stream=None):
    """q8_0 ``[n_tok, hidden/32*34]`` of the RMS-normed rows of ``x``."""
    import torch
    n_tok, hidden = x.shape
    _need(x, 4 * n_tok * hidden, "x", "f32")
    _need(w, 4 * hidden, "w", "f32")
    xq = torch.empty((n_tok, hidden // 32 * 34), dtype=torch.uint8, device=x.device)
    _check(lib().dsb_rmsnorm_q8_0(_ptr(x), _ptr(w), n_tok, hidden, float(eps), _ptr(xq), _stream(stream)))
    return xq


def silu_mul_q8_0(gu, stream=None):
    """q8_0 of silu(gate) * up for ``gu[n_tok, 2*ffn]`` = [gate | up]."""
    import torch
    n_tok, two_ffn = gu.shape
    ffn = two_ffn // 2
    _need(gu, 4 * gu.numel(), "gu", "f32")
    xq = torch.empty((n_tok, ffn // 32 * 34), dtype=torch.uint8, device=gu.device)
    _check(lib().dsb_silu_mul_q8_0(_ptr(gu), n_tok, ffn, _ptr(xq), _stream(stream)))
    return xq


def embed_q8_0(table, vocab: int, hidden: int, token_ids, ws: Workspace, stream=None):
    """float32 ``[n_tok, hidden]``: dequantised embedding rows of the tokens."""
    import torch
    tk, ptk = _i32(token_ids)
    _need(table, vocab * q8_rows_bytes(hidden), "table", "u8")
    h = torch.empty((len(tk), hidden), dtype=torch.float32, device=table.device)
    _check(lib().dsb_embed_q8_0(_ptr(table), vocab, hidden, ptk, len(tk), _ptr(h), ws.handle, _stream(stream)))
    return h


def rope_kv_write(qkv, n_q_heads: int, kv: KVCache, batch_index, tokens_per_seq: int, pos, theta: float,
                  ws: Workspace, stream=None, q_norm=None, k_norm=None, eps: float = 0.0, yarn=None):
    """Fused (optional per-head RMS norm +) RoPE + KV write on
    ``qkv[n_tok, (Hq + 2 Hkv) * D]`` (q rotated in place)."""
    bi, pbi = _i32(batch_index)
    n_tok = bi.size * tokens_per_seq
    ps, pp = _i32(pos, n_tok, "pos")
    _need(qkv, 4 * n_tok * (n_q_heads + 2 * kv.n_kv_heads) * kv.head_dim, "qkv", "f32")
    _need_opt(q_norm, 4 * kv.head_dim, "q_norm", "f32")
    _need_opt(k_norm, 4 * kv.head_dim, "k_norm", "f32")
    r = rope_params(theta, yarn)
    _check(lib().dsb_rope_kv_write(_ptr(qkv), n_q_heads, ctypes.byref(kv), pbi, len(bi), tokens_per_seq, pp,
                                   ctypes.byref(r), _ptr(q_norm), _ptr(k_norm), float(eps), ws.handle,
                                   _stream(stream)))
    return qkv


# ---------------------------------------------------------------- decode step
class ModelShapeC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope", RopeC)]


class LayerC(ctypes.Structure):
    _fields_ = [("wqkv", Q8Mat), ("wo", Q8Mat), ("wgu", Q8Mat), ("wdown", Q8Mat), ("attn_norm", ctypes.c_void_p),
                ("ffn_norm", ctypes.c_void_p), ("kv", KVCache), ("q_norm", ctypes.c_void_p),
                ("k_norm", ctypes.c_void_p)]


class ModelC(ctypes.Structure):
    _fields_ = [("shape", ModelShapeC), ("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerC)),
                ("final_norm", ctypes.c_void_p), ("head", Q8Mat)]


class LayerTraceC(ctypes.Structure):
    _fields_ = [("x_attn", ctypes.c_void_p), ("qkv", ctypes.c_void_p), ("qkv_rope", ctypes.c_void_p),
                ("att_q8", ctypes.c_void_p), ("h_attn", ctypes.c_void_p), ("x_ffn", ctypes.c_void_p),
                ("gu", ctypes.c_void_p), ("act_q8", ctypes.c_void_p), ("h_out", ctypes.c_void_p)]


class StepTraceC(ctypes.Structure):
    _fields_ = [("h_embed", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerTraceC)), ("x_final", ctypes.c_void_p)]


SIGNATURES.update({
    "dsb_probe_dp4a": (_I, [_I, _I, _I, _P, _P]),
    "dsb_probe_mma": (_I, [_I, _I, _I, _P, _P]),
    "dsb_step_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(ModelShapeC), _I, _I]),
    "dsb_decode_step": (_I, [ctypes.POINTER(ModelC), _PI32, _PI32, _I, _I, _PI32, _P, _P, _P]),
    "dsb_decode_step_paged": (_I, [ctypes.POINTER(ModelC), ctypes.POINTER(KVPages), _PI32, _I, _I, _PI32, _PI32, _I,
                                   _PI32, _PI32, _P, _P, _P]),
    "dsb_decode_step_trace": (_I, [ctypes.POINTER(ModelC), _PI32, _PI32, _I, _I, _PI32, _P, _P,
                                   ctypes.POINTER(StepTraceC), _P]),
    "dsb_step_graph_create": (_I, [ctypes.POINTER(ModelC), _I, _I, _P, _P, _P, ctypes.POINTER(_P)]),
    "dsb_step_graph_launch": (_I, [_P, _PI32, _PI32, _PI32, _P]),
    "dsb_step_graph_create_paged": (_I, [ctypes.POINTER(ModelC), ctypes.POINTER(KVPages), _I, _I, _I, _P, _P, _P,
                                         ctypes.POINTER(_P)]),
    "dsb_step_graph_launch_paged": (_I, [_P, _PI32, _PI32, _PI32, _PI32, _PI32, _P]),
    "dsb_step_graph_destroy": (_I, [_P]),
    "dsb_batch_former_create": (_I, [_I, _I, _I, ctypes.POINTER(_P)]),
    "dsb_batch_former_destroy": (None, [_P]),
    "dsb_batch_join": (_I, [_P, _I, _PI32]),
    "dsb_batch_leave": (_I, [_P, _I]),
    "dsb_batch_submit": (_I, [_P, _I, _PI32]),
    "dsb_batch_form": (_I, [_P, _PI32, _PI32, _PI32, _PI32]),
    "dsb_batch_commit": (_I, [_P, _PI32, _I]),
    "dsb_batch_length": (_I, [_P, _I]),
})


def probe_dp4a(mode: int, blocks: int, iters: int, out, stream=None):
    """The dp4a rate (mode 0) / latency (mode 1) probe; ``out`` device uint32[3]."""
    _need(out, 12, "out")
    _check(lib().dsb_probe_dp4a(mode, blocks, iters, _ptr(out), _stream(stream)))
    return out


def probe_mma(mode: int, blocks: int, iters: int, out, stream=None):
    """The mma.sync rate probe (mode 2: m16n8k16 f16, mode 3: m16n8k32 s8);
    ``out`` device uint32[1]."""
    _need(out, 4, "out")
    _check(lib().dsb_probe_mma(mode, blocks, iters, _ptr(out), _stream(stream)))
    return out


class BatchFormer:
    """Slot hand-out and per-step metadata for a live batch (host only)."""

    def __init__(self, full_batch_size: int, ctx: int, tokens_per_seq: int = 1):
        h = _P()
        _check(lib().dsb_batch_former_create(full_batch_size, ctx, tokens_per_seq, ctypes.byref(h)))
        self.handle, self.F, self.T = h, full_batch_size, tokens_per_seq

    def join(self, prefill_length: int) -> int:
        slot = ctypes.c_int32()
        _check(lib().dsb_batch_join(self.handle, prefill_length, ctypes.byref(slot)))
        return slot.value

    def leave(self, slot: int):
        _check(lib().dsb_batch_leave(self.handle, slot))

    def submit(self, slot: int, token_ids):
        arr, p = _i32(token_ids)
        if arr.size != self.T:
            raise ValueError("one token id per draft token")
        _check(lib().dsb_batch_submit(self.handle, slot, p))

    def form(self):
        bi = np.zeros(self.F, np.int32)
        sl = np.zeros(self.F, np.int32)
        tk = np.zeros(self.F * self.T, np.int32)
        n = ctypes.c_int32()
        _check(lib().dsb_batch_form(self.handle, bi.ctypes.data_as(_PI32), sl.ctypes.data_as(_PI32),
                                    tk.ctypes.data_as(_PI32), ctypes.byref(n)))
        k = n.value
        return bi[:k].copy(), sl[:k].copy(), tk[:k * self.T].copy()

    def commit(self, batch_index):
        arr, p = _i32(batch_index)
        _check(lib().dsb_batch_commit(self.handle, p, arr.size))

    def length(self, slot: int) -> int:
        return lib().dsb_batch_length(self.handle, slot)

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                lib().dsb_batch_former_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


class StepWorkspace(Workspace):
    """Workspace sized for decode steps of up to ``max_tokens`` rows."""

    def __init__(self, shape: ModelShapeC, max_tokens: int, ctx: int, device=None):
        import torch
        nbytes = lib().dsb_step_workspace_bytes(ctypes.byref(shape), max_tokens, ctx)
        if nbytes == 0:
            raise ValueError("step workspace size arguments out of range")
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        aligned = (self.buffer.data_ptr() + 255) // 256 * 256
        handle = _P()
        _check(lib().dsb_workspace_create(_P(aligned), nbytes, ctypes.byref(handle)))
        self.handle = handle
        self.nbytes = nbytes


class DecodeModel:
    """Device tensors of a llama-style q8_0 model plus its retained KV caches,
    described to the library as a ``dsb_model``.

    ``weights`` maps names to *device* tensors: q8_0 byte matrices ``embed,
    head`` and per-layer lists ``wqkv, wo, wgu, wdown``; float32 ``final_norm``
    and per-layer ``attn_norm, ffn_norm`` (optionally per-layer ``q_norm,
    k_norm`` of width D: the per-head RMS norm before the rope).
    ``k_caches / v_caches`` are per-layer device tensors ``[F, Hkv, ctx, D]``
    of a 16-bit dtype.
    """

    def __init__(self, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, n_layers, weights, k_caches, v_caches,
                 cache_dtype: int, rms_eps=1e-6, rope_theta=10000.0, yarn=None):
        self.shape = ModelShapeC(hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, n_layers, rms_eps,
                                 rope_params(rope_theta, yarn))
        self.w = weights
        self.k_caches, self.v_caches = k_caches, v_caches
        qkv_rows = (n_q_heads + 2 * n_kv_heads) * head_dim
        layers = (LayerC * n_layers)()
        for l in range(n_layers):
            layers[l].wqkv = _mat(weights["wqkv"][l], qkv_rows, hidden, f"wqkv[{l}]")
            layers[l].wo = _mat(weights["wo"][l], hidden, n_q_heads * head_dim, f"wo[{l}]")
            layers[l].wgu = _mat(weights["wgu"][l], 2 * ffn, hidden, f"wgu[{l}]")
            layers[l].wdown = _mat(weights["wdown"][l], hidden, ffn, f"wdown[{l}]")
            _need(weights["attn_norm"][l], 4 * hidden, f"attn_norm[{l}]", "f32")
            _need(weights["ffn_norm"][l], 4 * hidden, f"ffn_norm[{l}]", "f32")
            if tuple(k_caches[l].shape[1:]) != (k_caches[0].shape[1], k_caches[0].shape[2], head_dim) or \
                    k_caches[l].shape[1] != n_kv_heads:
                raise ValueError(f"k_caches[{l}] must be [F, n_kv_heads={n_kv_heads}, ctx, head_dim={head_dim}]")
            layers[l].attn_norm = _ptr(weights["attn_norm"][l])
            layers[l].ffn_norm = _ptr(weights["ffn_norm"][l])
            layers[l].kv = kv_cache(k_caches[l], v_caches[l], cache_dtype)
            if "q_norm" in weights:
                _need(weights["q_norm"][l], 4 * head_dim, f"q_norm[{l}]", "f32")
                layers[l].q_norm = _ptr(weights["q_norm"][l])
            if "k_norm" in weights:
                _need(weights["k_norm"][l], 4 * head_dim, f"k_norm[{l}]", "f32")
                layers[l].k_norm = _ptr(weights["k_norm"][l])
        self._layers = layers
        _need(weights["embed"], vocab * q8_rows_bytes(hidden), "embed", "u8")
        _need(weights["final_norm"], 4 * hidden, "final_norm", "f32")
        self.c = ModelC(self.shape, _ptr(weights["embed"]), layers, _ptr(weights["final_norm"]),
                        _mat(weights["head"], vocab, hidden, "head"))
        self.vocab = vocab
        self.ctx = k_caches[0].shape[2]
        self.full_batch_size = k_caches[0].shape[0]

    def workspace(self, max_tokens: int) -> StepWorkspace:
        return StepWorkspace(self.shape, max_tokens, self.ctx)

    def step(self, token_ids, batch_index, tokens_per_seq: int, seq_lens, ws: Workspace, logits=None, stream=None):
        import torch
        n_seq = len(batch_index)
        if logits is None:
            logits = torch.empty((n_seq * tokens_per_seq, self.vocab), dtype=torch.float32, device="cuda")
        _need(logits, 4 * n_seq * tokens_per_seq * self.vocab, "logits", "f32")
        tk, ptk = _i32(token_ids, n_seq * tokens_per_seq, "token_ids")
        bi, pbi = _i32(batch_index)
        sl, psl = _i32(seq_lens, n_seq, "seq_lens")
        _check(lib().dsb_decode_step(ctypes.byref(self.c), ptk, pbi, n_seq, tokens_per_seq, psl, _ptr(logits),
                                     ws.handle, _stream(stream)))
        return logits

    def step_paged(self, pages, token_ids, tokens_per_seq: int, seq_lens, block_table, n_blocks, window,
                   ws: Workspace, logits=None, stream=None):
        """The step on page pools (dsb_decode_step_paged): ``pages`` is one
        ``KVPages`` per layer (see ``kv_pages``); the block geometry is
        ``block_table [n_seq][max_blocks]``, ``n_blocks`` and ``window``
        (host int32, as ``attention_decode_paged``)."""
        import torch
        if len(pages) != self.shape.n_layers:
            raise ValueError(f"pages: one pool per layer ({self.shape.n_layers}), got {len(pages)}")
        bt, pbt, nb, pnb, win, pwin = _geometry(block_table, n_blocks, window)
        n_seq = bt.shape[0]
        if logits is None:
            logits = torch.empty((n_seq * tokens_per_seq, self.vocab), dtype=torch.float32, device="cuda")
        _need(logits, 4 * n_seq * tokens_per_seq * self.vocab, "logits", "f32")
        tk, ptk = _i32(token_ids, n_seq * tokens_per_seq, "token_ids")
        sl, psl = _i32(seq_lens, n_seq, "seq_lens")
        arr = (KVPages * len(pages))(*pages)
        _check(lib().dsb_decode_step_paged(ctypes.byref(self.c), arr, ptk, n_seq, tokens_per_seq, psl, pbt,
                                           bt.shape[1], pnb, pwin, _ptr(logits), ws.handle, _stream(stream)))
        return logits

    def step_trace(self, token_ids, batch_index, tokens_per_seq: int, seq_lens, ws: Workspace, stream=None):
        """The step with every stage's result copied out (dsb_decode_step_trace).

        Returns ``(logits, trace)``: ``trace`` maps ``"h_embed"`` and
        ``"x_final"`` to device tensors and ``"layers"`` to one dict per layer
        (``x_attn, qkv, qkv_rope, att_q8, h_attn, x_ffn, gu, act_q8, h_out``);
        q8_0 stages are uint8 ``[n_tok, cols/32*34]``, the others float32."""
        import torch
        n_seq = len(batch_index)
        n_tok = n_seq * tokens_per_seq
        sh = self.shape
        hid, hq, hkv, d, ffn = sh.hidden, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.ffn

        def f32(cols):
            return torch.empty((n_tok, cols), dtype=torch.float32, device="cuda")

        def q8(cols):
            return torch.empty((n_tok, q8_rows_bytes(cols)), dtype=torch.uint8, device="cuda")

        layers = []
        arr = (LayerTraceC * sh.n_layers)()
        for l in range(sh.n_layers):
            t = {"x_attn": q8(hid), "qkv": f32((hq + 2 * hkv) * d), "qkv_rope": f32((hq + 2 * hkv) * d),
                 "att_q8": q8(hq * d), "h_attn": f32(hid), "x_ffn": q8(hid), "gu": f32(2 * ffn), "act_q8": q8(ffn),
                 "h_out": f32(hid)}
            for k, v in t.items():
                setattr(arr[l], k, _ptr(v))
            layers.append(t)
        trace = {"h_embed": f32(hid), "x_final": q8(hid), "layers": layers}
        c = StepTraceC(_ptr(trace["h_embed"]), arr, _ptr(trace["x_final"]))
        logits = torch.empty((n_tok, self.vocab), dtype=torch.float32, device="cuda")
        tk, ptk = _i32(token_ids, n_tok, "token_ids")
        bi, pbi = _i32(batch_index)
        sl, psl = _i32(seq_lens, n_seq, "seq_lens")
        _check(lib().dsb_decode_step_trace(ctypes.byref(self.c), ptk, pbi, n_seq, tokens_per_seq, psl, _ptr(logits),
                                           ws.handle, ctypes.byref(c), _stream(stream)))
        return logits, trace

    def graph(self, n_seq: int, tokens_per_seq: int, logits, ws: Workspace, stream=None) -> "StepGraph":
        return StepGraph(self, n_seq, tokens_per_seq, logits, ws, stream)

    def graph_paged(self, pages, max_blocks: int, n_seq: int, tokens_per_seq: int, logits, ws: Workspace,
                    stream=None) -> "StepGraph":
        """The paged step captured for block tables ``max_blocks`` wide
        (dsb_step_graph_create_paged); replay with ``launch_paged``."""
        return StepGraph(self, n_seq, tokens_per_seq, logits, ws, stream, pages=pages, max_blocks=max_blocks)


class StepGraph:
    """A decode step captured once for a fixed (n_seq, T) and replayed."""

    def __init__(self, model: DecodeModel, n_seq: int, tokens_per_seq: int, logits, ws: Workspace, stream=None,
                 pages=None, max_blocks: int = 0):
        self.model, self.logits, self.ws = model, logits, ws
        self.n_seq, self.T = n_seq, tokens_per_seq
        self.pages, self.max_blocks = pages, max_blocks
        _need(logits, 4 * n_seq * tokens_per_seq * model.vocab, "logits", "f32")
        handle = _P()
        if pages is None:
            _check(lib().dsb_step_graph_create(ctypes.byref(model.c), n_seq, tokens_per_seq, _ptr(logits), ws.handle,
                                               _stream(stream), ctypes.byref(handle)))
        else:
            if len(pages) != model.shape.n_layers:
                raise ValueError(f"pages: one pool per layer ({model.shape.n_layers}), got {len(pages)}")
            arr = (KVPages * len(pages))(*pages)
            _check(lib().dsb_step_graph_create_paged(ctypes.byref(model.c), arr, max_blocks, n_seq, tokens_per_seq,
                                                     _ptr(logits), ws.handle, _stream(stream), ctypes.byref(handle)))
        self.handle = handle

    def launch(self, token_ids, batch_index, seq_lens, stream=None):
        tk, ptk = _i32(token_ids, self.n_seq * self.T, "token_ids")
        bi, pbi = _i32(batch_index, self.n_seq, "batch_index")
        sl, psl = _i32(seq_lens, self.n_seq, "seq_lens")
        _check(lib().dsb_step_graph_launch(self.handle, ptk, pbi, psl, _stream(stream)))
        return self.logits

    def launch_paged(self, token_ids, seq_lens, block_table, n_blocks, window, stream=None):
        """Replay of a graph on page pools with this step's geometry
        (``block_table [n_seq][max_blocks]`` as captured)."""
        bt, pbt, nb, pnb, win, pwin = _geometry(block_table, n_blocks, window)
        if bt.shape != (self.n_seq, self.max_blocks):
            raise ValueError(f"block_table: shape ({self.n_seq}, {self.max_blocks}) expected, got {bt.shape}")
        tk, ptk = _i32(token_ids, self.n_seq * self.T, "token_ids")
        sl, psl = _i32(seq_lens, self.n_seq, "seq_lens")
        _check(lib().dsb_step_graph_launch_paged(self.handle, ptk, psl, pbt, pnb, pwin, _stream(stream)))
        return self.logits

    def close(self):
        if getattr(self, "handle", None):
            lib().dsb_step_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
