"""ctypes binding of the C ABI declared in ``include/attn.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libattn_gb300.so``. The library is loaded on first use; if it is
missing, the call raises -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_FILE = os.path.join(_HERE, "libattn_gb300.so")

ATTN_BF16, ATTN_FP16, ATTN_FP32 = 0, 1, 2
PATH_AUTO, PATH_SIMT, PATH_PREFILL, PATH_DECODE, PATH_PREFILL_PAIR = 0, 1, 2, 3, 4
ATTN_OK = 0

_DTYPES = {torch.bfloat16: ATTN_BF16, torch.float16: ATTN_FP16, torch.float32: ATTN_FP32}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({strerror(status)})")


def library_path() -> str:
    return _LIB_FILE


def lib() -> ctypes.CDLL:
    """Load the shared library (raises FileNotFoundError if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_FILE):
                raise FileNotFoundError(
                    f"{_LIB_FILE} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_LIB_FILE)
            vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [vp, vp, vp, vp] + [ci] * 8 + [cf, ci, vp]
            L.attn_fwd.restype = ci
            L.attn_fwd_ex.argtypes = [vp, vp, vp, vp] + [ci] * 8 + [cf, ci, ci, vp, sz, vp]
            L.attn_fwd_ex.restype = ci
            L.attn_workspace_bytes.argtypes = [ci] * 7
            L.attn_workspace_bytes.restype = sz
            L.attn_workspace_bytes_ex.argtypes = [ci] * 9
            L.attn_workspace_bytes_ex.restype = sz
            L.attn_fwd_ws.argtypes = [vp, vp, vp, vp] + [ci] * 8 + [cf, ci, vp, sz, vp]
            L.attn_fwd_ws.restype = ci
            L.attn_merge.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, vp]
            L.attn_merge.restype = ci
            L.attn_fwd_host.argtypes = [vp] * 8 + [ci] * 8 + [cf, ci, vp, sz, vp]
            L.attn_fwd_host.restype = ci
            L.attn_strerror.argtypes = [ci]
            L.attn_strerror.restype = ctypes.c_char_p
            L.attn_last_device_status.argtypes = [vp]
            L.attn_last_device_status.restype = ci
            L.attn_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp] + [ci] * 8 + [cf, ci, vp]
            L.attn_fwd_decode_noalloc.restype = ci
            L.attn_decode_paged_workspace_bytes.argtypes = [ci] * 10
            L.attn_decode_paged_workspace_bytes.restype = sz
            L.attn_decode_paged.argtypes = [vp] * 6 + [ci] * 11 + [cf, ci, vp, sz, vp]
            L.attn_decode_paged.restype = ci
            L.attn_decode_paged_fp8.argtypes = [vp] * 6 + [ci] * 11 + [cf] * 4 + [ci, vp, sz, vp]
            L.attn_decode_paged_fp8.restype = ci
            L.attn_fwd_lse.argtypes = [vp] * 5 + [ci] * 8 + [cf, ci, ci, vp, sz, vp]
            L.attn_fwd_lse.restype = ci
            L.attn_fwd_fp8.argtypes = [vp] * 5 + [ci] * 8 + [cf, cf, cf, cf, ci, ci, vp, sz, vp]
            L.attn_fwd_fp8.restype = ci
            L.attn_fwd_fp8_workspace_bytes.argtypes = [ci] * 9
            L.attn_fwd_fp8_workspace_bytes.restype = sz
            L.attn_decode_paged_fp8_workspace_bytes.argtypes = [ci] * 10
            L.attn_decode_paged_fp8_workspace_bytes.restype = sz
            L.attn_bwd_workspace_bytes.argtypes = [ci, ci, ci]
            L.attn_bwd_workspace_bytes.restype = sz
            L.attn_bwd.argtypes = [vp] * 9 + [ci] * 8 + [cf, ci, vp, sz, vp]
            L.attn_bwd.restype = ci
            L.attn_split_softmax_workspace_bytes.argtypes = [ci, ci, ci]
            L.attn_split_softmax_workspace_bytes.restype = sz
            L.attn_split_softmax.argtypes = [vp, vp, ci, ci, ci, ci, vp, sz, vp]
            L.attn_split_softmax.restype = ci
            L.attn_selftest_bounded_wait.argtypes = [ctypes.c_uint, vp]
            L.attn_selftest_bounded_wait.restype = ci
            L.attn_selftest_prefill_abort.argtypes = [vp] * 4 + [ci] * 7 + [ctypes.c_longlong, vp]
            L.attn_selftest_prefill_abort.restype = ci
            L.attn_version.argtypes = []
            L.attn_version.restype = ci
            _lib = L
        return _lib


def strerror(status: int) -> str:
    try:
        return lib().attn_strerror(int(status)).decode()
    except FileNotFoundError:
        return "library not loaded"


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)


def _dims(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: Optional[torch.Tensor]):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D: [B, Hq, M, D] and [B, Hkv, N, D]")
    B, Hq, M, D = q.shape
    Bk, Hkv, N, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if o is not None and tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have the shape of q")
    for t in (q, k, v) + ((o,) if o is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.dtype != q.dtype:
            raise ValueError("q, k, v, o must share one dtype")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("dtype must be bfloat16 or float16")
    return B, Hq, Hkv, M, N, D


def attn_workspace_bytes(B, Hq, Hkv, M, N, D, window=0) -> int:
    """C-ABI ``attn_workspace_bytes``: workspace bytes ``attn_fwd_ws`` needs (either causal value)."""
    return int(lib().attn_workspace_bytes(B, Hq, Hkv, M, N, D, int(window)))


def attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, causal=False, window=0, path=PATH_AUTO) -> int:
    """C-ABI ``attn_workspace_bytes_ex``: workspace bytes ``attn_fwd_ex`` needs on ``path``."""
    return int(lib().attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, int(bool(causal)), int(window), int(path)))


def attn_fwd(q, k, v, o, causal=False, window=0, scale=0.0, stream=None) -> None:
    """C-ABI ``attn_fwd`` on device tensors; writes ``o`` in place."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D, int(bool(causal)), int(window),
                        float(scale or 0.0), _DTYPES[q.dtype], _stream(stream))
    _check(st, "attn_fwd")


def attn_fwd_ws(q, k, v, o, causal=False, window=0, scale=0.0, workspace=None, stream=None) -> None:
    """C-ABI ``attn_fwd_ws``: the path ``attn_fwd`` takes, with caller workspace (a uint8 device tensor)."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D, int(bool(causal)),
                           int(window), float(scale or 0.0), _DTYPES[q.dtype], _ptr(workspace), ws_bytes,
                           _stream(stream))
    _check(st, "attn_fwd_ws")


def attn_fwd_ex(q, k, v, o, causal=False, window=0, scale=0.0, path=PATH_AUTO, workspace=None,
                stream=None) -> None:
    """C-ABI ``attn_fwd_ex``: explicit path, caller workspace (a uint8 device tensor)."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D, int(bool(causal)),
                           int(window), float(scale or 0.0), _DTYPES[q.dtype], int(path), _ptr(workspace),
                           ws_bytes, _stream(stream))
    _check(st, "attn_fwd_ex")


def attn_fwd_lse(q, k, v, o, lse, causal=False, window=0, scale=0.0, path=PATH_AUTO, workspace=None,
                 stream=None) -> None:
    """C-ABI ``attn_fwd_lse``: writes ``o`` and the per-row log-sum-exp ``lse``
    (float32 [B, Hq, M]); ``workspace`` None lets the library allocate it."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    if lse.shape != (B, Hq, M) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, M] tensor")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, M, N, D,
                            int(bool(causal)), int(window), float(scale or 0.0), _DTYPES[q.dtype], int(path),
                            _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "attn_fwd_lse")


def attention_lse(q, k, v, causal=False, window=0, scale=0.0, path=PATH_AUTO, stream=None):
    """New output and log-sum-exp tensors, then the forward into them: (o, lse)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    attn_fwd_lse(q, k, v, o, lse, causal, window, scale, path, None, stream)
    return o, lse


def attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, M, N, D, causal=False, window=0, path=PATH_AUTO) -> int:
    return int(lib().attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, M, N, D, int(bool(causal)), int(window), int(path)))


def attn_decode_paged_fp8_workspace_bytes(B, Hq, Hkv, M, D, page_size, max_pages, max_seq_len, causal=True,
                                          window=0) -> int:
    return int(lib().attn_decode_paged_fp8_workspace_bytes(B, Hq, Hkv, M, D, page_size, max_pages, max_seq_len,
                                                           int(bool(causal)), int(window)))


def attn_fwd_fp8(q, k, v, o, lse=None, causal=False, window=0, scale=0.0, q_descale=1.0, k_descale=1.0,
                 v_descale=1.0, path=PATH_AUTO, workspace=None, stream=None) -> None:
    """C-ABI ``attn_fwd_fp8``: q, k, v are E4M3 (``torch.float8_e4m3fn``) device
    tensors, ``o`` BF16 or FP16 of q's shape, ``lse`` an optional float32
    [B, Hq, M] tensor; ``workspace`` None lets the library allocate the decode
    path's workspace."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D: [B, Hq, M, D] and [B, Hkv, N, D]")
    B, Hq, M, D = q.shape
    Bk, Hkv, N, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or tuple(o.shape) != tuple(q.shape):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)} o{tuple(o.shape)}")
    for t in (q, k, v):
        if t.dtype != torch.float8_e4m3fn or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous float8_e4m3fn tensors")
    if o.dtype not in (torch.bfloat16, torch.float16) or not o.is_contiguous():
        raise ValueError("o must be a contiguous bfloat16 or float16 tensor")
    if lse is not None and (lse.shape != (B, Hq, M) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [B, Hq, M] tensor")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, M, N, D,
                            int(bool(causal)), int(window), float(scale or 0.0), float(q_descale),
                            float(k_descale), float(v_descale), _DTYPES[o.dtype], int(path), _ptr(workspace),
                            ws_bytes, _stream(stream))
    _check(st, "attn_fwd_fp8")


def attention_fp8(q, k, v, causal=False, window=0, scale=0.0, q_descale=1.0, k_descale=1.0, v_descale=1.0,
                  out_dtype=torch.bfloat16, with_lse=False, path=PATH_AUTO, stream=None):
    """New output tensor (and log-sum-exp when ``with_lse``), then ``attn_fwd_fp8`` into it."""
    o = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if with_lse else None
    attn_fwd_fp8(q, k, v, o, lse, causal, window, scale, q_descale, k_descale, v_descale, path, None, stream)
    return (o, lse) if with_lse else o


def attn_bwd_workspace_bytes(B, Hq, M) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, Hq, M))


def attn_bwd(q, k, v, o, d_o, lse, dq, dk, dv, causal=False, window=0, scale=0.0, workspace=None,
             stream=None) -> None:
    """C-ABI ``attn_bwd``: writes dq, dk, dv (shapes and dtype of q, k, v)."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    for t, ref in ((d_o, q), (dq, q), (dk, k), (dv, k)):
        if tuple(t.shape) != tuple(ref.shape) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("d_o/dq must match q and dk/dv must match k (shape, dtype, contiguous)")
    if lse.shape != (B, Hq, M) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, M] tensor")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, Hq, Hkv, M, N, D, int(bool(causal)), int(window), float(scale or 0.0), _DTYPES[q.dtype],
                        _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "attn_bwd")


def attention(q, k, v, causal=False, window=0, scale=0.0, path=PATH_AUTO, stream=None) -> torch.Tensor:
    """Makes a new contiguous output tensor on q's device, then runs the forward into it."""
    o = torch.empty_like(q)
    if path == PATH_AUTO:
        attn_fwd(q, k, v, o, causal, window, scale, stream)
    else:
        B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
        nbytes = attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, causal, window, path)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
        attn_fwd_ex(q, k, v, o, causal, window, scale, path, ws, stream)
    return o


def attn_merge(m, l, acc, out_dtype=torch.float32, with_stats=False, stream=None):
    """C-ABI ``attn_merge``: m, l [rows, S] and acc [rows, S, D] float32 device tensors."""
    rows, S = m.shape
    D = acc.shape[-1]
    o = torch.empty((rows, D), dtype=out_dtype, device=m.device)
    mo = torch.empty(rows, dtype=torch.float32, device=m.device) if with_stats else None
    lo = torch.empty(rows, dtype=torch.float32, device=m.device) if with_stats else None
    st = lib().attn_merge(_ptr(m), _ptr(l), _ptr(acc), _ptr(o), _ptr(mo), _ptr(lo), rows, S, D,
                          _DTYPES[out_dtype], _stream(stream))
    _check(st, "attn_merge")
    return (o, mo, lo) if with_stats else o


def attn_fwd_host(q_h, k_h, v_h, o_h, q_d, k_d, v_d, o_d, causal=False, window=0, scale=0.0, workspace=None,
                  stream=None) -> None:
    """C-ABI ``attn_fwd_host``: host (pinned) tensors in and out, device staging buffers."""
    B, Hq, Hkv, M, N, D = _dims(q_d, k_d, v_d, o_d)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(q_d), _ptr(k_d), _ptr(v_d),
                             _ptr(o_d), B, Hq, Hkv, M, N, D, int(bool(causal)), int(window), float(scale or 0.0),
                             _DTYPES[q_d.dtype], _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "attn_fwd_host")


def attn_fwd_decode_noalloc(q, k, v, o, causal=False, window=0, scale=0.0, stream=None) -> None:
    """C-ABI ``attn_fwd_decode_noalloc``: the split-KV decode path using the
    library's fixed scratch array, for callers that cannot allocate."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    st = lib().attn_fwd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D, int(bool(causal)),
                                       int(window), float(scale or 0.0), _DTYPES[q.dtype], _stream(stream))
    _check(st, "attn_fwd_decode_noalloc")


def _paged_dims(q, k_pages, v_pages, block_table, seq_lens, o, e4m3=False):
    if q.dim() != 4 or k_pages.dim() != 4 or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("q is [B, Hq, M, D]; k_pages and v_pages are [num_pages, Hkv, page_size, D]")
    B, Hq, M, D = q.shape
    num_pages, Hkv, page_size, Dk = k_pages.shape
    if Dk != D or (o is not None and tuple(o.shape) != tuple(q.shape)):
        raise ValueError("head dimensions or output shape do not match")
    if block_table.dim() != 2 or block_table.shape[0] != B or block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seq_lens.shape != (B,) or seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32 [B]")
    for t in (q, k_pages, v_pages, block_table, seq_lens) + ((o,) if o is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if e4m3:
        if any(t.dtype != torch.float8_e4m3fn for t in (q, k_pages, v_pages)):
            raise ValueError("q, k_pages, v_pages must be float8_e4m3fn")
        if o.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("o must be bfloat16 or float16")
    else:
        if k_pages.dtype != q.dtype or v_pages.dtype != q.dtype or (o is not None and o.dtype != q.dtype):
            raise ValueError("q, k_pages, v_pages, o must share one dtype")
        if q.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("dtype must be bfloat16 or float16")
    return B, Hq, Hkv, M, D, num_pages, page_size, block_table.shape[1]


def attn_decode_paged_workspace_bytes(B, Hq, Hkv, M, D, page_size, max_pages, max_seq_len, causal=True,
                                      window=0) -> int:
    return int(lib().attn_decode_paged_workspace_bytes(B, Hq, Hkv, M, D, page_size, max_pages, max_seq_len,
                                                       int(bool(causal)), int(window)))


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, max_seq_len, causal=True, window=0,
                      scale=0.0, workspace=None, stream=None) -> None:
    """C-ABI ``attn_decode_paged``: decode over a paged KV cache; writes ``o`` in place.
    ``workspace`` None lets the library allocate it stream-ordered."""
    B, Hq, Hkv, M, D, num_pages, page_size, max_pages = _paged_dims(q, k_pages, v_pages, block_table, seq_lens, o)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                 _ptr(o), B, Hq, Hkv, M, D, num_pages, page_size, max_pages, int(max_seq_len),
                                 int(bool(causal)), int(window), float(scale or 0.0), _DTYPES[q.dtype],
                                 _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "attn_decode_paged")


def attn_decode_paged_fp8(q, k_pages, v_pages, block_table, seq_lens, o, max_seq_len, causal=True, window=0,
                          scale=0.0, q_descale=1.0, k_descale=1.0, v_descale=1.0, workspace=None,
                          stream=None) -> None:
    """C-ABI ``attn_decode_paged_fp8``: q and the pools are float8_e4m3fn, ``o``
    BF16 or FP16; writes ``o`` in place."""
    B, Hq, Hkv, M, D, num_pages, page_size, max_pages = _paged_dims(q, k_pages, v_pages, block_table, seq_lens, o,
                                                                     e4m3=True)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_decode_paged_fp8(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                     _ptr(o), B, Hq, Hkv, M, D, num_pages, page_size, max_pages, int(max_seq_len),
                                     int(bool(causal)), int(window), float(scale or 0.0), float(q_descale),
                                     float(k_descale), float(v_descale), _DTYPES[o.dtype], _ptr(workspace),
                                     ws_bytes, _stream(stream))
    _check(st, "attn_decode_paged_fp8")


def attn_split_softmax_workspace_bytes(M, N, chunk=1024) -> int:
    return int(lib().attn_split_softmax_workspace_bytes(M, N, chunk))


def split_softmax(x, chunk=1024, y=None, workspace=None, stream=None) -> torch.Tensor:
    """C-ABI ``attn_split_softmax``: row softmax of a contiguous 2-D tensor; returns y."""
    if x.dim() != 2 or not x.is_contiguous() or x.dtype not in _DTYPES:
        raise ValueError("x must be a contiguous 2-D float32/float16/bfloat16 tensor")
    M, N = x.shape
    if y is None:
        y = torch.empty_like(x)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_split_softmax(_ptr(x), _ptr(y), M, N, int(chunk), _DTYPES[x.dtype], _ptr(workspace), ws_bytes,
                                  _stream(stream))
    _check(st, "attn_split_softmax")
    return y


def selftest_bounded_wait(timeout_us=20000, stream=None) -> None:
    """C-ABI ``attn_selftest_bounded_wait``: a wait that runs out on purpose (no fault)."""
    _check(lib().attn_selftest_bounded_wait(int(timeout_us), _stream(stream)), "attn_selftest_bounded_wait")


def selftest_prefill_abort(q, k, v, o, withhold_at=2, stream=None) -> None:
    """C-ABI ``attn_selftest_prefill_abort``: the prefill kernel with one P-ready
    arrival withheld, so every CTA takes its abort path (no fault)."""
    B, Hq, Hkv, M, N, D = _dims(q, k, v, o)
    _check(lib().attn_selftest_prefill_abort(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D,
                                             _DTYPES[q.dtype], int(withhold_at), _stream(stream)),
           "attn_selftest_prefill_abort")


def last_device_status(stream=None) -> int:
    return int(lib().attn_last_device_status(_stream(stream)))
