"""ctypes binding of libsink_attn.so (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
include/sink_attn.h).  Tensors are torch tensors on a CUDA device; torch only
provides the device memory and the current stream.  Nothing here computes any
part of the attention: if the library is missing the calls raise, there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_LIB = None

OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
                4: "device-side wait timed out", 5: "out of device memory"}
OUT_BF16 = 0
OUT_F32 = 1

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

EXPORTS = {
    "sink_attn_prefill": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _P]),
    "sink_attn_prefill_rope": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _F, _P, _I, _P, _P]),
    "sink_attn_decode": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I, _P, _I, _P,
                              _P, _SZ, _P]),
    "sink_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I, _P, _I, _P,
                                      _P]),
    "sink_attn_decode_rope": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I, _P, _P, _F, _P, _I,
                                   _P, _P, _SZ, _P]),
    "sink_attn_decode_multi": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I, _P, _I,
                                    _P, _P, _SZ, _P]),
    "sink_attn_prefill_paged": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I,
                                     _P, _I, _P, _P, _SZ, _P]),
    "sink_attn_prefill_paged_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "sink_attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "sink_attn_decode_multi_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "sink_attn_decode_max_splits": (_I, [_I, _I, _I, _I, _I]),
    "sink_attn_qkv_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _P, _P, _I, _I, _P]),
    "sink_attn_yarn_inv_freq": (_I, [_I, ctypes.c_double, ctypes.c_double, _I, ctypes.c_double, ctypes.c_double,
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]),
    "sink_attn_status_string": (ctypes.c_char_p, [_I]),
    "sink_attn_get_device_error": (_I, [_P]),
    "sink_attn_version": (_I, []),
}


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, 'unknown status')} (status {status})")


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load the shared library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gqa_attention_head_sink_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == library_path():
        _LIB = lib
    return lib


def _check(status: int, where: str):
    if status != OK:
        raise SinkAttnError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _workspace(n: int, device, stream):
    """A workspace of n bytes from PyTorch's caching allocator, tied to the
    stream the call runs on (None when the call needs none, or when n is the
    size query's error value: the call itself then reports the arguments)."""
    if n == 0 or n == ctypes.c_size_t(-1).value:
        return None
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)
    return ws


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _same_device(ref: torch.Tensor, **tensors):
    for name, t in tensors.items():
        if t is not None and t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, q on {ref.device}: every tensor must be on one device")


def _check_outputs(out, lse, out_shape, lse_shape):
    """out must be bf16/fp32 with out_shape, lse fp32 with lse_shape: a smaller
    buffer would be written past its end on the device."""
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    if tuple(out.shape) != tuple(out_shape):
        raise ValueError(f"out must have shape {tuple(out_shape)}, got {tuple(out.shape)}")
    if lse is not None and tuple(lse.shape) != tuple(lse_shape):
        raise ValueError(f"lse must have shape {tuple(lse_shape)}, got {tuple(lse.shape)}")
    _need(out, "out", out.dtype, len(out_shape))
    if lse is not None:
        _need(lse, "lse", torch.float32, len(lse_shape))


def _check_paged(q, k_pages, v_pages, page_table, seqlens, sinks, batch, hq, d):
    """Shapes the paged calls read through: the pools alike, one page-table row
    and one length per sequence, one sink per query head."""
    if v_pages.shape != k_pages.shape or k_pages.shape[3] != d:
        raise ValueError("k_pages and v_pages must both be [num_pages, Hkv, page_size, D]")
    if page_table.shape[0] != batch or seqlens.shape[0] != batch:
        raise ValueError("page_table and seqlens need one row per sequence")
    if sinks.shape[0] != hq:
        raise ValueError("sinks must have one entry per query head")


def sink_attn_status_string(status: int) -> str:
    return load().sink_attn_status_string(int(status)).decode()


def sink_attn_version() -> int:
    return load().sink_attn_version()


def sink_attn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) a recorded device timeout."""
    return load().sink_attn_get_device_error(_stream_ptr(stream))


def sink_attn_prefill(q, k, v, sinks, cu_seqlens, scale: float, out=None, out_dtype=torch.float32,
                      lse=None, max_seqlen: Optional[int] = None, stream=None):
    """Causal varlen prefill.  q [T,Hq,64], k/v [T,Hkv,64] bf16; sinks [Hq] fp32;
    cu_seqlens [B+1] int32.  Returns out [T,Hq,64] (bf16 or fp32).
    ``max_seqlen`` (host upper bound on the lengths) defaults to T, which
    needs no read of the device, so the call can be captured in a CUDA graph."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(sinks, "sinks", torch.float32, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != (T, hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, D] with the same T and D as q")
    if sinks.shape[0] != hq:
        raise ValueError("sinks must have one entry per query head")
    B = cu_seqlens.shape[0] - 1
    if max_seqlen is None:  # an upper bound known without reading the device (graph-capturable)
        max_seqlen = T
    if out is None:
        out = torch.empty((T, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (T, hq, d), (T, hq))
    _same_device(q, k=k, v=v, sinks=sinks, cu_seqlens=cu_seqlens, out=out, lse=lse)
    st = load().sink_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens), B, T, int(max_seqlen),
                                  hq, hkv, d, float(scale), _ptr(out),
                                  OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse),
                                  _stream_ptr(stream))
    _check(st, "sink_attn_prefill")
    return out


def sink_attn_prefill_rope(q, k, v, sinks, cu_seqlens, scale: float, inv_freq, attn_factor: float = 1.0,
                           q_bias=None, out=None, out_dtype=torch.float32, lse=None,
                           max_seqlen: Optional[int] = None, stream=None):
    """sink_attn_prefill with the query's bias and rotary encoding applied in
    the kernel: q [T,Hq,64] bf16 is the raw projection, token i of a sequence
    at position i; k and v are ready (sink_attn_qkv_rope with q=None).
    inv_freq [32] fp64 (CUDA), q_bias [Hq,64] bf16 or None.  Returns out."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(sinks, "sinks", torch.float32, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(inv_freq, "inv_freq", torch.float64, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != (T, hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, D] with the same T and D as q")
    if sinks.shape[0] != hq or inv_freq.shape[0] != d // 2:
        raise ValueError("sinks [Hq] and inv_freq [D/2]")
    if q_bias is not None:
        _need(q_bias, "q_bias", torch.bfloat16, 2)
        if tuple(q_bias.shape) != (hq, d):
            raise ValueError("q_bias must be [Hq, D]")
    B = cu_seqlens.shape[0] - 1
    if max_seqlen is None:
        max_seqlen = T
    if out is None:
        out = torch.empty((T, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (T, hq, d), (T, hq))
    _same_device(q, k=k, v=v, sinks=sinks, cu_seqlens=cu_seqlens, out=out, lse=lse, inv_freq=inv_freq,
                 q_bias=q_bias)
    st = load().sink_attn_prefill_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens), B, T,
                                       int(max_seqlen), hq, hkv, d, float(scale), _ptr(q_bias), _ptr(inv_freq),
                                       float(attn_factor), _ptr(out),
                                       OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse),
                                       _stream_ptr(stream))
    _check(st, "sink_attn_prefill_rope")
    return out


def sink_attn_decode_workspace_bytes(batch: int, max_seqlen: int, num_q_heads: int, num_kv_heads: int,
                                     head_dim: int = 64, page_size: int = 16, num_splits: int = 0) -> int:
    n = load().sink_attn_decode_workspace_bytes(batch, max_seqlen, num_q_heads, num_kv_heads, head_dim,
                                                page_size, num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise SinkAttnError(1, "sink_attn_decode_workspace_bytes")
    return n


def sink_attn_decode_multi_workspace_bytes(batch: int, q_len: int, max_seqlen: int, num_q_heads: int,
                                           num_kv_heads: int, head_dim: int = 64, page_size: int = 16,
                                           num_splits: int = 0) -> int:
    n = load().sink_attn_decode_multi_workspace_bytes(batch, q_len, max_seqlen, num_q_heads, num_kv_heads,
                                                      head_dim, page_size, num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise SinkAttnError(1, "sink_attn_decode_multi_workspace_bytes")
    return n


def sink_attn_decode_max_splits(batch: int, max_seqlen: int, num_kv_heads: int, page_size: int = 16,
                                num_splits: int = 0) -> int:
    return load().sink_attn_decode_max_splits(batch, max_seqlen, num_kv_heads, page_size, num_splits)


def sink_attn_decode(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float, num_splits: int = 0,
                     out=None, out_dtype=torch.float32, lse=None, max_seqlen: Optional[int] = None,
                     workspace=None, stream=None):
    """Split-KV paged decode.  q [B,Hq,64] bf16; k_pages/v_pages
    [num_pages,Hkv,16,64] bf16; page_table [B,stride] int32; seqlens [B]
    int32; sinks [Hq] fp32.  ``workspace``: optional uint8 CUDA tensor of at
    least sink_attn_decode_workspace_bytes(...) bytes (else one comes from
    PyTorch's caching allocator for this call).  ``max_seqlen`` (host upper bound on the
    lengths, fixes the grid) defaults to stride * page_size, which needs no
    read of the device (graph-capturable); the true maximum sizes the work
    exactly.  Returns out [B,Hq,64]."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    B, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_pages.shape
    _check_paged(q, k_pages, v_pages, page_table, seqlens, sinks, B, hq, d)
    if max_seqlen is None:  # the page-table width bounds every length: no device read
        max_seqlen = page_table.shape[1] * page_size
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (B, hq, d), (B, hq))
    _same_device(q, k_pages=k_pages, v_pages=v_pages, page_table=page_table, seqlens=seqlens, sinks=sinks,
                 out=out, lse=lse, workspace=workspace)
    if workspace is None:
        workspace = _workspace(load().sink_attn_decode_workspace_bytes(B, int(max_seqlen), hq, hkv, d, page_size,
                                                                       int(num_splits)), q.device, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = load().sink_attn_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), page_table.shape[1],
                                 _ptr(seqlens), B, int(max_seqlen), num_pages, _ptr(sinks), hq, hkv, d, page_size,
                                 float(scale), int(num_splits), _ptr(out),
                                 OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse), ws_ptr,
                                 ws_bytes, _stream_ptr(stream))
    _check(st, "sink_attn_decode")
    return out


def sink_attn_decode_rope(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float, inv_freq,
                          attn_factor: float = 1.0, q_bias=None, num_splits: int = 0, out=None,
                          out_dtype=torch.float32, lse=None, max_seqlen: Optional[int] = None, workspace=None,
                          stream=None):
    """sink_attn_decode with the query's bias and rotary encoding applied in the
    kernel: q [B,Hq,64] bf16 is the raw projection; the query of sequence b is
    rotated by position seqlens[b] - 1.  inv_freq [32] fp64 (CUDA), q_bias
    [Hq,64] bf16 or None.  The cache holds rotated keys (sink_attn_qkv_rope
    with q=None).  Returns out [B,Hq,64]."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    _need(inv_freq, "inv_freq", torch.float64, 1)
    B, hq, d = q.shape
    if inv_freq.shape[0] != d // 2:
        raise ValueError("inv_freq must have head_dim / 2 entries")
    if q_bias is not None:
        _need(q_bias, "q_bias", torch.bfloat16, 2)
        if tuple(q_bias.shape) != (hq, d):
            raise ValueError("q_bias must be [Hq, D]")
    num_pages, hkv, page_size, _ = k_pages.shape
    _check_paged(q, k_pages, v_pages, page_table, seqlens, sinks, B, hq, d)
    if max_seqlen is None:  # the page-table width bounds every length: no device read
        max_seqlen = page_table.shape[1] * page_size
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (B, hq, d), (B, hq))
    _same_device(q, k_pages=k_pages, v_pages=v_pages, page_table=page_table, seqlens=seqlens, sinks=sinks,
                 out=out, lse=lse, workspace=workspace, inv_freq=inv_freq, q_bias=q_bias)
    if workspace is None:
        workspace = _workspace(load().sink_attn_decode_workspace_bytes(B, int(max_seqlen), hq, hkv, d, page_size,
                                                                       int(num_splits)), q.device, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = load().sink_attn_decode_rope(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), page_table.shape[1],
                                      _ptr(seqlens), B, int(max_seqlen), num_pages, _ptr(sinks), hq, hkv, d,
                                      page_size, float(scale), int(num_splits), _ptr(q_bias), _ptr(inv_freq),
                                      float(attn_factor), _ptr(out), OUT_F32 if out.dtype == torch.float32 else OUT_BF16,
                                      _ptr(lse), ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(st, "sink_attn_decode_rope")
    return out


def sink_attn_decode_multi(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float, num_splits: int = 0,
                           out=None, out_dtype=torch.float32, lse=None, max_seqlen: Optional[int] = None,
                           workspace=None, stream=None):
    """Multi-token decode.  q [B,n,Hq,64] bf16 holds the last n tokens of each
    sequence's cache (token t at position seqlens[b] - n + t, causal among the
    new tokens); the other arguments are those of sink_attn_decode
    (workspace: sink_attn_decode_multi_workspace_bytes(...)).  Returns out
    [B,n,Hq,64]."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    B, n, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_pages.shape
    _check_paged(q, k_pages, v_pages, page_table, seqlens, sinks, B, hq, d)
    if max_seqlen is None:  # the page-table width bounds every length: no device read
        max_seqlen = page_table.shape[1] * page_size
    if out is None:
        out = torch.empty((B, n, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (B, n, hq, d), (B, n, hq))
    _same_device(q, k_pages=k_pages, v_pages=v_pages, page_table=page_table, seqlens=seqlens, sinks=sinks,
                 out=out, lse=lse, workspace=workspace)
    if workspace is None:
        workspace = _workspace(load().sink_attn_decode_multi_workspace_bytes(B, n, int(max_seqlen), hq, hkv, d,
                                                                             page_size, int(num_splits)),
                               q.device, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = load().sink_attn_decode_multi(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                       page_table.shape[1], _ptr(seqlens), B, n, int(max_seqlen), num_pages,
                                       _ptr(sinks), hq, hkv, d, page_size, float(scale), int(num_splits), _ptr(out),
                                       OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse), ws_ptr,
                                       ws_bytes, _stream_ptr(stream))
    _check(st, "sink_attn_decode_multi")
    return out


def sink_attn_prefill_paged_workspace_bytes(batch: int, total_q: int, max_seqlen_q: int, max_seqlen_k: int,
                                            num_q_heads: int, num_kv_heads: int, head_dim: int = 64,
                                            page_size: int = 16, num_splits: int = 0) -> int:
    n = load().sink_attn_prefill_paged_workspace_bytes(batch, total_q, max_seqlen_q, max_seqlen_k, num_q_heads,
                                                       num_kv_heads, head_dim, page_size, num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise SinkAttnError(1, "sink_attn_prefill_paged_workspace_bytes")
    return n


def sink_attn_prefill_paged(q, k_pages, v_pages, page_table, cu_seqlens_q, seqlens_k, sinks, scale: float,
                            num_splits: int = 0, out=None, out_dtype=torch.float32, lse=None,
                            max_seqlen_q: Optional[int] = None, max_seqlen_k: Optional[int] = None,
                            workspace=None, stream=None):
    """Chunked prefill against the paged cache.  q [total_q,Hq,64] bf16 packed
    by cu_seqlens_q [B+1] int32: the new tokens of sequence b are the last
    n_b of its seqlens_k[b] cached tokens (token t at position L - n_b + t,
    causal).  Other arguments as sink_attn_decode.  Returns out
    [total_q,Hq,64]."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(seqlens_k, "seqlens_k", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    total_q, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_pages.shape
    B = seqlens_k.shape[0]
    _check_paged(q, k_pages, v_pages, page_table, seqlens_k, sinks, B, hq, d)
    if cu_seqlens_q.shape[0] != B + 1:
        raise ValueError("cu_seqlens_q needs one offset per sequence (plus one)")
    # upper bounds known without reading the device (graph-capturable); pass the true
    # maxima to size the work exactly
    if max_seqlen_q is None:
        max_seqlen_q = total_q
    if max_seqlen_k is None:
        max_seqlen_k = page_table.shape[1] * page_size
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (total_q, hq, d), (total_q, hq))
    _same_device(q, k_pages=k_pages, v_pages=v_pages, page_table=page_table, cu_seqlens_q=cu_seqlens_q,
                 seqlens_k=seqlens_k, sinks=sinks, out=out, lse=lse, workspace=workspace)
    if workspace is None:
        workspace = _workspace(load().sink_attn_prefill_paged_workspace_bytes(B, total_q, int(max_seqlen_q),
                                                                              int(max_seqlen_k), hq, hkv, d,
                                                                              page_size, int(num_splits)),
                               q.device, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = load().sink_attn_prefill_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                        page_table.shape[1], _ptr(cu_seqlens_q), _ptr(seqlens_k), B, total_q,
                                        int(max_seqlen_q), int(max_seqlen_k), num_pages, _ptr(sinks), hq, hkv, d,
                                        page_size, float(scale), int(num_splits), _ptr(out),
                                        OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse), ws_ptr,
                                        ws_bytes, _stream_ptr(stream))
    _check(st, "sink_attn_prefill_paged")
    return out


def sink_attn_yarn_inv_freq(head_dim: int = 64, base: float = 10000.0, factor: float = 1.0,
                            original_max_position: int = 4096, beta_fast: float = 32.0, beta_slow: float = 1.0):
    """YaRN rotary frequencies (host computation in the library).  Returns
    (inv_freq as a CPU float64 tensor [head_dim / 2], attn_factor)."""
    if head_dim <= 0 or head_dim % 2:
        raise SinkAttnError(1, "sink_attn_yarn_inv_freq")
    buf = (ctypes.c_double * (head_dim // 2))()
    af = ctypes.c_float()
    st = load().sink_attn_yarn_inv_freq(head_dim, float(base), float(factor), int(original_max_position),
                                        float(beta_fast), float(beta_slow), buf, ctypes.byref(af))
    _check(st, "sink_attn_yarn_inv_freq")
    return torch.tensor(list(buf), dtype=torch.float64), float(af.value)


def sink_attn_qkv_rope(q, k, v, positions, inv_freq, attn_factor: float = 1.0, q_bias=None, k_bias=None,
                       v_bias=None, slot_mapping=None, k_pages=None, v_pages=None, stream=None):
    """In place: q <- rot(q + q_bias), k <- rot(k + k_bias), v <- v + v_bias,
    rotation by positions[t] * inv_freq (half-split planes) times attn_factor.
    q [T,Hq,64] (or None: left to sink_attn_prefill_rope / sink_attn_decode_rope),
    k/v [T,Hkv,64] bf16; biases [H,64] bf16 or None; positions [T]
    int32; inv_freq [32] fp64 (CUDA).  With slot_mapping [T] int32 the new k/v
    are also written to k_pages/v_pages [num_pages,Hkv,16,64] at those slots."""
    if q is not None:
        _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(positions, "positions", torch.int32, 1)
    _need(inv_freq, "inv_freq", torch.float64, 1)
    for name, b in (("q_bias", q_bias), ("k_bias", k_bias), ("v_bias", v_bias)):
        if b is not None:
            _need(b, name, torch.bfloat16, 2)
    T, hkv, d = k.shape
    hq = q.shape[1] if q is not None else (q_bias.shape[0] if q_bias is not None else hkv)
    if (q is not None and (q.shape[0] != T or q.shape[2] != d)) or k.shape != v.shape or positions.shape[0] != T \
            or inv_freq.shape[0] != d // 2:
        raise ValueError("q [T,Hq,D], k and v [T,Hkv,D], positions [T], inv_freq [D/2]")
    # the kernel reads a bias row per head and writes cache slots per kv head: smaller buffers
    # would be read or written past their ends on the device
    for name, b, h in (("q_bias", q_bias, hq), ("k_bias", k_bias, hkv), ("v_bias", v_bias, hkv)):
        if b is not None and tuple(b.shape) != (h, d):
            raise ValueError(f"{name} must be [{h}, {d}], got {tuple(b.shape)}")
    _same_device(k, q=q, v=v, positions=positions, inv_freq=inv_freq, q_bias=q_bias, k_bias=k_bias, v_bias=v_bias,
                 slot_mapping=slot_mapping, k_pages=k_pages, v_pages=v_pages)
    num_pages, page_size = 0, 16
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int32, 1)
        _need(k_pages, "k_pages", torch.bfloat16, 4)
        _need(v_pages, "v_pages", torch.bfloat16, 4)
        num_pages, page_size = k_pages.shape[0], k_pages.shape[2]
        if slot_mapping.shape[0] != T:
            raise ValueError("slot_mapping needs one slot per token")
        if v_pages.shape != k_pages.shape or k_pages.shape[1] != hkv or k_pages.shape[3] != d:
            raise ValueError("k_pages and v_pages must both be [num_pages, Hkv, page_size, D] with the Hkv and D of k")
    st = load().sink_attn_qkv_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(q_bias), _ptr(k_bias), _ptr(v_bias),
                                   _ptr(positions), _ptr(inv_freq), float(attn_factor), T, hq, hkv, d,
                                   _ptr(slot_mapping), _ptr(k_pages), _ptr(v_pages), num_pages, page_size,
                                   _stream_ptr(stream))
    _check(st, "sink_attn_qkv_rope")
    return q, k, v


NOALLOC_SCRATCH_BYTES = 16 << 20


def sink_attn_decode_noalloc(q, k_pages, v_pages, page_table, seqlens, sinks, scale: float, num_splits: int = 0,
                             out=None, out_dtype=torch.float32, lse=None, max_seqlen: Optional[int] = None,
                             stream=None):
    """sink_attn_decode without a workspace, for callers that cannot allocate
    device memory at decode time: the partial states use the library's own
    16 MiB scratch array.  Pass ``out`` (and ``lse``) preallocated to keep the
    call itself free of allocations.  Concurrent calls on different streams
    race on that array."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    B, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_pages.shape
    _check_paged(q, k_pages, v_pages, page_table, seqlens, sinks, B, hq, d)
    if max_seqlen is None:  # the page-table width bounds every length: no device read
        max_seqlen = page_table.shape[1] * page_size
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=q.device)
    _check_outputs(out, lse, (B, hq, d), (B, hq))
    _same_device(q, k_pages=k_pages, v_pages=v_pages, page_table=page_table, seqlens=seqlens, sinks=sinks,
                 out=out, lse=lse)
    st = load().sink_attn_decode_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                         page_table.shape[1], _ptr(seqlens), B, int(max_seqlen), num_pages,
                                         _ptr(sinks), hq, hkv, d, page_size, float(scale), int(num_splits), _ptr(out),
                                         OUT_F32 if out.dtype == torch.float32 else OUT_BF16, _ptr(lse),
                                         _stream_ptr(stream))
    _check(st, "sink_attn_decode_noalloc")
    return out
