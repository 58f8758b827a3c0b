"""Python binding of libsp_attn (ctypes).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels, and the schedules are built by its C++ host code.
PyTorch supplies device buffers and streams. If the library cannot be built
or loaded, every call raises; there is no fallback.

Names match the C-ABI declared in include/sp_attn.h.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np

from . import _build

SP_OK = 0
SP_SCHED_RING, SP_SCHED_ZIGZAG, SP_SCHED_TASP = 0, 1, 2
SP_DTYPE_BF16, SP_DTYPE_FP32 = 0, 1

_STATUS = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_UNSUPPORTED", 3: "SP_ERR_BUFFER_TOO_SMALL",
           4: "SP_ERR_CUDA", 5: "SP_ERR_TIMEOUT", 6: "SP_ERR_INTERNAL"}

EXPORTED = ["sp_schedule_build", "sp_schedule_build_chunked", "sp_schedule_build_hier", "sp_chunk_bounds",
            "sp_schedule_link_bytes_hier", "sp_schedule_split_documents",
            "sp_tasp_cycles", "sp_packed_attention_ex", "sp_schedule_link_bytes", "sp_partial_attn", "sp_lse_merge",
            "sp_packed_attention_workspace_size", "sp_packed_attention",
            "sp_packed_attention_static_ws", "sp_packed_attention_backward_workspace_size",
            "sp_packed_attention_backward", "sp_check_device_status",
            "sp_selftest_bounded_wait", "sp_status_string"]


class SpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_STATUS.get(code, code)}")


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Builds (if stale) and loads libsp_attn.so; returns the ctypes handle."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        f32 = ctypes.c_float
        lib.sp_schedule_build.restype = ctypes.c_int
        lib.sp_schedule_build.argtypes = [ctypes.c_int, i32, i32, vp, i32, i32, u64, vp,
                                          ctypes.POINTER(i64)]
        lib.sp_schedule_build_chunked.restype = ctypes.c_int
        lib.sp_schedule_build_chunked.argtypes = [ctypes.c_int, i32, i32, vp, i32, i32, u64, vp, vp,
                                                  ctypes.POINTER(ctypes.c_int64)]
        lib.sp_schedule_link_bytes_hier.restype = ctypes.c_int
        lib.sp_schedule_link_bytes_hier.argtypes = [ctypes.c_int, i32, i32, i32, vp, i32, i32, u64, i32, i32,
                                                    i32, i32, i32, vp, vp]
        lib.sp_schedule_build_hier.restype = ctypes.c_int
        lib.sp_schedule_build_hier.argtypes = [ctypes.c_int, i32, i32, i32, vp, i32, i32, u64, i32, vp, vp,
                                               vp, ctypes.POINTER(ctypes.c_int64)]
        lib.sp_schedule_split_documents.restype = ctypes.c_int
        lib.sp_schedule_split_documents.argtypes = [vp, vp, i64, vp, i32, i32, vp, vp, ctypes.POINTER(i64)]
        lib.sp_packed_attention_ex.restype = ctypes.c_int
        lib.sp_packed_attention_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                               vp, i32, i32, f32, vp, vp, i64, vp, ctypes.c_size_t, vp]
        lib.sp_chunk_bounds.restype = ctypes.c_int
        lib.sp_chunk_bounds.argtypes = [i32, i32, i32, vp, i32, i32, vp]
        lib.sp_tasp_cycles.restype = ctypes.c_int
        lib.sp_tasp_cycles.argtypes = [i32, u64, vp]
        lib.sp_schedule_link_bytes.restype = ctypes.c_int
        lib.sp_schedule_link_bytes.argtypes = [ctypes.c_int, i32, i32, vp, i32, i32, u64, i64, i32, vp]
        lib.sp_partial_attn.restype = ctypes.c_int
        lib.sp_partial_attn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                        i32, i32, i32, i32, vp, i32, i32, f32, vp]
        lib.sp_lse_merge.restype = ctypes.c_int
        lib.sp_lse_merge.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        lib.sp_packed_attention_workspace_size.restype = ctypes.c_size_t
        lib.sp_packed_attention_workspace_size.argtypes = [i64]
        lib.sp_packed_attention.restype = ctypes.c_int
        lib.sp_packed_attention.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                            vp, i32, i32, f32, vp, i64, vp, ctypes.c_size_t, vp]
        lib.sp_packed_attention_static_ws.restype = ctypes.c_int
        lib.sp_packed_attention_static_ws.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                      ctypes.c_int, vp, i32, i32, f32, vp, i64, vp]
        lib.sp_packed_attention_backward_workspace_size.restype = ctypes.c_size_t
        lib.sp_packed_attention_backward_workspace_size.argtypes = [i64, i32, i32]
        lib.sp_packed_attention_backward.restype = ctypes.c_int
        lib.sp_packed_attention_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                     i32, ctypes.c_int, vp, i32, i32, f32, vp, i64,
                                                     vp, ctypes.c_size_t, vp]
        lib.sp_check_device_status.restype = ctypes.c_int
        lib.sp_check_device_status.argtypes = [vp]
        lib.sp_selftest_bounded_wait.restype = ctypes.c_int
        lib.sp_selftest_bounded_wait.argtypes = [u64, vp]
        lib.sp_status_string.restype = ctypes.c_char_p
        lib.sp_status_string.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _check(code: int, where: str):
    if code != SP_OK:
        raise SpError(code, where)


def sp_status_string(code: int) -> str:
    return load().sp_status_string(int(code)).decode()


# ----------------------------------------------------------------- host calls

def sp_schedule_build(kind: int, P: int, total_tokens: int, cu_seqlens, causal: bool,
                      seed: int = 0, bounds=None) -> np.ndarray:
    """Items [n, 8] int32: rank, step, cycle, q_begin, q_end, kv_begin, kv_end, flags.
    bounds: chunk boundaries [P+1] for RING / TASP (sp_chunk_bounds); None = equal chunks."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    nd = len(cu) - 1
    bd = None if bounds is None else np.ascontiguousarray(np.asarray(bounds, dtype=np.int32))
    bp = None if bd is None else bd.ctypes.data
    if bd is not None:
        _need(bd.shape == (P + 1,), "bounds must hold P + 1 values")
    n = ctypes.c_int64(0)
    _check(lib.sp_schedule_build_chunked(kind, P, total_tokens, cu.ctypes.data, nd, int(causal), seed,
                                         bp, None, ctypes.byref(n)), "sp_schedule_build")
    out = np.zeros((max(n.value, 1), 8), dtype=np.int32)
    cap = ctypes.c_int64(n.value)
    _check(lib.sp_schedule_build_chunked(kind, P, total_tokens, cu.ctypes.data, nd, int(causal), seed,
                                         bp, out.ctypes.data, ctypes.byref(cap)), "sp_schedule_build")
    return out[:cap.value]


def sp_schedule_build_hier(inter_kind: int, R: int, U: int, total_tokens: int, cu_seqlens, causal: bool,
                           Hq: int, seed: int = 0, bounds=None):
    """Two-level schedule on R x U virtual ranks: (items [n, 8], heads [n, 2])."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    nd = len(cu) - 1
    bd = None if bounds is None else np.ascontiguousarray(np.asarray(bounds, dtype=np.int32))
    bp = None if bd is None else bd.ctypes.data
    n = ctypes.c_int64(0)
    _check(lib.sp_schedule_build_hier(inter_kind, R, U, total_tokens, cu.ctypes.data, nd, int(causal), seed,
                                      Hq, bp, None, None, ctypes.byref(n)), "sp_schedule_build_hier")
    items = np.zeros((max(n.value, 1), 8), dtype=np.int32)
    heads = np.zeros((max(n.value, 1), 2), dtype=np.int32)
    cap = ctypes.c_int64(n.value)
    _check(lib.sp_schedule_build_hier(inter_kind, R, U, total_tokens, cu.ctypes.data, nd, int(causal), seed,
                                      Hq, bp, items.ctypes.data, heads.ctypes.data, ctypes.byref(cap)),
           "sp_schedule_build_hier")
    return items[:cap.value], heads[:cap.value]


def sp_schedule_split_documents(items, cu_seqlens, causal: bool, heads=None):
    """Every item cut at the document boundaries (one document's pairs per item).
    Returns items [m, 8], or (items, heads [m, 2]) when head ranges are given."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    it = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 8))
    hd = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32).reshape(-1, 2))
    if hd is not None:
        _need(len(hd) == len(it), "heads must hold one range per item")
    if hd is not None and len(hd) == 0:
        hd = np.zeros((1, 2), dtype=np.int32)  # never read with no items; marks "heads given"
    ip = it.ctypes.data if len(it) else None
    hp = None if hd is None else hd.ctypes.data
    n = ctypes.c_int64(0)
    _check(lib.sp_schedule_split_documents(ip, hp, len(it), cu.ctypes.data, len(cu) - 1, int(causal), None,
                                           None, ctypes.byref(n)), "sp_schedule_split_documents")
    out = np.zeros((max(n.value, 1), 8), dtype=np.int32)
    out_h = np.zeros((max(n.value, 1), 2), dtype=np.int32)
    cap = ctypes.c_int64(n.value)
    _check(lib.sp_schedule_split_documents(ip, hp, len(it), cu.ctypes.data, len(cu) - 1, int(causal),
                                           out.ctypes.data, out_h.ctypes.data if hd is not None else None,
                                           ctypes.byref(cap)), "sp_schedule_split_documents")
    if hd is None:
        return out[:cap.value]
    return out[:cap.value], out_h[:cap.value]


def sp_schedule_link_bytes_hier(inter_kind: int, R: int, U: int, total_tokens: int, cu_seqlens, causal: bool,
                                Hq: int, Hkv: int, d: int, elem_bytes: int = 2, seed: int = 0,
                                needed_only: bool = False):
    """Two-level communication model: (intra [P, P], inter [R-1, P, P]) bytes per directed link."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    P = R * U
    intra = np.zeros((P, P), dtype=np.int64)
    inter = np.zeros((max(R - 1, 0), P, P), dtype=np.int64)
    _check(lib.sp_schedule_link_bytes_hier(inter_kind, R, U, total_tokens, cu.ctypes.data, len(cu) - 1,
                                           int(causal), seed, Hq, Hkv, d, elem_bytes, int(needed_only),
                                           intra.ctypes.data, inter.ctypes.data if inter.size else None),
           "sp_schedule_link_bytes_hier")
    return intra, inter


SP_CHUNK_EQUAL, SP_CHUNK_BALANCED, SP_CHUNK_BALANCED_DOC = 0, 1, 2
SP_MAX_GROUPS = 8192  # include/sp_attn.h: groups sp_packed_attention takes


def n_groups(items, heads=None) -> int:
    """Groups of an item list as sp_packed_attention forms them: maximal runs
    of consecutive items sharing rank, Q range and (if given) head range."""
    it = np.asarray(items).reshape(-1, 8)
    if len(it) == 0:
        return 0
    key = it[:, [0, 3, 4]]
    if heads is not None:
        key = np.concatenate([key, np.asarray(heads).reshape(-1, 2)], axis=1)
    return int(1 + np.count_nonzero((key[1:] != key[:-1]).any(axis=1)))


def sp_chunk_bounds(mode: int, P: int, total_tokens: int, cu_seqlens, causal: bool) -> np.ndarray:
    """Chunk boundaries [P+1] of a chunking policy (SP_CHUNK_*)."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    out = np.zeros(P + 1, dtype=np.int32)
    _check(lib.sp_chunk_bounds(int(mode), int(P), int(total_tokens), cu.ctypes.data, len(cu) - 1,
                               int(causal), out.ctypes.data), "sp_chunk_bounds")
    return out


def sp_tasp_cycles(P: int, seed: int = 0) -> np.ndarray:
    lib = load()
    out = np.zeros((max(P - 1, 0), P), dtype=np.int32)
    _check(lib.sp_tasp_cycles(P, seed, out.ctypes.data if out.size else None), "sp_tasp_cycles")
    return out


def sp_schedule_link_bytes(kind: int, P: int, total_tokens: int, cu_seqlens, causal: bool,
                           seed: int = 0, bytes_per_token: int = 1,
                           needed_only: bool = False) -> np.ndarray:
    """Bytes per directed link per transfer iteration: int64 [P-1, P, P] (src, dst)."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    out = np.zeros((max(P - 1, 0), P, P), dtype=np.int64)
    _check(lib.sp_schedule_link_bytes(kind, P, total_tokens, cu.ctypes.data, len(cu) - 1, int(causal),
                                      seed, bytes_per_token, int(needed_only),
                                      out.ctypes.data if out.size else None),
           "sp_schedule_link_bytes")
    return out


# --------------------------------------------------------------- device calls

def _torch():
    import torch
    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SP_DTYPE_BF16
    if t.dtype == torch.float32:
        return SP_DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _check_qkv(q, k, v):
    _need(q.dim() == 3 and k.dim() == 3 and v.dim() == 3, "q, k, v must be [T, H, d]")
    _need(q.is_cuda and k.is_cuda and v.is_cuda, "q, k, v must be CUDA tensors")
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v must share a dtype")
    T, Hq, d = q.shape
    _need(k.shape == v.shape and k.shape[0] == T and k.shape[2] == d, "k, v must be [T, Hkv, d]")
    return T, Hq, k.shape[1], d


def sp_partial_attn(q, k, v, o_part, lse_part, q_begin: int, q_end: int, kv_begin: int, kv_end: int,
                    cu_seqlens, causal: bool, scale: float | None = None, stream=None):
    """o_part: fp32 [q_end-q_begin, Hq, d]; lse_part: fp32 [Hq, q_end-q_begin] (device)."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    torch = _torch()
    rows = q_end - q_begin
    _need(o_part.dtype == torch.float32 and tuple(o_part.shape) == (rows, Hq, d) and
          o_part.is_contiguous(), "o_part must be fp32 [rows, Hq, d]")
    _need(lse_part.dtype == torch.float32 and tuple(lse_part.shape) == (Hq, rows) and
          lse_part.is_contiguous(), "lse_part must be fp32 [Hq, rows]")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens must be int32 on device")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().sp_partial_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(o_part), _ptr(lse_part), T, Hq, Hkv,
                                  d, _dtype_code(q), q_begin, q_end, kv_begin, kv_end,
                                  _ptr(cu_seqlens), cu_seqlens.numel() - 1, int(causal), scale,
                                  _stream(stream)), "sp_partial_attn")


def sp_lse_merge(o_acc, lse_acc, o_part, lse_part, stream=None):
    """In place: (o_acc, lse_acc) <- merge with (o_part, lse_part). o: [rows, Hq, d], lse: [Hq, rows]."""
    torch = _torch()
    for t in (o_acc, lse_acc, o_part, lse_part):
        _need(t.dtype == torch.float32 and t.is_cuda and t.is_contiguous(), "fp32 contiguous CUDA")
    rows, Hq, d = o_acc.shape
    _need(o_part.shape == o_acc.shape and tuple(lse_acc.shape) == (Hq, rows) and
          lse_part.shape == lse_acc.shape, "shape mismatch")
    _check(load().sp_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_part), _ptr(lse_part), rows, Hq, d,
                               _stream(stream)), "sp_lse_merge")


def sp_packed_attention_workspace_size(n_items: int) -> int:
    return int(load().sp_packed_attention_workspace_size(int(n_items)))


def sp_packed_attention(q, k, v, o, lse, cu_seqlens, causal: bool, items_dev, workspace,
                        scale: float | None = None, stream=None):
    """o: [T, Hq, d] in q's dtype; lse: fp32 [Hq, T]; items_dev: int32 [n, 8] on device;
    workspace: uint8 device tensor of sp_packed_attention_workspace_size(n) bytes."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    torch = _torch()
    _need(o.dtype == q.dtype and tuple(o.shape) == (T, Hq, d) and o.is_contiguous(), "o: [T, Hq, d]")
    _need(lse.dtype == torch.float32 and tuple(lse.shape) == (Hq, T) and lse.is_contiguous(),
          "lse must be fp32 [Hq, T]")
    _need(items_dev.dtype == torch.int32 and items_dev.is_cuda and items_dev.dim() == 2 and
          items_dev.shape[1] == 8 and items_dev.is_contiguous(), "items_dev: int32 [n, 8] on device")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens must be int32 on device")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().sp_packed_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, Hq, Hkv, d,
                                      _dtype_code(q), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                      int(causal), scale, _ptr(items_dev), items_dev.shape[0],
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "sp_packed_attention")


def sp_packed_attention_ex(q, k, v, o, lse, cu_seqlens, causal: bool, items_dev, heads_dev, workspace,
                           scale: float | None = None, stream=None):
    """sp_packed_attention over items with query-head ranges (heads_dev: int32 [n, 2] on device)."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    torch = _torch()
    _need(o.dtype == q.dtype and tuple(o.shape) == (T, Hq, d) and o.is_contiguous(), "o: [T, Hq, d]")
    _need(lse.dtype == torch.float32 and tuple(lse.shape) == (Hq, T) and lse.is_contiguous(),
          "lse must be fp32 [Hq, T]")
    _need(items_dev.dtype == torch.int32 and items_dev.is_cuda and items_dev.dim() == 2 and
          items_dev.shape[1] == 8 and items_dev.is_contiguous(), "items_dev: int32 [n, 8] on device")
    _need(heads_dev.dtype == torch.int32 and heads_dev.is_cuda and tuple(heads_dev.shape) == (items_dev.shape[0], 2)
          and heads_dev.is_contiguous(), "heads_dev: int32 [n, 2] on device")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens must be int32 on device")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().sp_packed_attention_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, Hq, Hkv, d,
                                         _dtype_code(q), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                         int(causal), scale, _ptr(items_dev), _ptr(heads_dev),
                                         items_dev.shape[0], _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)),
           "sp_packed_attention_ex")


def sp_packed_attention_static_ws(q, k, v, o, lse, cu_seqlens, causal: bool, items_dev,
                                  scale: float | None = None, stream=None):
    """sp_packed_attention without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed scratch array is used instead
    (schedules of at most SP_STATIC_WS_MAX_ITEMS items; calls that overlap on
    the GPU race on that array)."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    torch = _torch()
    _need(o.dtype == q.dtype and tuple(o.shape) == (T, Hq, d) and o.is_contiguous(), "o: [T, Hq, d]")
    _need(lse.dtype == torch.float32 and tuple(lse.shape) == (Hq, T) and lse.is_contiguous(),
          "lse must be fp32 [Hq, T]")
    _need(items_dev.dtype == torch.int32 and items_dev.is_cuda and items_dev.dim() == 2 and
          items_dev.shape[1] == 8 and items_dev.is_contiguous(), "items_dev: int32 [n, 8] on device")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens must be int32 on device")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().sp_packed_attention_static_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, Hq,
                                                Hkv, d, _dtype_code(q), _ptr(cu_seqlens),
                                                cu_seqlens.numel() - 1, int(causal), scale,
                                                _ptr(items_dev), items_dev.shape[0],
                                                _stream(stream)), "sp_packed_attention_static_ws")


def sp_packed_attention_backward_workspace_size(n_items: int, T: int, Hq: int) -> int:
    return int(load().sp_packed_attention_backward_workspace_size(int(n_items), int(T), int(Hq)))


def sp_packed_attention_backward(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, causal: bool,
                                 items_dev, workspace, scale: float | None = None, stream=None):
    """Gradients of sp_packed_attention (bf16): dq [T, Hq, d], dk and dv [T, Hkv, d];
    o, lse: the forward's outputs; dout: the gradient of o; workspace: uint8 device
    tensor of sp_packed_attention_backward_workspace_size(n, T, Hq) bytes."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    torch = _torch()
    for name, t, shape in (("o", o, (T, Hq, d)), ("dout", dout, (T, Hq, d)), ("dq", dq, (T, Hq, d)),
                           ("dk", dk, (T, Hkv, d)), ("dv", dv, (T, Hkv, d))):
        _need(t.dtype == q.dtype and tuple(t.shape) == shape and t.is_contiguous() and t.is_cuda,
              f"{name} must be contiguous {q.dtype} {list(shape)} on device")
    _need(lse.dtype == torch.float32 and tuple(lse.shape) == (Hq, T) and lse.is_contiguous(),
          "lse must be fp32 [Hq, T]")
    _need(items_dev.dtype == torch.int32 and items_dev.is_cuda and items_dev.dim() == 2 and
          items_dev.shape[1] == 8 and items_dev.is_contiguous(), "items_dev: int32 [n, 8] on device")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens must be int32 on device")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().sp_packed_attention_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), T, Hq,
        Hkv, d, _dtype_code(q), _ptr(cu_seqlens), cu_seqlens.numel() - 1, int(causal), scale,
        _ptr(items_dev), items_dev.shape[0], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "sp_packed_attention_backward")


def sp_check_device_status(stream=None):
    _check(load().sp_check_device_status(_stream(stream)), "device status")


def sp_check_device_status_code(stream=None) -> int:
    return int(load().sp_check_device_status(_stream(stream)))


def sp_selftest_bounded_wait(timeout_ns: int, stream=None):
    _check(load().sp_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "sp_selftest_bounded_wait")


class PackedAttention:
    """Holds one packing layout's schedule and device buffers; each call runs
    sp_packed_attention. Only buffer management lives here."""

    def __init__(self, cu_seqlens, causal: bool, kind: int, P: int, Hq: int, seed: int = 0,
                 device="cuda", chunking: int = SP_CHUNK_EQUAL, ulysses: int = 1,
                 split_documents: bool = True):
        """ulysses > 1: two-level schedule, P / ulysses groups running `kind`
        between them and a query-head split over `ulysses` ranks inside each.
        split_documents: the schedule's items are cut at document boundaries
        (sp_schedule_split_documents), so that every document of a rank's chunk
        runs as a group of its own, unless that would make more than
        SP_MAX_GROUPS groups (`documents_cut` tells which); False keeps the
        items as built."""
        torch = _torch()
        self.cu_host = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        self.T = int(self.cu_host[-1])
        self.causal = bool(causal)
        self.kind, self.P, self.seed = kind, P, seed
        self.ulysses = int(ulysses)
        _need(self.ulysses >= 1 and P % self.ulysses == 0, "P must be a multiple of ulysses")
        groups = P // self.ulysses
        self.bounds = (None if chunking == SP_CHUNK_EQUAL else
                       sp_chunk_bounds(chunking, groups, self.T, self.cu_host, causal))
        self.heads = None
        if self.ulysses > 1:
            self.items, self.heads = sp_schedule_build_hier(kind, groups, self.ulysses, self.T, self.cu_host,
                                                            causal, Hq, seed, bounds=self.bounds)
        else:
            self.items = sp_schedule_build(kind, P, self.T, self.cu_host, causal, seed, bounds=self.bounds)
        self.documents_cut = False
        if split_documents:
            if self.heads is None:
                cut, cut_heads = sp_schedule_split_documents(self.items, self.cu_host, causal), None
            else:
                cut, cut_heads = sp_schedule_split_documents(self.items, self.cu_host, causal, heads=self.heads)
            # A packing of very many documents keeps the items as built when the
            # cut would pass the group limit of sp_packed_attention.
            if n_groups(cut, cut_heads) <= SP_MAX_GROUPS:
                self.items, self.heads, self.documents_cut = cut, cut_heads, True
        self.cu_dev = torch.from_numpy(self.cu_host).to(device)
        self.items_dev = torch.from_numpy(self.items).to(device)
        self.heads_dev = None if self.heads is None else torch.from_numpy(self.heads).to(device)
        nbytes = sp_packed_attention_workspace_size(len(self.items))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, q, k, v, o=None, lse=None, scale=None, stream=None):
        torch = _torch()
        T, Hq, d = q.shape
        if o is None:
            o = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
        if self.heads_dev is not None:
            sp_packed_attention_ex(q, k, v, o, lse, self.cu_dev, self.causal, self.items_dev, self.heads_dev,
                                   self.workspace, scale=scale, stream=stream)
        else:
            sp_packed_attention(q, k, v, o, lse, self.cu_dev, self.causal, self.items_dev, self.workspace,
                                scale=scale, stream=stream)
        return o, lse

    def backward(self, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, scale=None, stream=None):
        """Gradients (dq, dk, dv) of the forward call that returned (o, lse).
        With a two-level schedule the items of all ranks together cover every
        head and pair, so the gradients are those of all heads too."""
        torch = _torch()
        T, Hq, d = q.shape
        nbytes = sp_packed_attention_backward_workspace_size(len(self.items), T, Hq)
        if getattr(self, "bwd_workspace", None) is None or self.bwd_workspace.numel() < nbytes:
            self.bwd_workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        sp_packed_attention_backward(q, k, v, o, dout, lse, dq, dk, dv, self.cu_dev, self.causal,
                                     self.items_dev, self.bwd_workspace, scale=scale, stream=stream)
        return dq, dk, dv
