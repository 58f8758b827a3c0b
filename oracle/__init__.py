"""fp64 CPU oracle for blockwise packed attention and its chunk schedules.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU baseline
leg of the benchmark are the only callers. The product package never imports
this module, and this module imports nothing from the product.

The arithmetic lives in ``oracle.cpp`` (plain C++, double precision, OpenMP
over rows); this file builds it with g++ and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lib = None

DT_F64, DT_F32, DT_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (OpenMP) if it is missing or stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Declares the argument and result types of every exported function of a
    loaded oracle library (the built one, or a test's variant of the source)."""
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    lib.oracle_attn.restype = ctypes.c_int
    lib.oracle_attn.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int,
                                ctypes.c_double, ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                ctypes.c_int, f64p, f64p, ctypes.c_int]
    lib.oracle_attn_backward.restype = ctypes.c_int
    lib.oracle_attn_backward.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_double, f64p, f64p, f64p,
                                         ctypes.c_int]
    lib.oracle_attn_backward_sampled.restype = ctypes.c_int
    lib.oracle_attn_backward_sampled.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double, i32p,
                                                 ctypes.c_int, f64p, i32p, ctypes.c_int, f64p, f64p,
                                                 ctypes.c_int]
    lib.oracle_lse_merge.restype = None
    lib.oracle_lse_merge.argtypes = [f64p, f64p, f64p, f64p, ctypes.c_longlong, ctypes.c_int,
                                     f64p, f64p]
    lib.oracle_valid_pairs.restype = ctypes.c_longlong
    lib.oracle_valid_pairs.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_closed_form_schedule.restype = ctypes.c_longlong
    lib.oracle_closed_form_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p,
                                                ctypes.c_int, ctypes.c_int, i32p,
                                                ctypes.c_longlong]
    lib.oracle_check_hamiltonian.restype = ctypes.c_int
    lib.oracle_check_hamiltonian.argtypes = [ctypes.c_int, i32p]
    lib.oracle_check_schedule.restype = ctypes.c_int
    lib.oracle_check_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p,
                                          ctypes.c_int, ctypes.c_int, i32p, ctypes.c_longlong,
                                          i32p, ctypes.c_int, ctypes.c_char_p, ctypes.c_int, i32p]
    lib.oracle_check_hier_schedule.restype = ctypes.c_int
    lib.oracle_check_hier_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, i32p,
                                               i32p, ctypes.c_longlong, i32p, ctypes.c_int,
                                               ctypes.c_char_p, ctypes.c_int, i32p]
    lib.oracle_link_bytes_hier.restype = ctypes.c_int
    lib.oracle_link_bytes_hier.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p,
                                           ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)]
    lib.oracle_chunk_bounds.restype = ctypes.c_int
    lib.oracle_chunk_bounds.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                        ctypes.c_int, i32p]
    lib.oracle_link_bytes.restype = ctypes.c_int
    lib.oracle_link_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                      ctypes.c_int, i32p, ctypes.c_longlong, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_longlong)]
    lib.oracle_check_cu_seqlens.restype = ctypes.c_int
    lib.oracle_check_cu_seqlens.argtypes = [i32p, ctypes.c_int, ctypes.c_int]
    lib.oracle_doc_of.restype = ctypes.c_int
    lib.oracle_doc_of.argtypes = [i32p, ctypes.c_int, ctypes.c_int]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as_input(x):
    """Returns (contiguous array, dtype code). bf16 data is passed as uint16 bits."""
    if x.dtype == np.float64:
        return np.ascontiguousarray(x), DT_F64
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), DT_F32
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), DT_BF16
    raise TypeError(f"oracle input dtype {x.dtype} not supported")


def attn(q, k, v, cu_seqlens, causal: bool, scale: float | None = None, rows=None,
         kv_range=None, threads: int = 0, q_rows_only: bool = False):
    """Exact attention in fp64.

    q: [T, Hq, d] (or [len(rows), Hq, d] with q_rows_only); k, v: [T, Hkv, d]
    (float64, float32, or uint16 bf16 bits). rows: query tokens to evaluate
    (default all). kv_range: (kv_begin, kv_end).
    Returns (o [n, Hq, d] float64, lse [n, Hq] float64), n = len(rows).
    """
    lib = _load()
    q, dt = _as_input(q)
    k, dk = _as_input(k)
    v, dv = _as_input(v)
    assert dt == dk == dv, "q, k, v must share a dtype"
    _, Hq, d = q.shape
    T, Hkv = k.shape[0], k.shape[1]
    assert k.shape == (T, Hkv, d) and v.shape == (T, Hkv, d)
    assert q_rows_only or q.shape[0] == T
    cu, cup = _i32(cu_seqlens)
    ndocs = len(cu) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if rows is None:
        assert not q_rows_only
        rows_arr, rowsp, n = None, None, T
    else:
        rows_arr, rowsp = _i32(rows)
        n = len(rows_arr)
        assert not q_rows_only or q.shape[0] == n
    kb, ke = (0, T) if kv_range is None else kv_range
    o = np.empty((n, Hq, d), dtype=np.float64)
    lse = np.empty((n, Hq), dtype=np.float64)
    rc = lib.oracle_attn(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, T, Hq, Hkv, d, cup,
                         ndocs, int(causal), float(scale), int(kb), int(ke), rowsp, n,
                         int(q_rows_only), o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn rejected its arguments (code {rc})")
    return o, lse


def attn_backward(q, k, v, dout, cu_seqlens, causal: bool, scale: float | None = None,
                  threads: int = 0):
    """Gradients (dq [T,Hq,d], dk [T,Hkv,d], dv [T,Hkv,d]) in fp64 of the masked
    attention for the output gradient dout [T,Hq,d]."""
    lib = _load()
    q, dt = _as_input(q)
    k, dk_ = _as_input(k)
    v, dv_ = _as_input(v)
    dout, dd = _as_input(dout)
    assert dt == dk_ == dv_ == dd
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu, cup = _i32(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.empty((T, Hq, d))
    dk = np.empty((T, Hkv, d))
    dv = np.empty((T, Hkv, d))
    f = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_attn_backward(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dt,
                                  T, Hq, Hkv, d, cup, len(cu) - 1, int(causal), float(scale),
                                  f(dq), f(dk), f(dv), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_backward rejected its arguments (code {rc})")
    return dq, dk, dv


def attn_backward_sampled(q, k, v, dout, cu_seqlens, causal: bool, qrows=(), krows=(),
                          scale: float | None = None, threads: int = 0):
    """fp64 gradients at chosen outputs: dq of the rows qrows [nq, Hq, d], and
    dk, dv of the keys krows [nk, Hkv, d]. Same definitions as attn_backward."""
    lib = _load()
    q, dt = _as_input(q)
    k, dk_ = _as_input(k)
    v, dv_ = _as_input(v)
    dout, dd = _as_input(dout)
    assert dt == dk_ == dv_ == dd
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu, cup = _i32(cu_seqlens)
    qr, qrp = _i32(np.asarray(qrows, dtype=np.int64).reshape(-1))
    kr, krp = _i32(np.asarray(krows, dtype=np.int64).reshape(-1))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.empty((len(qr), Hq, d))
    dk = np.empty((len(kr), Hkv, d))
    dv = np.empty((len(kr), Hkv, d))
    f = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_attn_backward_sampled(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                          dt, T, Hq, Hkv, d, cup, len(cu) - 1, int(causal), float(scale),
                                          qrp, len(qr), f(dq), krp, len(kr), f(dk), f(dv), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_backward_sampled rejected its arguments (code {rc})")
    return dq, dk, dv


def lse_merge(o1, l1, o2, l2):
    """Merge two normalised partials. o*: [..., d], l*: [...]. Returns (o, lse)."""
    lib = _load()
    d = o1.shape[-1]
    n = int(np.prod(l1.shape))
    o1c, o1p = _f64(o1)
    o2c, o2p = _f64(o2)
    l1c, l1p = _f64(l1)
    l2c, l2p = _f64(l2)
    o = np.empty(o1.shape, dtype=np.float64)
    lo = np.empty(l1.shape, dtype=np.float64)
    lib.oracle_lse_merge(o1p, l1p, o2p, l2p, n, d, o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         lo.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return o, lo


def valid_pairs(cu_seqlens, causal: bool, qa: int, qb: int, ka: int, kb: int) -> int:
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    return int(lib.oracle_valid_pairs(cup, len(cu) - 1, int(causal), qa, qb, ka, kb))


def doc_of(cu_seqlens, t: int) -> int:
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    return int(lib.oracle_doc_of(cup, len(cu) - 1, int(t)))


def check_cu_seqlens(cu_seqlens, T: int) -> int:
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    return int(lib.oracle_check_cu_seqlens(cup, len(cu) - 1, int(T)))


def closed_form_schedule(kind: int, P: int, T: int, cu_seqlens, causal: bool):
    """Expected RING (0) / ZIGZAG (1) items [n, 8] (flags column left 0), or None."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    n = lib.oracle_closed_form_schedule(kind, P, T, cup, len(cu) - 1, int(causal), None, 0)
    if n < 0:
        return None
    out = np.zeros((max(n, 1), 8), dtype=np.int32)
    lib.oracle_closed_form_schedule(kind, P, T, cup, len(cu) - 1, int(causal),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n)
    return out[:n]


def check_hamiltonian(P: int, succ) -> int:
    lib = _load()
    s, sp = _i32(succ)
    return int(lib.oracle_check_hamiltonian(P, sp))


def check_schedule(kind: int, P: int, T: int, cu_seqlens, causal: bool, items, succ=None,
                   brute: bool = False, bounds=None):
    """Returns (code, message); code 0 means every property holds. bounds:
    chunk boundaries [P+1] of a RING or TASP schedule (None: equal chunks)."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    it, itp = _i32(np.asarray(items).reshape(-1, 8))
    if succ is None:
        succ = np.zeros((max(P - 1, 1), max(P, 1)), dtype=np.int32)
    sc, scp = _i32(succ)
    bp = None
    if bounds is not None:
        bd, bp = _i32(bounds)
    buf = ctypes.create_string_buffer(256)
    rc = lib.oracle_check_schedule(kind, P, T, cup, len(cu) - 1, int(causal), itp, len(it), scp,
                                   int(brute), buf, 256, bp)
    return int(rc), buf.value.decode()


def check_hier_schedule(kind: int, R: int, U: int, Hq: int, T: int, cu_seqlens, causal: bool, items, heads,
                        succ=None, brute: bool = False, bounds=None):
    """Two-level schedule check; returns (code, message), 0 when every property holds."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    it, itp = _i32(np.asarray(items).reshape(-1, 8))
    hd, hdp = _i32(np.asarray(heads).reshape(-1, 2))
    if succ is None:
        succ = np.zeros((max(R - 1, 1), max(R, 1)), dtype=np.int32)
    sc, scp = _i32(succ)
    bp = None
    if bounds is not None:
        bd, bp = _i32(bounds)
    buf = ctypes.create_string_buffer(256)
    rc = lib.oracle_check_hier_schedule(kind, R, U, Hq, T, cup, len(cu) - 1, int(causal), itp, hdp, len(it),
                                        scp, int(brute), buf, 256, bp)
    return int(rc), buf.value.decode()


def link_bytes_hier(kind: int, R: int, U: int, T: int, cu_seqlens, causal: bool, Hq: int, Hkv: int, d: int,
                    elem_bytes: int = 2, succ=None, needed_only: bool = False):
    """Two-level communication restated per token and head: (intra [P, P], inter [R-1, P, P])."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    if succ is None:
        succ = np.zeros((max(R - 1, 1), max(R, 1)), dtype=np.int32)
    sc, scp = _i32(succ)
    P = R * U
    intra = np.zeros((P, P), dtype=np.int64)
    inter = np.zeros((max(R - 1, 1), P, P), dtype=np.int64)
    ll = ctypes.POINTER(ctypes.c_longlong)
    rc = lib.oracle_link_bytes_hier(kind, R, U, T, cup, len(cu) - 1, int(causal), scp, Hq, Hkv, d, elem_bytes,
                                    int(needed_only), intra.ctypes.data_as(ll), inter.ctypes.data_as(ll))
    if rc != 0:
        raise ValueError(f"oracle_link_bytes_hier rejected its arguments (code {rc})")
    return intra, inter[:max(R - 1, 0)]


def chunk_bounds(mode: int, P: int, T: int, cu_seqlens, causal: bool):
    """Chunk boundaries [P+1] of a chunking policy (0 equal, 1 balanced work,
    2 balanced then moved onto document starts that are near in work)."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    out = np.zeros(P + 1, dtype=np.int32)
    rc = lib.oracle_chunk_bounds(int(mode), int(P), int(T), cup, len(cu) - 1, int(causal),
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    if rc != 0:
        raise ValueError(f"oracle_chunk_bounds rejected its arguments (code {rc})")
    return out


def link_bytes(kind: int, P: int, T: int, cu_seqlens, causal: bool, succ=None,
               bytes_per_token: int = 1, needed_only: bool = False):
    """Bytes per directed link per AllGather iteration, int64 [P-1, P, P] (src, dst)."""
    lib = _load()
    cu, cup = _i32(cu_seqlens)
    if succ is None:
        succ = np.zeros((max(P - 1, 1), max(P, 1)), dtype=np.int32)
    sc, scp = _i32(succ)
    out = np.zeros((max(P - 1, 1), P, P), dtype=np.int64)
    rc = lib.oracle_link_bytes(kind, P, T, cup, len(cu) - 1, int(causal), scp, int(bytes_per_token),
                               int(needed_only), out.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)))
    if rc != 0:
        raise ValueError(f"oracle_link_bytes rejected its arguments (code {rc})")
    return out[:max(P - 1, 0)]
