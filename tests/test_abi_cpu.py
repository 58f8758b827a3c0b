"""The C-ABI library loads, exports every symbol include/sp_attn.h declares, and
rejects bad arguments before touching a device (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import sequence_blockwise_gb300 as sb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "sp_attn.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported():
    lib = sb.load()
    syms = declared_symbols()
    assert "sp_packed_attention" in syms and len(syms) >= 9
    for name in syms:
        assert hasattr(lib, name), name
    assert sorted(sb.EXPORTED) == syms


def test_status_strings():
    assert sb.sp_status_string(0) == "SP_OK"
    assert sb.sp_status_string(5) == "SP_ERR_TIMEOUT"
    assert sb.sp_status_string(99) == "SP_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x100000)  # aligned, never dereferenced by the checks below


def _partial(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, T=256, Hq=4, Hkv=2, d=128, dtype=0, qb=0,
                qe=128, kb=0, ke=128, cu=FAKE, nd=1, causal=1, scale=0.125)
    args.update(kw)
    a = args
    return sb.load().sp_partial_attn(a["q"], a["k"], a["v"], a["o"], a["lse"], a["T"], a["Hq"],
                                     a["Hkv"], a["d"], a["dtype"], a["qb"], a["qe"], a["kb"], a["ke"],
                                     a["cu"], a["nd"], a["causal"], a["scale"], None)


def test_partial_argument_checks():
    assert _partial(d=96) == 2                       # unsupported head dim
    assert _partial(d=0) == 1
    assert _partial(Hq=3, Hkv=2) == 1                # Hq % Hkv
    assert _partial(scale=0.0) == 1
    assert _partial(scale=float("nan")) == 1
    assert _partial(qb=10, qe=5) == 1
    assert _partial(qe=300) == 1
    assert _partial(kb=-1) == 1
    assert _partial(dtype=7) == 1
    assert _partial(nd=0) == 1
    assert _partial(q=None) == 1
    assert _partial(o=ctypes.c_void_p(0x100004)) == 1  # misaligned
    assert _partial(qb=5, qe=5) == 0                 # empty row range: no work, no device call


def test_merge_and_packed_argument_checks():
    lib = sb.load()
    assert lib.sp_lse_merge(FAKE, FAKE, FAKE, FAKE, 0, 4, 128, None) == 0
    assert lib.sp_lse_merge(FAKE, FAKE, FAKE, FAKE, 10, 4, 6, None) == 1
    assert lib.sp_lse_merge(FAKE, FAKE, FAKE, FAKE, -1, 4, 128, None) == 1
    assert lib.sp_lse_merge(None, FAKE, FAKE, FAKE, 4, 4, 128, None) == 1

    def packed(n_items=10, ws_bytes=None, **kw):
        ws = sb.sp_packed_attention_workspace_size(n_items) if ws_bytes is None else ws_bytes
        a = dict(T=512, Hq=4, Hkv=4, d=128, dtype=0, nd=1, causal=1, scale=0.1, items=FAKE)
        a.update(kw)
        return lib.sp_packed_attention(FAKE, FAKE, FAKE, FAKE, FAKE, a["T"], a["Hq"], a["Hkv"], a["d"],
                                       a["dtype"], FAKE, a["nd"], a["causal"], a["scale"], a["items"],
                                       n_items, FAKE, ws, None)

    assert packed(n_items=-1) == 1
    assert packed(n_items=0) == 0
    assert packed(T=0) == 0
    assert packed(items=None) == 1
    assert packed(d=32) == 2
    assert packed(ws_bytes=16) == 3
    assert sb.sp_packed_attention_workspace_size(0) > 0
    assert sb.sp_packed_attention_workspace_size(1000) >= 1000 * 64


def test_schedule_argument_checks():
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_TASP, 4, 256, [0, 256], True)
    assert e.value.code == 2
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_TASP, 6, 256, [0, 256], True)
    assert e.value.code == 2
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_ZIGZAG, 3, 256, [0, 256], True)  # 256 % 6 != 0
    assert e.value.code == 2
    for bad_cu in ([0, 100], [1, 256], [0, 100, 100, 256], [0, 300, 256]):
        with pytest.raises(sb.SpError) as e:
            sb.sp_schedule_build(sb.SP_SCHED_RING, 4, 256, bad_cu, True)
        assert e.value.code == 1
    with pytest.raises(sb.SpError):
        sb.sp_schedule_build(sb.SP_SCHED_RING, 0, 256, [0, 256], True)
    # Two-call protocol: a short buffer reports the needed count.
    lib = sb.load()
    cu = np.array([0, 256], dtype=np.int32)
    n = ctypes.c_int64(0)
    assert lib.sp_schedule_build(0, 4, 256, cu.ctypes.data, 1, 1, 0, None, ctypes.byref(n)) == 0
    assert n.value == 10
    buf = np.zeros((3, 8), dtype=np.int32)
    cap = ctypes.c_int64(3)
    assert lib.sp_schedule_build(0, 4, 256, cu.ctypes.data, 1, 1, 0, buf.ctypes.data,
                                 ctypes.byref(cap)) == 3
    assert cap.value == 10
    # Empty sequence.
    assert len(sb.sp_schedule_build(sb.SP_SCHED_RING, 4, 0, [0], True)) == 0


def test_backward_argument_checks():
    lib = sb.load()

    def bwd(n_items=10, ws_bytes=None, **kw):
        a = dict(T=512, Hq=4, Hkv=2, d=128, dtype=0, nd=1, causal=1, scale=0.1, items=FAKE,
                 dq=FAKE, dout=FAKE)
        a.update(kw)
        ws = (sb.sp_packed_attention_backward_workspace_size(n_items, a["T"], a["Hq"])
              if ws_bytes is None else ws_bytes)
        return lib.sp_packed_attention_backward(FAKE, FAKE, FAKE, FAKE, a["dout"], FAKE, a["dq"], FAKE,
                                                FAKE, a["T"], a["Hq"], a["Hkv"], a["d"], a["dtype"],
                                                FAKE, a["nd"], a["causal"], a["scale"], a["items"],
                                                n_items, FAKE, ws, None)

    assert bwd(dtype=1) == 2                      # fp32 backward not offered
    assert bwd(d=32) == 2
    assert bwd(Hq=3) == 1
    assert bwd(T=0) == 0
    assert bwd(n_items=0) == 1                    # T > 0 needs a schedule
    assert bwd(n_items=-3) == 1
    assert bwd(ws_bytes=64) == 3
    assert bwd(dout=None) == 1
    assert bwd(dq=ctypes.c_void_p(0x100008)) == 1  # misaligned
    assert bwd(items=None) == 1
    # Two fp32 [Hq][T] row vectors and the fp32 [T][Hq][128] dQ accumulator; the
    # item count does not enter.
    need = 2 * 512 * 4 * 4 + 512 * 4 * 128 * 4
    assert sb.sp_packed_attention_backward_workspace_size(10, 512, 4) >= need
    assert (sb.sp_packed_attention_backward_workspace_size(10, 512, 4)
            == sb.sp_packed_attention_backward_workspace_size(10 ** 6, 512, 4))


def test_packed_ex_and_static_ws_argument_checks():
    lib = sb.load()
    max_items = int(re.search(r"#define SP_STATIC_WS_MAX_ITEMS (\d+)", open(HEADER).read()).group(1))
    base = dict(T=512, Hq=4, Hkv=4, d=128, dtype=0, nd=1, causal=1, scale=0.1)

    def ex(n_items=10, ws_bytes=None, q=FAKE, heads=FAKE, **kw):
        ws = sb.sp_packed_attention_workspace_size(n_items) if ws_bytes is None else ws_bytes
        a = dict(base, **kw)
        return lib.sp_packed_attention_ex(q, FAKE, FAKE, FAKE, FAKE, a["T"], a["Hq"], a["Hkv"], a["d"],
                                          a["dtype"], FAKE, a["nd"], a["causal"], a["scale"], FAKE, heads,
                                          n_items, FAKE, ws, None)

    assert ex(n_items=-1) == 1
    assert ex(n_items=0) == 0 and ex(T=0) == 0
    assert ex(q=None) == 1
    assert ex(q=ctypes.c_void_p(0x100008)) == 1        # device pointers: 16-byte aligned
    assert ex(heads=ctypes.c_void_p(0x100004)) == 1    # head ranges: int32 pairs, 8-byte aligned
    assert ex(d=32) == 2 and ex(Hq=6, Hkv=4) == 1 and ex(scale=float("inf")) == 1
    assert ex(ws_bytes=16) == 3

    def static(n_items=10, **kw):
        a = dict(base, **kw)
        return lib.sp_packed_attention_static_ws(FAKE, FAKE, FAKE, FAKE, FAKE, a["T"], a["Hq"], a["Hkv"],
                                                 a["d"], a["dtype"], FAKE, a["nd"], a["causal"], a["scale"],
                                                 FAKE, n_items, None)

    assert static(n_items=max_items + 1) == 3
    assert static(d=32) == 2 and static(scale=0.0) == 1 and static(Hq=3, Hkv=2) == 1
    assert static(n_items=-1) == 1
    assert static(n_items=0) == 0 and static(T=0) == 0
