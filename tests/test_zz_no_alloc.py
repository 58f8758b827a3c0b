"""sp_packed_attention_static_ws: the entry point for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, a
binding without a CUDA allocator, a serving loop that must not call
cudaMalloc/cudaFree while it runs). It uses the library's fixed scratch array
instead of a caller workspace.

Called through the C-ABI twice in a row, on two different packing layouts:
each result must be bit-identical to the workspace entry point's on the same
inputs (same kernels, same schedule), and the first case is also held to the
oracle. A second call on the same device must not change the free device
memory or torch's allocator: the entry point allocates nothing. This file is
collected last, so that a run stopping at the first failure has run every
other test before it; it passes alone in a fresh process too."""
import ctypes
import os
import re

import numpy as np
import pytest

import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, max_errs, oracle_rows

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(__file__), "..", "include", "sp_attn.h")
MAX_ITEMS = int(re.search(r"#define SP_STATIC_WS_MAX_ITEMS (\d+)", open(HEADER).read()).group(1))


def _case(T, docs, Hq, Hkv, kind, P, seed):
    cu = wl.cu_from_lengths(docs)
    q = wl.random_normal((T, Hq, 128), seed, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, 128), seed + 1, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, 128), seed + 2, "cuda", "bf16")
    items = sb.sp_schedule_build(kind, P, T, cu, True, seed=seed)
    return cu, q, k, v, items


def _static_ws_abi(q, k, v, o, lse, cu_dev, ndocs, items_dev, n_items):
    import torch
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    return sb.load().sp_packed_attention_static_ws(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), T, Hq, Hkv, 128, sb.SP_DTYPE_BF16,
        ctypes.c_void_p(cu_dev.data_ptr()), ndocs, 1, 1.0 / np.sqrt(128.0),
        ctypes.c_void_p(items_dev.data_ptr()), n_items,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_entry_point_matches_workspace_entry_point():
    import torch
    cases = [(3000, [1000, 17, 1983], 8, 2, sb.SP_SCHED_TASP, 7, 1),
             (2048, [2048], 4, 4, sb.SP_SCHED_ZIGZAG, 4, 2)]
    for ci, (T, docs, Hq, Hkv, kind, P, seed) in enumerate(cases):
        cu, q, k, v, items = _case(T, docs, Hq, Hkv, kind, P, seed)
        cu_dev = torch.from_numpy(cu).cuda()
        items_dev = torch.from_numpy(items).cuda()
        # Reference: the workspace entry point.
        ws = torch.empty(sb.sp_packed_attention_workspace_size(len(items)), dtype=torch.uint8,
                         device="cuda")
        o_ref = torch.empty_like(q)
        l_ref = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
        sb.sp_packed_attention(q, k, v, o_ref, l_ref, cu_dev, True, items_dev, ws)
        # Allocation-free entry point, straight through the C-ABI.
        o = torch.empty_like(q)
        lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
        rc = _static_ws_abi(q, k, v, o, lse, cu_dev, len(cu) - 1, items_dev, len(items))
        assert rc == 0, sb.sp_status_string(rc)
        sb.sp_check_device_status()
        # The same kernels on the same schedule: bit-identical.
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        if ci == 0:
            # And held to the oracle, every row.
            rows = np.arange(T)
            o_or, l_or = oracle_rows(q, k, v, cu, True, rows)
            eo, el = max_errs(o.double().cpu().numpy(), lse.double().cpu().numpy().T, o_or, l_or)
            assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_static_scratch_allocates_nothing():
    import torch
    T, docs, Hq, Hkv, kind, P, seed = 4096, [1500, 2596], 8, 2, sb.SP_SCHED_RING, 8, 3
    cu, q, k, v, items = _case(T, docs, Hq, Hkv, kind, P, seed)
    cu_dev = torch.from_numpy(cu).cuda()
    items_dev = torch.from_numpy(items).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    o2 = torch.empty_like(q)
    lse2 = torch.empty_like(lse)
    # The first call on a device (here through the Python binding) looks up the
    # scratch array's address; the kernels are loaded by then.
    sb.sp_packed_attention_static_ws(q, k, v, o, lse, cu_dev, True, items_dev)
    torch.cuda.synchronize()
    sb.sp_check_device_status()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    rc = _static_ws_abi(q, k, v, o2, lse2, cu_dev, len(cu) - 1, items_dev, len(items))
    assert rc == 0, sb.sp_status_string(rc)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert (free1, torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == (free0, alloc0, reserved0)
    sb.sp_check_device_status()
    # Two calls in a row give the same result.
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_static_scratch_rejects_oversized_schedule():
    lib = sb.load()
    fake = ctypes.c_void_p(0x100000)
    rc = lib.sp_packed_attention_static_ws(fake, fake, fake, fake, fake, 1024, 4, 4, 128, 0, fake, 1,
                                           1, 0.1, fake, MAX_ITEMS + 1, None)
    assert rc == 3  # SP_ERR_BUFFER_TOO_SMALL, nothing launched
