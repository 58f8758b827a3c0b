"""sp_packed_attention_static_ws: the entry point for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, a
binding without a CUDA allocator, a serving loop that must not call
cudaMalloc/cudaFree while it runs). It uses the library's fixed scratch array
instead of a caller workspace. Here it is called through the C-ABI twice in a
row, on two different packing layouts, and each result is compared with the
workspace entry point's on the same inputs."""
import ctypes

import numpy as np
import pytest

import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O

pytestmark = pytest.mark.gpu

MAX_ITEMS = 40000  # SP_STATIC_WS_MAX_ITEMS in include/sp_attn.h


def _case(T, docs, Hq, Hkv, kind, P, seed):
    import torch
    cu = wl.cu_from_lengths(docs)
    q = wl.random_normal((T, Hq, 128), seed, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, 128), seed + 1, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, 128), seed + 2, "cuda", "bf16")
    items = sb.sp_schedule_build(kind, P, T, cu, True, seed=seed)
    return cu, q, k, v, items


def test_static_scratch_entry_point_matches_workspace_entry_point():
    import torch
    cases = [(3000, [1000, 17, 1983], 8, 2, sb.SP_SCHED_TASP, 7, 1),
             (2048, [2048], 4, 4, sb.SP_SCHED_ZIGZAG, 4, 2)]
    for T, docs, Hq, Hkv, kind, P, seed in cases:
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
        rc = sb.load().sp_packed_attention_static_ws(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), T, Hq, Hkv, 128, sb.SP_DTYPE_BF16,
            ctypes.c_void_p(cu_dev.data_ptr()), len(cu) - 1, 1, 1.0 / np.sqrt(128.0),
            ctypes.c_void_p(items_dev.data_ptr()), len(items),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, sb.sp_status_string(rc)
        sb.sp_check_device_status()
        assert float((o.float() - o_ref.float()).abs().max()) <= TOL_BF16_O
        assert float((lse - l_ref).abs().max()) <= TOL_BF16_LSE


def test_static_scratch_rejects_oversized_schedule():
    lib = sb.load()
    fake = ctypes.c_void_p(0x100000)
    rc = lib.sp_packed_attention_static_ws(fake, fake, fake, fake, fake, 1024, 4, 4, 128, 0, fake, 1,
                                           1, 0.1, fake, MAX_ITEMS + 1, None)
    assert rc == 3  # SP_ERR_BUFFER_TOO_SMALL, nothing launched
