"""The multi-GPU split of the benchmark on one GPU: GPU g of N runs the items of
the virtual ranks r with r mod N = g. The GPUs' launches do not wait on one
another (each writes only its own Q chunks), so running every GPU's share in
turn on this device, into one output buffer, must give exactly the result of
the whole schedule in one launch: every row is computed by the same kernel
walk over the same items of its group, whichever launch it is in. Rows a share
does not own stay untouched."""
import numpy as np
import pytest

import bench
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _case(T, docs, Hq, Hkv, seed):
    cu = wl.cu_from_lengths(docs)
    q = wl.random_normal((T, Hq, 128), seed, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, 128), seed + 1, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, 128), seed + 2, "cuda", "bf16")
    return cu, q, k, v


@pytest.mark.parametrize("kind,P,T,docs", [(sb.SP_SCHED_ZIGZAG, 8, 8192, [8192]),
                                           (sb.SP_SCHED_TASP, 8, 12000, [3000, 517, 6000, 2483]),
                                           (sb.SP_SCHED_RING, 5, 7000, [1, 4000, 2999])],
                         ids=["zigzag8", "tasp8-packed", "ring5-packed"])
def test_split_shares_reproduce_the_whole_schedule(kind, P, T, docs):
    import torch
    Hq, Hkv = 8, 2
    cu, q, k, v = _case(T, docs, Hq, Hkv, 11 + P)
    cu_dev = torch.from_numpy(cu).cuda()
    items = sb.sp_schedule_build(kind, P, T, cu, True, seed=3)
    ws = torch.empty(sb.sp_packed_attention_workspace_size(len(items)), dtype=torch.uint8, device="cuda")
    o_ref = torch.empty_like(q)
    l_ref = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    sb.sp_packed_attention(q, k, v, o_ref, l_ref, cu_dev, True, torch.from_numpy(items).cuda(), ws)
    for N in (2, 3, 4):
        o = torch.full_like(q, 5.0)
        lse = torch.full((Hq, T), 5.0, dtype=torch.float32, device="cuda")
        owned = np.zeros(T, dtype=bool)
        for g in range(N):
            mine = bench.split_items(items, N, g)
            if len(mine) == 0:
                continue
            sb.sp_packed_attention(q, k, v, o, lse, cu_dev, True, torch.from_numpy(mine).cuda(), ws)
            rows = bench.row_intervals(mine)
            for a, b in rows:
                assert not owned[a:b].any()  # no row is written by two shares
                owned[a:b] = True
        sb.sp_check_device_status()
        assert owned.all()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), N
