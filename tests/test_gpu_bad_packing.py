"""The packing descriptor on the device is checked before anything is written.

A malformed device cu_seqlens (not starting at 0, not ending at T, not
strictly increasing), or one that differs from the descriptor the schedule was
built from so that some item holds no valid pair, would silently change the
masks: packed documents would attend across their boundaries, the
cross-contamination the HSAP abstract names. The forward's set-up kernel and
the backward's row-dot kernel reject such a descriptor with SP_ERR_INTERNAL and
leave every output untouched. Bad inputs only: nothing here faults a GPU.
"""
import numpy as np
import pytest

import sequence_blockwise_gb300 as sb

pytestmark = pytest.mark.gpu

T, HQ, HKV, D = 512, 2, 2, 128
MALFORMED = ([0, 300, 200, 512], [0, 256, 500], [1, 256, 512], [0, 256, 256, 512])


def _torch():
    import torch
    return torch


def _inputs(seed=5):
    torch = _torch()
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda h: torch.randn((T, h, D), generator=g, device="cuda").to(torch.bfloat16)
    return mk(HQ), mk(HKV), mk(HKV)


def _forward(q, k, v, cu_dev, items):
    torch = _torch()
    items_dev = torch.from_numpy(items).cuda()
    ws = torch.empty(sb.sp_packed_attention_workspace_size(len(items)), dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((HQ, T), 7.0, dtype=torch.float32, device="cuda")
    sb.sp_packed_attention(q, k, v, o, lse, cu_dev, True, items_dev, ws)
    return o, lse


def test_forward_rejects_malformed_or_mismatched_descriptor():
    torch = _torch()
    sb.sp_check_device_status()
    q, k, v = _inputs()
    # A single-document schedule: its items attend across the middle of [0, T).
    items = sb.sp_schedule_build(sb.SP_SCHED_RING, 4, T, [0, T], True)
    # [0, 256, 512] is well formed, but the item of rows [256, 384) over keys
    # [0, 128) holds no valid pair under it: the schedule was built for another
    # packing.
    for cu in MALFORMED + ([0, 256, 512],):
        cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
        o, lse = _forward(q, k, v, cu_dev, items)
        assert sb.sp_check_device_status_code() == 6, cu  # SP_ERR_INTERNAL
        assert bool((o == 7.0).all()) and bool((lse == 7.0).all()), cu
    # The matching descriptor runs and clears nothing it should not.
    o, lse = _forward(q, k, v, torch.tensor([0, T], dtype=torch.int32, device="cuda"), items)
    assert sb.sp_check_device_status_code() == 0
    assert bool(torch.isfinite(lse).all()) and not bool((o == 7.0).any())


def test_backward_rejects_malformed_descriptor():
    torch = _torch()
    sb.sp_check_device_status()
    q, k, v = _inputs(6)
    items = sb.sp_schedule_build(sb.SP_SCHED_RING, 4, T, [0, T], True)
    items_dev = torch.from_numpy(items).cuda()
    good = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    o, lse = _forward(q, k, v, good, items)
    assert sb.sp_check_device_status_code() == 0
    dout = torch.randn_like(q.float()).to(torch.bfloat16)
    ws = torch.empty(sb.sp_packed_attention_backward_workspace_size(len(items), T, HQ), dtype=torch.uint8,
                     device="cuda")
    for cu in MALFORMED:
        dq, dk, dv = torch.full_like(q, 3.0), torch.full_like(k, 3.0), torch.full_like(v, 3.0)
        sb.sp_packed_attention_backward(q, k, v, o, dout, lse, dq, dk, dv,
                                        torch.tensor(cu, dtype=torch.int32, device="cuda"), True,
                                        items_dev, ws)
        assert sb.sp_check_device_status_code() == 6, cu
        assert bool((dq == 3.0).all()) and bool((dk == 3.0).all()) and bool((dv == 3.0).all()), cu
    # The same workspace serves a good call right after.
    dq, dk, dv = torch.full_like(q, 3.0), torch.full_like(k, 3.0), torch.full_like(v, 3.0)
    sb.sp_packed_attention_backward(q, k, v, o, dout, lse, dq, dk, dv, good, True, items_dev, ws)
    assert sb.sp_check_device_status_code() == 0
    assert not bool((dq == 3.0).any()) and not bool((dk == 3.0).any())
