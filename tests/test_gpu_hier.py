"""GPU parity of two-level schedules (Inter-SP schedule between groups,
query heads split inside a group) run through sp_packed_attention_ex: every
row and head against the fp64 oracle on small packings (head slices of whole
key/value groups, slices inside one group, MHA), the 64K full-mask workload as
2 groups x 8 at full size on sampled rows, one head slice alone (other heads
untouched), and a head range that straddles key/value groups rejected."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, host_inputs, max_errs, oracle_rows, row_cost, sample_rows

pytestmark = pytest.mark.gpu


def _inputs(T, Hq, Hkv, seed):
    return (wl.random_normal((T, Hq, 128), seed, "cuda", "bf16"),
            wl.random_normal((T, Hkv, 128), seed + 1, "cuda", "bf16"),
            wl.random_normal((T, Hkv, 128), seed + 2, "cuda", "bf16"))


CASES = [
    # Hq, Hkv, kind, groups, ulysses, causal
    (8, 4, sb.SP_SCHED_RING, 2, 2, True),     # slices of 4 heads = 2 whole KV groups
    (8, 2, sb.SP_SCHED_TASP, 3, 4, True),     # slices of 2 heads inside a KV group of 4
    (4, 4, sb.SP_SCHED_ZIGZAG, 2, 4, True),   # MHA, one head per rank
    (8, 2, sb.SP_SCHED_RING, 2, 2, False),
    (16, 16, sb.SP_SCHED_TASP, 5, 8, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}x{c[1]}-k{c[2]}-R{c[3]}xU{c[4]}-c{int(c[5])}")
def test_hier_schedule_matches_oracle(case):
    Hq, Hkv, kind, R, U, causal = case
    docs = [130, 1, 269, 300, 20] if kind != sb.SP_SCHED_ZIGZAG else [130, 1, 269, 320]
    cu = wl.cu_from_lengths(docs)
    q, k, v = _inputs(int(cu[-1]), Hq, Hkv, 50 + Hq)
    att = sb.PackedAttention(cu, causal, kind, R * U, Hq, seed=2, ulysses=U)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o.float().cpu().numpy().astype(np.float64), lse.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_hier_full_size_noncausal_2x8():
    import torch
    w = wl.WORKLOADS[3]
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    att = sb.PackedAttention(cu, w.causal, sb.SP_SCHED_RING, 16, w.Hq, ulysses=8)
    assert len(att.items) == 8 * 2 * 2
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    rows = sample_rows(cu, w.T, [0, w.T // 2, w.T], n_random=24, seed=9)
    rows = rows[:32]
    o_ref, l_ref = oracle_rows(q, k, v, cu, w.causal, rows)
    rt = torch.from_numpy(rows).cuda()
    eo, el = max_errs(o[rt].float().cpu().numpy().astype(np.float64),
                      lse[:, rt].t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_one_head_slice_alone_and_straddling_range_rejected():
    import torch
    cu = wl.cu_from_lengths([300, 212])
    T, Hq, Hkv = 512, 8, 2
    q, k, v = _inputs(T, Hq, Hkv, 77)
    items, heads = sb.sp_schedule_build_hier(sb.SP_SCHED_RING, 2, 4, T, cu, True, Hq)
    sel = (items[:, 0] % 4) == 1          # heads 2..3 of every group
    it_d = torch.from_numpy(np.ascontiguousarray(items[sel])).cuda()
    hd_d = torch.from_numpy(np.ascontiguousarray(heads[sel])).cuda()
    o = torch.full_like(q, 3.0)
    lse = torch.full((Hq, T), 3.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(sb.sp_packed_attention_workspace_size(len(it_d)), dtype=torch.uint8, device="cuda")
    cu_d = torch.from_numpy(cu).cuda()
    sb.sp_packed_attention_ex(q, k, v, o, lse, cu_d, True, it_d, hd_d, ws)
    sb.sp_check_device_status()
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, True)
    eo, el = max_errs(o[:, 2:4].float().cpu().numpy().astype(np.float64),
                      lse[2:4].t().cpu().numpy().astype(np.float64), o_ref[:, 2:4], l_ref[:, 2:4])
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
    others = [0, 1, 4, 5, 6, 7]
    assert bool((o[:, others].float() == 3.0).all()) and bool((lse[others] == 3.0).all())
    # Heads 3..5 straddle the key/value groups {0..3} and {4..7}: rejected, nothing written.
    bad = hd_d.clone()
    bad[:, 0] = 3
    bad[:, 1] = 6
    o2 = torch.full_like(q, 3.0)
    sb.sp_packed_attention_ex(q, k, v, o2, lse, cu_d, True, it_d, bad, ws)
    assert sb.sp_check_device_status_code() == 6
    assert bool((o2.float() == 3.0).all())
