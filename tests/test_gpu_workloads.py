"""The five workloads at full size, in the launch configuration the benchmark
times (one sp_packed_attention over the whole schedule), against the fp64
oracle on sampled rows (document, chunk and tile edges plus random rows, all
heads), and against properties that hold at any size."""
import numpy as np
import pytest

import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import (TOL_BF16_LSE, TOL_BF16_O, TOL_FP32, max_errs, oracle_rows, row_cost,
                      sample_rows)

pytestmark = pytest.mark.gpu

# Oracle budget per workload, in valid keys x heads x d (about 4 flop each).
BUDGET = 2.0e10


def _chunk_bounds(w):
    if w.kind == sb.SP_SCHED_ZIGZAG:
        c = w.T // (2 * w.P)
        return [i * c for i in range(2 * w.P + 1)]
    base, extra = divmod(w.T, w.P)
    out, s = [0], 0
    for r in range(w.P):
        s += base + (1 if r < extra else 0)
        out.append(s)
    return out


def _pick_rows(w, cu):
    cand = sample_rows(cu, w.T, _chunk_bounds(w), n_random=4096, seed=w.seed)
    cost = row_cost(cu, w.causal, cand).astype(np.float64) * w.Hq * w.d
    rng = np.random.default_rng(w.seed + 7)
    order = np.argsort(cost, kind="stable")
    cheap = order[cost[order] <= 4096 * w.Hq * w.d]
    rest = rng.permutation(order[cost[order] > 4096 * w.Hq * w.d])
    chosen, total = list(cheap[:512]), float(cost[cheap[:512]].sum())
    for i in rest:
        if total + cost[i] > BUDGET:
            continue
        chosen.append(i)
        total += cost[i]
    return np.array(sorted(cand[chosen]), dtype=np.int64)


@pytest.mark.parametrize("w", wl.WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(w):
    import torch
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()

    # Every row attends at least itself: all LSE finite, O finite.
    assert bool(torch.isfinite(lse).all())
    assert bool(torch.isfinite(o.float()).all()) if w.T <= 65536 else True

    # First token of every document attends only itself: O is that token's V
    # exactly (weight 1), for every head.
    G = w.Hq // w.Hkv
    firsts = torch.from_numpy(cu[:-1].astype(np.int64)).cuda()
    if w.causal:
        vo = v[firsts].repeat_interleave(G, dim=1)
        assert torch.equal(o[firsts].float(), vo.float())

    rows = _pick_rows(w, cu)
    o_ref, l_ref = oracle_rows(q, k, v, cu, w.causal, rows)
    rows_t = torch.from_numpy(rows).cuda()
    got_o = o[rows_t].float().cpu().numpy().astype(np.float64)
    got_l = lse[:, rows_t].t().cpu().numpy().astype(np.float64)
    eo, el = max_errs(got_o, got_l, o_ref, l_ref)
    tol_o, tol_l = (TOL_FP32, TOL_FP32) if w.dtype == "fp32" else (TOL_BF16_O, TOL_BF16_LSE)
    print(f"{w.name}: {len(rows)} rows x {w.Hq} heads, max|dO|={eo:.3e} max|dLSE|={el:.3e}")
    assert eo <= tol_o and el <= tol_l, (eo, el)


def test_hybrid_packing_schedule_invariance_full_size():
    """TASP, RING and ZIGZAG schedules of the 128K hybrid-packed workload give
    the same attention at every row (each visits every valid pair once)."""
    import torch
    w = wl.WORKLOADS[2]
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    o1, l1 = sb.PackedAttention(cu, True, sb.SP_SCHED_TASP, w.P, w.Hq, seed=w.seed)(q, k, v)
    o2, l2 = sb.PackedAttention(cu, True, sb.SP_SCHED_RING, w.P, w.Hq)(q, k, v)
    o3, l3 = sb.PackedAttention(cu, True, sb.SP_SCHED_ZIGZAG, w.P, w.Hq)(q, k, v)
    sb.sp_check_device_status()
    for o, l in ((o2, l2), (o3, l3)):
        assert float((o.float() - o1.float()).abs().max()) <= 2 * TOL_BF16_O
        assert float((l - l1).abs().max()) <= 2 * TOL_BF16_LSE
