"""GPU parity of schedules over balanced chunks: the whole schedule in one
launch against the fp64 oracle on small packings (every row), the 128K
hybrid-packed and 512K workloads at full size on sampled rows, and one
virtual rank's items run alone (its rows equal the oracle, other rows are
left unwritten)."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, host_inputs, max_errs, oracle_rows, row_cost, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [sb.SP_CHUNK_BALANCED, sb.SP_CHUNK_BALANCED_DOC])
@pytest.mark.parametrize("kind,P", [(sb.SP_SCHED_RING, 3), (sb.SP_SCHED_TASP, 5), (sb.SP_SCHED_TASP, 7)])
@pytest.mark.parametrize("causal", [True, False])
def test_chunked_schedule_matches_oracle(mode, kind, P, causal):
    docs = [130, 1, 269, 300, 61, 700]
    cu = wl.cu_from_lengths(docs)
    T = int(cu[-1])
    q = wl.random_normal((T, 4, 128), 31, "cuda", "bf16")
    k = wl.random_normal((T, 2, 128), 32, "cuda", "bf16")
    v = wl.random_normal((T, 2, 128), 33, "cuda", "bf16")
    att = sb.PackedAttention(cu, causal, kind, P, 4, seed=3, chunking=mode)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o.float().cpu().numpy().astype(np.float64), lse.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


@pytest.mark.parametrize("idx,mode", [(2, sb.SP_CHUNK_BALANCED_DOC), (4, sb.SP_CHUNK_BALANCED)])
def test_chunked_workload_full_size(idx, mode):
    import torch
    w = wl.WORKLOADS[idx]
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed, chunking=mode)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    bounds = [int(x) for x in att.bounds]
    cand = sample_rows(cu, w.T, bounds, n_random=512, seed=w.seed + 5)
    cost = row_cost(cu, w.causal, cand)
    rows = cand[np.argsort(cost, kind="stable")][:400]  # the cheapest 400 for the fp64 oracle
    rows = np.sort(rows)
    o_ref, l_ref = oracle_rows(q, k, v, cu, w.causal, rows)
    rt = torch.from_numpy(rows).cuda()
    eo, el = max_errs(o[rt].float().cpu().numpy().astype(np.float64),
                      lse[:, rt].t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_one_virtual_rank_alone():
    """Rank r's items alone write exactly rank r's rows, equal to the oracle."""
    import torch
    docs = [300, 5, 400, 319]
    cu = wl.cu_from_lengths(docs)
    T, P, causal = int(cu[-1]), 5, True
    q = wl.random_normal((T, 2, 128), 41, "cuda", "bf16")
    k = wl.random_normal((T, 1, 128), 42, "cuda", "bf16")
    v = wl.random_normal((T, 1, 128), 43, "cuda", "bf16")
    bounds = sb.sp_chunk_bounds(sb.SP_CHUNK_BALANCED, P, T, cu, causal)
    items = sb.sp_schedule_build(sb.SP_SCHED_TASP, P, T, cu, causal, seed=1, bounds=bounds)
    r = 3
    mine = torch.from_numpy(np.ascontiguousarray(items[items[:, 0] == r])).cuda()
    o = torch.full_like(q, 7.0)
    lse = torch.full((2, T), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(sb.sp_packed_attention_workspace_size(mine.shape[0]), dtype=torch.uint8, device="cuda")
    sb.sp_packed_attention(q, k, v, o, lse, torch.from_numpy(cu).cuda(), causal, mine, ws)
    sb.sp_check_device_status()
    a, b = int(bounds[r]), int(bounds[r + 1])
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o[a:b].float().cpu().numpy().astype(np.float64),
                      lse[:, a:b].t().cpu().numpy().astype(np.float64), o_ref[a:b], l_ref[a:b])
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
    assert bool((o[:a].float() == 7.0).all()) and bool((o[b:].float() == 7.0).all())
    assert bool((lse[:, :a] == 7.0).all()) and bool((lse[:, b:] == 7.0).all())
