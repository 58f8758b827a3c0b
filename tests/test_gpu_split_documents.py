"""GPU parity of schedules cut at document boundaries
(sp_schedule_split_documents): every document of a rank's chunk runs as a
group of its own. Small packings against the fp64 oracle on every row, for the
CTA-pair kernel (two query heads per key/value head), the one-CTA kernel (one
query head per key/value head) and head-split schedules; the per-rank launches
of a cut schedule against its whole launch, bit for bit; and, at full size, the
512K-token packing over 32 balanced ranks on rows at the tail of its longest
documents (the longest walks) and at document edges."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, host_inputs, max_errs, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

DOCS = [2100, 1, 37, 640, 3000, 255, 1200]  # a long document, tiny ones, 128-ragged lengths


def _inputs(T, Hq, Hkv, seed):
    q = wl.random_normal((T, Hq, 128), seed, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, 128), seed + 1, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, 128), seed + 2, "cuda", "bf16")
    return q, k, v


def _run(q, k, v, cu, causal, items, heads=None):
    import torch
    T, Hq = q.shape[0], q.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(sb.sp_packed_attention_workspace_size(len(items)), dtype=torch.uint8, device="cuda")
    it = torch.from_numpy(np.ascontiguousarray(items)).cuda()
    cu_dev = torch.from_numpy(cu).cuda()
    if heads is None:
        sb.sp_packed_attention(q, k, v, o, lse, cu_dev, causal, it, ws)
    else:
        hd = torch.from_numpy(np.ascontiguousarray(heads)).cuda()
        sb.sp_packed_attention_ex(q, k, v, o, lse, cu_dev, causal, it, hd, ws)
    sb.sp_check_device_status()
    return o, lse


def _vs_oracle(q, k, v, cu, causal, o, lse):
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    return max_errs(o.float().cpu().numpy().astype(np.float64), lse.t().cpu().numpy().astype(np.float64),
                    o_ref, l_ref)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (2, 2)], ids=["pair-kernel", "one-cta"])
@pytest.mark.parametrize("kind,P,chunking", [(sb.SP_SCHED_TASP, 5, sb.SP_CHUNK_BALANCED),
                                             (sb.SP_SCHED_RING, 3, sb.SP_CHUNK_EQUAL),
                                             (sb.SP_SCHED_TASP, 8, sb.SP_CHUNK_EQUAL)],
                         ids=["tasp5-balanced", "ring3", "tasp8"])
@pytest.mark.parametrize("causal", [True, False])
def test_cut_schedule_matches_oracle(Hq, Hkv, kind, P, chunking, causal):
    cu = wl.cu_from_lengths(DOCS)
    T = int(cu[-1])
    q, k, v = _inputs(T, Hq, Hkv, 60 + P)
    bounds = None if chunking == sb.SP_CHUNK_EQUAL else sb.sp_chunk_bounds(chunking, P, T, cu, causal)
    items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=4, bounds=bounds)
    cut = sb.sp_schedule_split_documents(items, cu, causal)
    assert len(cut) > len(items)  # some chunk spans several documents
    o, lse = _run(q, k, v, cu, causal, cut)
    eo, el = _vs_oracle(q, k, v, cu, causal, o, lse)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_cut_head_split_schedule_matches_oracle():
    cu = wl.cu_from_lengths(DOCS)
    T, Hq, Hkv = int(cu[-1]), 8, 2
    q, k, v = _inputs(T, Hq, Hkv, 71)
    items, heads = sb.sp_schedule_build_hier(sb.SP_SCHED_RING, 2, 2, T, cu, True, Hq)
    cut, cheads = sb.sp_schedule_split_documents(items, cu, True, heads=heads)
    o, lse = _run(q, k, v, cu, True, cut, cheads)
    eo, el = _vs_oracle(q, k, v, cu, True, o, lse)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_cut_rank_launches_reproduce_the_whole_launch():
    """Each virtual rank's pieces in a launch of their own write that rank's
    rows exactly as the whole cut schedule's launch does (the groups of one
    launch do not interact), and leave every other row untouched."""
    import torch
    cu = wl.cu_from_lengths(DOCS)
    T, Hq, Hkv, P = int(cu[-1]), 4, 2, 5
    q, k, v = _inputs(T, Hq, Hkv, 81)
    bounds = sb.sp_chunk_bounds(sb.SP_CHUNK_BALANCED, P, T, cu, True)
    cut = sb.sp_schedule_split_documents(sb.sp_schedule_build(sb.SP_SCHED_TASP, P, T, cu, True, seed=2,
                                                              bounds=bounds), cu, True)
    o_all, l_all = _run(q, k, v, cu, True, cut)
    cu_dev = torch.from_numpy(cu).cuda()
    o = torch.full_like(q, 3.0)
    lse = torch.full((Hq, T), 3.0, dtype=torch.float32, device="cuda")
    for r in range(P):
        mine = np.ascontiguousarray(cut[cut[:, 0] == r])
        ws = torch.empty(sb.sp_packed_attention_workspace_size(len(mine)), dtype=torch.uint8, device="cuda")
        sb.sp_packed_attention(q, k, v, o, lse, cu_dev, True, torch.from_numpy(mine).cuda(), ws)
        sb.sp_check_device_status()
        a, b = int(bounds[r]), int(bounds[r + 1])
        assert torch.equal(o[a:b], o_all[a:b]) and torch.equal(lse[:, a:b], l_all[:, a:b]), r
        assert bool((o[b:].float() == 3.0).all()), r


def test_cut_512k_balanced_full_size_long_walks():
    import torch
    w = wl.WORKLOADS[4]
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed, chunking=sb.SP_CHUNK_BALANCED)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    lens = np.diff(cu)
    longest = np.argsort(lens)[::-1][:2]
    tails = [int(cu[d + 1]) - 1 for d in longest] + [int(cu[d + 1]) - 129 for d in longest]
    edges = sample_rows(cu, w.T, [int(x) for x in att.bounds], n_random=0, seed=1)
    cheap = [int(r) for r in edges if r - int(cu[np.searchsorted(cu, r, side="right") - 1]) < 300]
    rows = np.unique(np.array(tails + cheap[:60], dtype=np.int64))
    o_ref, l_ref = oracle_rows(q, k, v, cu, w.causal, rows)
    rt = torch.from_numpy(rows).cuda()
    eo, el = max_errs(o[rt].float().cpu().numpy().astype(np.float64),
                      lse[:, rt].t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


@pytest.mark.parametrize("ndocs,kind,P,causal", [(2000, sb.SP_SCHED_TASP, 5, True),
                                                 (2000, sb.SP_SCHED_RING, 4, False),
                                                 (9000, sb.SP_SCHED_RING, 2, True)],
                         ids=["2000docs-tasp5", "2000docs-ring4-full", "9000docs-ring2-uncut"])
def test_many_short_documents(ndocs, kind, P, causal):
    """Thousands of 1-20-token documents, every row against the oracle: cut at
    documents (2,000) and, above the group limit, as built (9,000)."""
    rng = np.random.default_rng(ndocs + P)
    lens = rng.integers(1, 21, size=ndocs)
    cu = wl.cu_from_lengths(lens.tolist())
    T, Hq, Hkv = int(cu[-1]), 4, 2
    q, k, v = _inputs(T, Hq, Hkv, 90 + P)
    att = sb.PackedAttention(cu, causal, kind, P, Hq, seed=1)
    assert att.documents_cut == (ndocs == 2000)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    eo, el = _vs_oracle(q, k, v, cu, causal, o, lse)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
