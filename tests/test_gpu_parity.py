"""GPU parity of the CUDA path (through the C-ABI) against the fp64 oracle on
sizes the oracle finishes in seconds, spanning several 128-row / 128-key tiles
with ragged tails, every schedule kind, causal and not, GQA and MHA, d 64 and
128, plus the edge cases: one-token documents, empty items, rows without keys."""
import math

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, TOL_FP32, host_inputs, max_errs

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _inputs(T, Hq, Hkv, d, dtype, seed):
    torch = _torch()
    q = wl.random_normal((T, Hq, d), seed, "cuda", dtype)
    k = wl.random_normal((T, Hkv, d), seed + 1, "cuda", dtype)
    v = wl.random_normal((T, Hkv, d), seed + 2, "cuda", dtype)
    return q, k, v


def _run_packed(q, k, v, cu, causal, kind, P, seed=0):
    att = sb.PackedAttention(cu, causal, kind, P, q.shape[1], seed=seed)
    o, lse = att(q, k, v)
    sb.sp_check_device_status()
    return o, lse, att


def _full_oracle(q, k, v, cu, causal):
    return oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)


CASES = [
    # T, docs, Hq, Hkv, d, causal, kind, P
    (700, [130, 1, 269, 300], 4, 2, 128, True, 2, 5),
    (700, [130, 1, 269, 300], 4, 2, 128, False, 0, 3),
    (704, [704], 2, 2, 128, True, 1, 4),
    (1000, [1, 1, 500, 498], 8, 2, 128, True, 2, 8),
    (640, [333, 307], 4, 4, 64, True, 0, 2),
    (640, [333, 307], 4, 1, 64, False, 2, 3),
    (129, [129], 1, 1, 128, True, 0, 1),
    (1, [1], 2, 1, 128, True, 0, 1),
    (1537, [900, 637], 4, 2, 128, True, 2, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}-H{c[2]}x{c[3]}-d{c[4]}-c{int(c[5])}-k{c[6]}P{c[7]}")
def test_packed_bf16_matches_oracle(case):
    torch = _torch()
    T, docs, Hq, Hkv, d, causal, kind, P = case
    cu = wl.cu_from_lengths(docs)
    q, k, v = _inputs(T, Hq, Hkv, d, "bf16", 11 + T)
    o, lse, _ = _run_packed(q, k, v, cu, causal, kind, P)
    o_ref, l_ref = _full_oracle(q, k, v, cu, causal)
    eo, el = max_errs(o.float().cpu().numpy().astype(np.float64),
                      lse.t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


@pytest.mark.parametrize("d", [64, 128])
def test_packed_fp32_tiny_workload(d):
    w = wl.WORKLOADS[0]
    cu = wl.cu_seqlens(w)
    torch = _torch()
    q, k, v = wl.make_qkv(w, "cuda")
    if d != w.d:
        q, k, v = _inputs(w.T, w.Hq, w.Hkv, d, "fp32", 5)
    o, lse, _ = _run_packed(q, k, v, cu, w.causal, w.kind, w.P)
    o_ref, l_ref = _full_oracle(q, k, v, cu, w.causal)
    eo, el = max_errs(o.cpu().numpy().astype(np.float64), lse.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    assert eo <= TOL_FP32 and el <= TOL_FP32, (eo, el)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_partial_steps_and_merge_match_oracle(dtype):
    """The API path: one sp_partial_attn per schedule item, folded with
    sp_lse_merge, equals both the oracle and the fused launch."""
    torch = _torch()
    T, Hq, Hkv, d, P = 600, 4, 2, 128, 3
    cu = wl.cu_from_lengths([250, 7, 343])
    causal = True
    q, k, v = _inputs(T, Hq, Hkv, d, dtype, 77)
    items = sb.sp_schedule_build(sb.SP_SCHED_TASP, P, T, cu, causal, seed=3)
    cu_dev = torch.from_numpy(cu).cuda()
    o_full = torch.zeros((T, Hq, d), dtype=torch.float32, device="cuda")
    l_full = torch.full((Hq, T), -math.inf, dtype=torch.float32, device="cuda")
    for it in items:
        _, _, _, qa, qb, ka, kb, _ = (int(x) for x in it)
        rows = qb - qa
        op = torch.empty((rows, Hq, d), dtype=torch.float32, device="cuda")
        lp = torch.empty((Hq, rows), dtype=torch.float32, device="cuda")
        sb.sp_partial_attn(q, k, v, op, lp, qa, qb, ka, kb, cu_dev, causal)
        # partial against the oracle restricted to the item's keys
        ro, rl = oracle.attn(host_inputs(q[qa:qb]), host_inputs(k), host_inputs(v), cu, causal,
                             rows=np.arange(qa, qb), kv_range=(ka, kb), q_rows_only=True)
        eo, el = max_errs(op.cpu().numpy().astype(np.float64), lp.t().cpu().numpy().astype(np.float64),
                          ro, rl)
        tol_o, tol_l = (TOL_BF16_O, TOL_BF16_LSE) if dtype == "bf16" else (TOL_FP32, TOL_FP32)
        assert eo <= tol_o and el <= tol_l, (it, eo, el)
        # rows without any valid key are exactly (-inf, 0)
        assert np.array_equal(np.isneginf(lp.t().cpu().numpy()), np.isneginf(rl))
        acc_o = o_full[qa:qb].contiguous()
        acc_l = l_full[:, qa:qb].contiguous()
        sb.sp_lse_merge(acc_o, acc_l, op, lp)
        o_full[qa:qb] = acc_o
        l_full[:, qa:qb] = acc_l
    sb.sp_check_device_status()
    o_ref, l_ref = _full_oracle(q, k, v, cu, causal)
    eo, el = max_errs(o_full.cpu().numpy().astype(np.float64), l_full.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    tol_o, tol_l = (TOL_BF16_O, TOL_BF16_LSE) if dtype == "bf16" else (TOL_FP32, TOL_FP32)
    assert eo <= tol_o and el <= tol_l, (eo, el)


def test_partial_ragged_ranges_and_empty_rows():
    torch = _torch()
    T, Hq, Hkv, d = 900, 2, 1, 128
    cu = wl.cu_from_lengths([300, 600])
    q, k, v = _inputs(T, Hq, Hkv, d, "bf16", 5)
    cu_dev = torch.from_numpy(cu).cuda()
    for (qa, qb, ka, kb, causal) in [(17, 530, 3, 811, True), (0, 900, 450, 451, False),
                                     (250, 420, 500, 900, True), (1, 2, 0, 900, False),
                                     (600, 900, 0, 0, True)]:
        rows = qb - qa
        op = torch.empty((rows, Hq, d), dtype=torch.float32, device="cuda")
        lp = torch.empty((Hq, rows), dtype=torch.float32, device="cuda")
        sb.sp_partial_attn(q, k, v, op, lp, qa, qb, ka, kb, cu_dev, causal)
        ro, rl = oracle.attn(host_inputs(q[qa:qb]), host_inputs(k), host_inputs(v), cu, causal,
                             rows=np.arange(qa, qb), kv_range=(ka, kb), q_rows_only=True)
        got_l = lp.t().cpu().numpy().astype(np.float64)
        eo, el = max_errs(op.cpu().numpy().astype(np.float64), got_l, ro, rl)
        assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (qa, qb, ka, kb, eo, el)
        assert np.array_equal(np.isneginf(got_l), np.isneginf(rl))
        assert np.all(op.cpu().numpy()[np.isneginf(rl)] == 0)
    sb.sp_check_device_status()


def test_lse_merge_kernel_matches_oracle():
    torch = _torch()
    rng = np.random.default_rng(0)
    rows, Hq, d = 1000, 3, 128
    o1 = rng.standard_normal((rows, Hq, d)).astype(np.float32)
    o2 = rng.standard_normal((rows, Hq, d)).astype(np.float32)
    l1 = (rng.standard_normal((Hq, rows)) * 5).astype(np.float32)
    l2 = (rng.standard_normal((Hq, rows)) * 5).astype(np.float32)
    l1[0, :10] = -np.inf
    l2[1, 5:20] = -np.inf
    l1[2, 30:40] = -np.inf
    l2[2, 30:40] = -np.inf
    o1[:, :, :][np.isneginf(l1.T)] = 0
    o2[:, :, :][np.isneginf(l2.T)] = 0
    ta, tl = torch.from_numpy(o1).cuda(), torch.from_numpy(l1).cuda()
    sb.sp_lse_merge(ta, tl, torch.from_numpy(o2).cuda(), torch.from_numpy(l2).cuda())
    ro, rl = oracle.lse_merge(o1.astype(np.float64), l1.T.astype(np.float64), o2.astype(np.float64),
                              l2.T.astype(np.float64))
    eo, el = max_errs(ta.cpu().numpy().astype(np.float64), tl.t().cpu().numpy().astype(np.float64),
                      ro, rl)
    assert eo <= 1e-5 and el <= 1e-5
    assert np.all(np.isneginf(tl.cpu().numpy()[2, 30:40]))


def test_document_isolation_bit_exact():
    torch = _torch()
    T, Hq, Hkv, d = 1100, 4, 2, 128
    docs = [300, 129, 671]
    cu = wl.cu_from_lengths(docs)
    q, k, v = _inputs(T, Hq, Hkv, d, "bf16", 9)
    o1, l1, att = _run_packed(q, k, v, cu, True, sb.SP_SCHED_TASP, 5)
    a, b = 300, 429
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    g = torch.Generator(device="cuda").manual_seed(1)
    q2[a:b] = torch.randn(q2[a:b].shape, generator=g, device="cuda").to(q.dtype) * 3
    k2[a:b] = -k2[a:b]
    v2[a:b] = v2[a:b] + 5
    o2, l2 = att(q2, k2, v2)
    sb.sp_check_device_status()
    keep = torch.ones(T, dtype=torch.bool, device="cuda")
    keep[a:b] = False
    assert torch.equal(o1[keep], o2[keep]) and torch.equal(l1[:, keep], l2[:, keep])
    assert not torch.equal(o1[a:b], o2[a:b])


def test_deterministic_and_schedule_invariant():
    torch = _torch()
    T, Hq, Hkv, d = 2048, 4, 2, 128
    cu = wl.cu_from_lengths([700, 1348])
    q, k, v = _inputs(T, Hq, Hkv, d, "bf16", 21)
    o1, l1, att = _run_packed(q, k, v, cu, True, sb.SP_SCHED_ZIGZAG, 4)
    o2, l2 = att(q, k, v)
    sb.sp_check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # Any schedule visits every valid pair once: results agree within the
    # rounding of the merge order.
    for kind, P in ((sb.SP_SCHED_RING, 8), (sb.SP_SCHED_TASP, 8), (sb.SP_SCHED_RING, 1)):
        o3, l3, _ = _run_packed(q, k, v, cu, True, kind, P)
        assert float((o3.float() - o1.float()).abs().max()) <= 2 * TOL_BF16_O
        assert float((l3 - l1).abs().max()) <= 2 * TOL_BF16_LSE


def test_bounded_wait_gives_up_and_reports():
    sb.sp_check_device_status()  # clear
    sb.sp_selftest_bounded_wait(2_000_000)  # 2 ms
    assert sb.sp_check_device_status_code() == 5  # SP_ERR_TIMEOUT
    assert sb.sp_check_device_status_code() == 0  # cleared, context still usable
    torch = _torch()
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_inconsistent_items_reported_not_hung():
    torch = _torch()
    T, Hq, Hkv, d = 512, 2, 2, 128
    q, k, v = _inputs(T, Hq, Hkv, d, "bf16", 3)
    cu = np.array([0, T], dtype=np.int32)
    # Two groups whose Q ranges overlap: rejected by the set-up kernel.
    items = np.array([[0, 0, 0, 0, 300, 0, 300, 0], [1, 0, 0, 200, 512, 0, 512, 0]], dtype=np.int32)
    items_dev = torch.from_numpy(items).cuda()
    ws = torch.empty(sb.sp_packed_attention_workspace_size(2), dtype=torch.uint8, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((Hq, T), dtype=torch.float32, device="cuda")
    sb.sp_packed_attention(q, k, v, o, lse, torch.from_numpy(cu).cuda(), True, items_dev, ws)
    assert sb.sp_check_device_status_code() == 6  # SP_ERR_INTERNAL
    assert float(o.float().abs().sum()) == 0.0
    assert sb.sp_check_device_status_code() == 0
