"""Device buffers at the C-ABI's minimum alignment (16 bytes).

The forward epilogue of the CTA-pair kernel writes O rows with 32-byte stores
when O is 32-byte aligned and with 16-byte stores otherwise; the other
kernels use 16-byte accesses throughout, and every TMA tensor map needs a
16-byte aligned base. Here every tensor of a call (Q, K, V, O, LSE, dO and the
gradients) is a copy placed 16 bytes past a 32-byte boundary. The arithmetic
does not depend on where a buffer starts, so each result must equal, bit for
bit, the same call on the allocator's (256-byte aligned) buffers, and match
the fp64 oracle."""
import math

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, TOL_FP32, host_inputs, max_errs

pytestmark = pytest.mark.gpu


def _at16(t):
    """A copy of t whose data starts 16 bytes past a 32-byte boundary."""
    import torch
    es = t.element_size()
    buf = torch.empty(t.numel() + 64 // es, dtype=t.dtype, device=t.device)
    off = (16 - buf.data_ptr() % 32) % 32 // es
    out = buf[off:off + t.numel()].view(t.shape)
    out.copy_(t)
    assert out.data_ptr() % 32 == 16 and out.is_contiguous()
    return out


CASES = [
    # T, docs, Hq, Hkv, d, causal, kind, P, dtype   (kernel)
    (700, [130, 1, 269, 300], 4, 2, 128, True, sb.SP_SCHED_TASP, 5, "bf16"),   # CTA pairs
    (704, [704], 2, 2, 128, True, sb.SP_SCHED_ZIGZAG, 4, "bf16"),             # one CTA, MHA
    (640, [333, 307], 4, 1, 64, False, sb.SP_SCHED_RING, 3, "bf16"),           # one CTA, d 64
    (256, [100, 156], 1, 1, 64, True, sb.SP_SCHED_RING, 4, "fp32"),            # fp32 path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}-H{c[2]}x{c[3]}-d{c[4]}-{c[8]}")
def test_packed_attention_on_16_byte_aligned_buffers(case):
    import torch
    T, docs, Hq, Hkv, d, causal, kind, P, dtype = case
    cu = wl.cu_from_lengths(docs)
    q = wl.random_normal((T, Hq, d), 21, "cuda", dtype)
    k = wl.random_normal((T, Hkv, d), 22, "cuda", dtype)
    v = wl.random_normal((T, Hkv, d), 23, "cuda", dtype)
    att = sb.PackedAttention(cu, causal, kind, P, Hq, seed=1)
    o1, l1 = att(q, k, v)
    q2, k2, v2 = _at16(q), _at16(k), _at16(v)
    o2, l2 = _at16(torch.zeros_like(o1)), _at16(torch.zeros_like(l1))
    att(q2, k2, v2, o2, l2)
    sb.sp_check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o2.float().cpu().numpy().astype(np.float64), l2.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    tol_o, tol_l = (TOL_FP32, TOL_FP32) if dtype == "fp32" else (TOL_BF16_O, TOL_BF16_LSE)
    assert eo <= tol_o and el <= tol_l, (eo, el)


def test_partial_step_and_merge_on_16_byte_aligned_buffers():
    """fp32 partials (the pair kernel's fp32-output epilogue for this GQA
    d = 128 layer) and the merge kernel."""
    import torch
    T, Hq, Hkv, d = 600, 4, 2, 128
    cu = wl.cu_from_lengths([250, 7, 343])
    q = wl.random_normal((T, Hq, d), 31, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, d), 32, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, d), 33, "cuda", "bf16")
    cu_dev = torch.from_numpy(cu).cuda()
    steps = [(0, 600, 0, 300), (0, 600, 300, 600)]
    results = []
    for place in (lambda t: t, _at16):
        qq, kk, vv = place(q), place(k), place(v)
        o_acc = place(torch.zeros((T, Hq, d), dtype=torch.float32, device="cuda"))
        l_acc = place(torch.full((Hq, T), -math.inf, dtype=torch.float32, device="cuda"))
        for (qa, qb, ka, kb) in steps:
            op = place(torch.empty((qb - qa, Hq, d), dtype=torch.float32, device="cuda"))
            lp = place(torch.empty((Hq, qb - qa), dtype=torch.float32, device="cuda"))
            sb.sp_partial_attn(qq, kk, vv, op, lp, qa, qb, ka, kb, cu_dev, True)
            sb.sp_lse_merge(o_acc, l_acc, op, lp)
        sb.sp_check_device_status()
        results.append((o_acc.clone(), l_acc.clone()))
    assert torch.equal(results[0][0], results[1][0]) and torch.equal(results[0][1], results[1][1])
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, True)
    eo, el = max_errs(results[1][0].cpu().numpy().astype(np.float64),
                      results[1][1].t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 128), (2, 2, 64)])
def test_backward_on_16_byte_aligned_buffers(Hq, Hkv, d):
    import torch
    T = 500
    cu = wl.cu_from_lengths([200, 300])
    q = wl.random_normal((T, Hq, d), 41, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, d), 42, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, d), 43, "cuda", "bf16")
    do = wl.random_normal((T, Hq, d), 44, "cuda", "bf16")
    att = sb.PackedAttention(cu, True, sb.SP_SCHED_RING, 2, Hq)
    o, lse = att(q, k, v)
    g1 = att.backward(q, k, v, o, lse, do)
    dq2, dk2, dv2 = (_at16(torch.zeros_like(t)) for t in (q, k, v))
    att.backward(_at16(q), _at16(k), _at16(v), _at16(o), _at16(lse), _at16(do), dq2, dk2, dv2)
    sb.sp_check_device_status()
    for a, b in zip(g1, (dq2, dk2, dv2)):
        assert torch.equal(a, b)
