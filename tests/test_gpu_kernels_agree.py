"""The two bf16 forward kernels compute the same thing. A GQA problem with
d = 128 runs on CTA pairs through sp_packed_attention (every item over all
heads); the same items with explicit head ranges [0, Hq) run on the one-CTA
kernel through sp_packed_attention_ex. Both take the same MMA steps per row
and the same softmax arithmetic, so O and LSE must agree bit for bit; both
are also checked against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, host_inputs, max_errs

pytestmark = pytest.mark.gpu

CASES = [
    # docs, Hq, Hkv, kind, P, causal
    ([333, 1, 666], 8, 2, sb.SP_SCHED_TASP, 5, True),
    ([700, 1348], 4, 2, sb.SP_SCHED_ZIGZAG, 4, True),
    ([129, 900, 2], 16, 4, sb.SP_SCHED_RING, 3, False),
    ([1], 2, 1, sb.SP_SCHED_RING, 1, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{sum(c[0])}-H{c[1]}x{c[2]}-k{c[3]}P{c[4]}-c{int(c[5])}")
def test_pair_and_single_cta_kernels_agree(case):
    import torch
    docs, Hq, Hkv, kind, P, causal = case
    cu = wl.cu_from_lengths(docs)
    T = int(cu[-1])
    q = wl.random_normal((T, Hq, 128), 31, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, 128), 32, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, 128), 33, "cuda", "bf16")
    items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=1)
    it_d = torch.from_numpy(items).cuda()
    heads = np.tile(np.array([[0, Hq]], dtype=np.int32), (len(items), 1))
    hd_d = torch.from_numpy(heads).cuda()
    cu_d = torch.from_numpy(cu).cuda()
    ws = torch.empty(sb.sp_packed_attention_workspace_size(len(items)), dtype=torch.uint8, device="cuda")
    o1 = torch.empty_like(q)
    l1 = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    sb.sp_packed_attention(q, k, v, o1, l1, cu_d, causal, it_d, ws)        # CTA pairs
    o2 = torch.empty_like(q)
    l2 = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    sb.sp_packed_attention_ex(q, k, v, o2, l2, cu_d, causal, it_d, hd_d, ws)  # one CTA
    sb.sp_check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o1.float().cpu().numpy().astype(np.float64), l1.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
