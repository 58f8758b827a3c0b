"""GQA with an odd group size above 1 (three query heads per key/value head).
Such layers run on the one-CTA forward kernel (the CTA-pair kernel takes two
query heads of one key/value head per cluster, so it needs an even group);
the forward and the backward are checked against the fp64 oracle."""
import math

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import TOL_BF16_LSE, TOL_BF16_O, host_inputs, max_errs
from test_gpu_backward import REL_FRO, _envelopes, _rel_fro

pytestmark = pytest.mark.gpu


def _inputs(T, Hq, Hkv, d, seed):
    return (wl.random_normal((T, Hq, d), seed, "cuda", "bf16"), wl.random_normal((T, Hkv, d), seed + 1, "cuda", "bf16"),
            wl.random_normal((T, Hkv, d), seed + 2, "cuda", "bf16"), wl.random_normal((T, Hq, d), seed + 3, "cuda", "bf16"))


@pytest.mark.parametrize("case", [
    (600, [250, 350], 6, 2, 128, True, sb.SP_SCHED_TASP, 5),
    (500, [500], 3, 1, 64, False, sb.SP_SCHED_RING, 2),
], ids=lambda c: f"T{c[0]}-H{c[2]}x{c[3]}-d{c[4]}-c{int(c[5])}")
def test_forward_odd_group(case):
    T, docs, Hq, Hkv, d, causal, kind, P = case
    cu = wl.cu_from_lengths(docs)
    q, k, v, _ = _inputs(T, Hq, Hkv, d, 70 + T)
    o, lse = sb.PackedAttention(cu, causal, kind, P, Hq, seed=1)(q, k, v)
    sb.sp_check_device_status()
    o_ref, l_ref = oracle.attn(host_inputs(q), host_inputs(k), host_inputs(v), cu, causal)
    eo, el = max_errs(o.float().cpu().numpy().astype(np.float64), lse.t().cpu().numpy().astype(np.float64),
                      o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)


def test_backward_odd_group():
    T, docs, Hq, Hkv, d = 400, [150, 250], 6, 2, 128
    cu = wl.cu_from_lengths(docs)
    q, k, v, do = _inputs(T, Hq, Hkv, d, 90)
    att = sb.PackedAttention(cu, True, sb.SP_SCHED_RING, 3, Hq)
    o, lse = att(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, do)
    sb.sp_check_device_status()
    ref = oracle.attn_backward(host_inputs(q), host_inputs(k), host_inputs(v), host_inputs(do), cu, True)
    env = _envelopes(q, k, v, do, cu, True, 1.0 / math.sqrt(d))
    for name, got, r, mm in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, env):
        g = got.double().cpu().numpy()
        err = np.abs(g - r)
        assert float(np.max(err / (2.0 ** -7 * mm + 2.0 ** -8 * np.abs(r) + 1e-6))) <= 1.0, name
        assert _rel_fro(g, r) <= REL_FRO, name
