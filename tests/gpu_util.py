"""Helpers shared by the GPU parity tests (inputs to host, comparisons)."""
import numpy as np

import oracle
from sequence_blockwise_gb300 import workloads as wl

# Tolerances: bf16 inputs (fp32 accumulate, bf16 P and O) against the fp64
# oracle on the same bf16-rounded inputs; fp32 inputs on the fp32 path.
TOL_BF16_O, TOL_BF16_LSE = 2e-2, 1e-3
TOL_FP32 = 1e-5


def host_inputs(t):
    """A torch tensor as the oracle reads it: bf16 -> uint16 bits, fp32 -> float32."""
    import torch
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits(t)
    return t.detach().cpu().numpy()


def oracle_rows(q, k, v, cu, causal, rows, scale=None, kv_range=None):
    """Oracle (O [n, Hq, d], LSE [n, Hq]) for the given query rows."""
    import torch
    rows = np.asarray(rows, dtype=np.int64)
    qr = q[torch.from_numpy(rows).to(q.device)]
    return oracle.attn(host_inputs(qr), host_inputs(k), host_inputs(v), cu, causal, scale=scale,
                       rows=rows.astype(np.int32), kv_range=kv_range, q_rows_only=True)


def max_errs(o_gpu_rows, lse_gpu_rows, o_ref, lse_ref):
    """o_gpu_rows [n, Hq, d], lse_gpu_rows [n, Hq] (float64 numpy)."""
    eo = float(np.max(np.abs(o_gpu_rows - o_ref))) if o_ref.size else 0.0
    both_inf = np.isneginf(lse_gpu_rows) & np.isneginf(lse_ref)
    a = np.where(both_inf, 0.0, lse_gpu_rows)
    b = np.where(both_inf, 0.0, lse_ref)
    diff = np.abs(a - b)
    el = float(np.max(diff)) if diff.size else 0.0
    return eo, el


def sample_rows(cu, T, bounds, n_random, seed, extra=()):
    """Rows at document and chunk edges, at 128/256-row tile edges near them,
    and n_random uniformly drawn rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in list(cu) + list(bounds):
        for dlt in (-2, -1, 0, 1, 127, 128, 255, 256):
            t = int(b) + dlt
            if 0 <= t < T:
                rows.add(t)
    rows.update(int(x) for x in extra if 0 <= x < T)
    rows.update(int(x) for x in rng.integers(0, T, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def row_cost(cu, causal, rows):
    """Valid keys per row (for sizing oracle samples)."""
    cu = np.asarray(cu)
    doc = np.searchsorted(cu, rows, side="right") - 1
    if causal:
        return rows - cu[doc] + 1
    return cu[doc + 1] - cu[doc]
