"""The binding's example (sequence_blockwise_gb300/example.py) runs, and its
outputs match the fp64 oracle on sampled rows (document edges, tile edges and
random rows)."""
import numpy as np
import pytest

from gpu_util import TOL_BF16_LSE, TOL_BF16_O, max_errs, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu


def test_example_runs_and_matches_oracle():
    import torch
    from sequence_blockwise_gb300 import example
    out = example.run()
    q, k, v, o, lse, cu = (out[n] for n in ("q", "k", "v", "o", "lse", "cu"))
    dq, dk, dv = out["dq"], out["dk"], out["dv"]
    T, Hq, d = q.shape
    assert o.shape == q.shape and o.dtype == torch.bfloat16
    assert lse.shape == (Hq, T) and lse.dtype == torch.float32
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    assert all(bool(torch.isfinite(t.float()).all()) for t in (o, lse, dq, dk, dv))
    rows = sample_rows(np.asarray(cu), T, [], n_random=48, seed=1)
    o_ref, l_ref = oracle_rows(q, k, v, np.asarray(cu, dtype=np.int32), True, rows)
    rows_t = torch.from_numpy(rows).cuda()
    eo, el = max_errs(o[rows_t].float().cpu().numpy().astype(np.float64),
                      lse[:, rows_t].t().cpu().numpy().astype(np.float64), o_ref, l_ref)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
