"""The library's schedules against the oracle's independent re-derivation:
RING / ZIGZAG element for element, TASP by its defining properties, every kind
by exact-once coverage of the valid (query, key) pairs (brute force on small
inputs, interval bookkeeping at full size)."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl


def _doc_flags(items, cu, causal):
    out = []
    for it in items:
        qa, qb, ka, kb = int(it[3]), int(it[4]), int(it[5]), int(it[6])
        f = 0
        if causal and kb - 1 > qa:
            f |= 1
        if oracle.doc_of(cu, min(qa, ka)) != oracle.doc_of(cu, max(qb, kb) - 1):
            f |= 2
        out.append(f)
    return np.array(out, dtype=np.int32)


def _rand_cu(rng, T, max_docs):
    nd = min(int(rng.integers(1, max_docs + 1)), T)
    cuts = np.sort(rng.choice(np.arange(1, T), size=nd - 1, replace=False)) if nd > 1 else []
    return np.concatenate([[0], cuts, [T]]).astype(np.int32)


@pytest.mark.parametrize("seed", range(12))
def test_random_small_all_kinds_brute(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 3, 5, 7, 8]))
    T = 2 * P * int(rng.integers(1, 40))
    cu = _rand_cu(rng, T, 6)
    for causal in (True, False):
        for kind in (0, 1, 2):
            items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=seed)
            succ = sb.sp_tasp_cycles(P, seed) if kind == 2 else None
            rc, msg = oracle.check_schedule(kind, P, T, cu, causal, items, succ, brute=True)
            assert rc == 0, (kind, P, T, msg)
            if kind < 2:
                exp = oracle.closed_form_schedule(kind, P, T, cu, causal)
                assert np.array_equal(items[:, :7], exp[:, :7]), (kind, P)
            assert np.array_equal(items[:, 7], _doc_flags(items, cu, causal))


@pytest.mark.parametrize("P", [2, 3, 5, 7, 8, 9, 10, 12, 15, 16, 24, 31, 32, 33, 48, 64])
def test_tasp_cycles_are_a_hamiltonian_decomposition(P):
    for seed in (0, 1, 12345):
        succ = sb.sp_tasp_cycles(P, seed)
        assert succ.shape == (P - 1, P)
        assert oracle.check_hamiltonian(P, succ) == 0
    assert np.array_equal(sb.sp_tasp_cycles(P, 7), sb.sp_tasp_cycles(P, 7))


def test_tasp_unsupported_sizes():
    for P in (4, 6, 65):
        with pytest.raises(sb.SpError):
            sb.sp_tasp_cycles(P, 0)


def test_golden_ring_schedule():
    items = sb.sp_schedule_build(0, 4, 256, [0, 100, 256], True)
    gold = []
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "ring_P4_T256_docs100_156_causal.txt")
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            gold.append([int(x) for x in line.split()])
    assert np.array_equal(items[:, :7], np.array(gold, dtype=np.int32))


@pytest.mark.parametrize("w", wl.WORKLOADS, ids=lambda w: w.name)
def test_workload_schedules(w):
    cu = wl.cu_seqlens(w)
    items = sb.sp_schedule_build(w.kind, w.P, w.T, cu, w.causal, seed=w.seed)
    succ = sb.sp_tasp_cycles(w.P, w.seed) if w.kind == 2 else None
    rc, msg = oracle.check_schedule(w.kind, w.P, w.T, cu, w.causal, items, succ, brute=w.T <= 4096)
    assert rc == 0, msg
    if w.kind < 2:
        exp = oracle.closed_form_schedule(w.kind, w.P, w.T, cu, w.causal)
        assert np.array_equal(items[:, :7], exp[:, :7])
    # Chunk pairs with work: c1 ring 8 of 16, c2 zigzag 136 of 256, c4 ring all 256.
    expected = {0: 8, 1: 136, 3: 256}
    idx = wl.WORKLOADS.index(w)
    if idx in expected:
        assert len(items) == expected[idx]
    # Items of a rank and Q range are contiguous.
    keys = [(int(r[0]), int(r[3]), int(r[4])) for r in items]
    seen = set()
    for i, key in enumerate(keys):
        if i == 0 or key != keys[i - 1]:
            assert key not in seen
            seen.add(key)
