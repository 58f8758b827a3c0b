"""The communication model of the schedules (bytes per link per AllGather
iteration) against the oracle's receiver-side restatement, closed forms and a
hand-derived sequence-aware case."""
import os

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand_derived_ring_needed_only():
    exp = np.zeros((3, 4, 4), dtype=np.int64)
    for line in open(os.path.join(GOLDEN, "ring_P4_T256_causal_needed_link_bytes.txt")):
        if line.strip() and not line.startswith("#"):
            t, u, v, b = (int(x) for x in line.split())
            exp[t - 1, u, v] = b
    return exp


def test_hand_derived_ring_needed_only():
    got = sb.sp_schedule_link_bytes(sb.SP_SCHED_RING, 4, 256, [0, 256], True, needed_only=True)
    assert np.array_equal(got, _hand_derived_ring_needed_only())


def test_oracle_hand_derived_ring_needed_only():
    got = oracle.link_bytes(0, 4, 256, [0, 256], True, needed_only=True)
    assert np.array_equal(got, _hand_derived_ring_needed_only())


def _full_allgather_closed_forms(ring, tasp, P, T):
    # Every token is delivered to the P-1 other ranks: same total for both.
    assert ring.sum() == tasp.sum() == 4 * T * (P - 1)
    # Ring: each iteration uses exactly the P ring links; TASP: all P(P-1) links.
    for t in range(P - 1):
        assert np.count_nonzero(ring[t]) == P
        assert all(ring[t, r, (r + 1) % P] > 0 for r in range(P))
        assert np.count_nonzero(tasp[t]) == P * (P - 1)
        assert np.all(np.diag(tasp[t]) == 0)
    # Busiest link per iteration: a chunk for Ring, one piece (chunk/(P-1)) for TASP.
    chunk = -(-T // P)
    piece = -(-chunk // (P - 1))
    assert ring.max() == 4 * chunk and tasp.max() == 4 * piece


@pytest.mark.parametrize("P", [2, 3, 5, 7, 8, 16])
def test_closed_forms_full_allgather(P):
    T = P * (P - 1) * 12 + 5 * P  # chunks and pieces not all equal
    cu = [0, T]
    ring = sb.sp_schedule_link_bytes(sb.SP_SCHED_RING, P, T, cu, False, bytes_per_token=4)
    tasp = sb.sp_schedule_link_bytes(sb.SP_SCHED_TASP, P, T, cu, False, bytes_per_token=4)
    _full_allgather_closed_forms(ring, tasp, P, T)


@pytest.mark.parametrize("P", [2, 3, 5, 7])
def test_oracle_closed_forms_full_allgather(P):
    """The same closed forms for the oracle's model, with the decomposition
    u -> u + s (s = 1 .. P-1) into Hamiltonian cycles for prime P."""
    T = P * (P - 1) * 12 + 5 * P
    cu = [0, T]
    succ = np.array([[(u + s) % P for u in range(P)] for s in range(1, P)], dtype=np.int32)
    ring = oracle.link_bytes(0, P, T, cu, False, bytes_per_token=4)
    tasp = oracle.link_bytes(2, P, T, cu, False, succ=succ, bytes_per_token=4)
    _full_allgather_closed_forms(ring, tasp, P, T)


def _rand_cu(rng, T, nd):
    cuts = np.sort(rng.choice(np.arange(1, T), size=nd - 1, replace=False))
    return np.concatenate([[0], cuts, [T]]).astype(np.int32)


@pytest.mark.parametrize("seed", range(8))
def test_matches_oracle_restatement(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([2, 3, 5, 7, 8, 9]))
    T = 2 * P * int(rng.integers(2, 30))
    cu = _rand_cu(rng, T, int(rng.integers(1, 6)))
    for kind in (0, 1, 2):
        succ = sb.sp_tasp_cycles(P, seed) if kind == 2 else None
        for causal in (False, True):
            for needed in (False, True):
                got = sb.sp_schedule_link_bytes(kind, P, T, cu, causal, seed=seed,
                                                bytes_per_token=3, needed_only=needed)
                exp = oracle.link_bytes(kind, P, T, cu, causal, succ, 3, needed)
                assert np.array_equal(got, exp), (kind, causal, needed)


def test_sequence_aware_never_sends_more_and_covers_every_item():
    cu = np.array([0, 700, 701, 2000, 4096], dtype=np.int32)
    T, P = 4096, 8
    for kind in (0, 1, 2):
        full = sb.sp_schedule_link_bytes(kind, P, T, cu, True)
        need = sb.sp_schedule_link_bytes(kind, P, T, cu, True, needed_only=True)
        assert np.all(need <= full) and need.sum() < full.sum()
        # Every key range a rank attends from another rank's chunk has to reach it.
        items = sb.sp_schedule_build(kind, P, T, cu, True)
        received = need.sum(axis=(0, 1))
        for r in range(P):
            remote = sum(int(it[6] - it[5]) for it in items if it[0] == r and it[1] > 0)
            assert received[r] >= remote
