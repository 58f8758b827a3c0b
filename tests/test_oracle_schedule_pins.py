"""Pins for the oracle's schedule checks: hand-derived item lists, a closed-form
Hamiltonian decomposition for prime P, exhaustive non-existence for P = 4, and
planted defects that each check must reject."""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_items(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([int(x) for x in line.split()] + [0])
    return np.array(rows, dtype=np.int32)


def test_ring_closed_form_matches_hand_derivation():
    gold = _load_items("ring_P4_T256_docs100_156_causal.txt")
    cu = np.array([0, 100, 256])
    got = oracle.closed_form_schedule(0, 4, 256, cu, True)
    assert np.array_equal(got[:, :7], gold[:, :7])
    rc, msg = oracle.check_schedule(0, 4, 256, cu, True, gold, brute=True)
    assert rc == 0, msg


def test_zigzag_closed_form_matches_hand_derivation():
    gold = _load_items("zigzag_P2_T8_causal.txt")
    cu = np.array([0, 8])
    got = oracle.closed_form_schedule(1, 2, 8, cu, True)
    assert np.array_equal(got[:, :7], gold[:, :7])
    rc, msg = oracle.check_schedule(1, 2, 8, cu, True, gold, brute=True)
    assert rc == 0, msg
    assert oracle.closed_form_schedule(1, 3, 8, cu, True) is None  # 8 % 6 != 0


def _cyclic_decomposition(P):
    """For prime P the arcs u -> u + s (s = 1..P-1) form P-1 Hamiltonian cycles."""
    return np.array([[(u + s) % P for u in range(P)] for s in range(1, P)], dtype=np.int32)


@pytest.mark.parametrize("P", [2, 3, 5, 7, 11, 13])
def test_hamiltonian_check_accepts_cyclic_prime(P):
    assert oracle.check_hamiltonian(P, _cyclic_decomposition(P)) == 0


def _ham_cycles(P):
    """Every directed Hamiltonian cycle of the complete digraph as a successor array."""
    out = []
    for perm in itertools.permutations(range(1, P)):
        order = (0,) + perm
        succ = [0] * P
        for a, b in zip(order, order[1:] + (0,)):
            succ[a] = b
        out.append(succ)
    return out


def test_no_decomposition_for_p4_exhaustive():
    cycles = _ham_cycles(4)
    assert len(cycles) == 6
    for trio in itertools.combinations(cycles, 3):
        assert oracle.check_hamiltonian(4, np.array(trio, dtype=np.int32)) != 0


def test_hamiltonian_check_rejects_defects():
    good = _cyclic_decomposition(5)
    bad = good.copy()
    bad[1] = bad[0]                       # repeated arcs
    assert oracle.check_hamiltonian(5, bad) == 3
    bad = good.copy()
    bad[0] = [1, 0, 3, 4, 2]              # a 2-cycle plus a 3-cycle
    assert oracle.check_hamiltonian(5, bad) == 2
    bad = good.copy()
    bad[2, 3] = 3                         # self loop
    assert oracle.check_hamiltonian(5, bad) == 1
    # Rows whose walk from vertex 0 is back at 0 after P arcs without having
    # visited every vertex (the cycle through 0 is shorter and its length
    # divides P). K_4* split into three factors of two 2-cycles uses every arc
    # exactly once and is still not a decomposition into Hamiltonian cycles.
    two_cycle_factors = np.array([[1, 0, 3, 2], [2, 3, 0, 1], [3, 2, 1, 0]], dtype=np.int32)
    assert oracle.check_hamiltonian(4, two_cycle_factors) == 2
    two_triangles = np.array([[1, 2, 0, 4, 5, 3]] + [[(u + 1) % 6 for u in range(6)]] * 4, dtype=np.int32)
    assert oracle.check_hamiltonian(6, two_triangles) == 2


def _split(n, parts, idx):
    base, extra = divmod(n, parts)
    b = idx * base + min(idx, extra)
    return b, b + base + (1 if idx < extra else 0)


def _tasp_items(P, T, cu, causal, succ):
    """TASP schedule restated from the abstract: step 0 is the local chunk; at
    step t every cycle c delivers piece c of the chunk t hops upstream."""
    pred = np.zeros_like(succ)
    for c in range(P - 1):
        pred[c, succ[c]] = np.arange(P)
    items = []
    for r in range(P):
        qa, qb = _split(T, P, r)
        cand = [(0, 0, _split(T, P, r))]
        for t in range(1, P):
            for c in range(P - 1):
                src = r
                for _ in range(t):
                    src = pred[c, src]
                cb, ce = _split(T, P, src)
                pb, pe = _split(ce - cb, P - 1, c)
                cand.append((t, c, (cb + pb, cb + pe)))
        for t, c, (ka, kb) in cand:
            if kb > ka and oracle.valid_pairs(cu, causal, qa, qb, ka, kb) > 0:
                items.append([r, t, c, qa, qb, ka, kb, 0])
    return np.array(items, dtype=np.int32)


@pytest.mark.parametrize("causal", [True, False])
def test_tasp_restatement_accepted_and_defects_rejected(causal):
    P, T = 5, 203
    cu = np.array([0, 17, 18, 120, 203])
    succ = _cyclic_decomposition(P)
    items = _tasp_items(P, T, cu, causal, succ)
    rc, msg = oracle.check_schedule(2, P, T, cu, causal, items, succ, brute=True)
    assert rc == 0, msg
    # Wrong source chunk for one relayed piece.
    bad = items.copy()
    i = int(np.nonzero(bad[:, 1] > 0)[0][0])
    bad[i, 1] = (bad[i, 1] % (P - 1)) + 1 if P > 2 else bad[i, 1]
    if not np.array_equal(bad, items):
        assert oracle.check_schedule(2, P, T, cu, causal, bad, succ)[0] != 0
    # A broken decomposition is caught before the items are looked at.
    bsucc = succ.copy()
    bsucc[1] = bsucc[0]
    assert oracle.check_schedule(2, P, T, cu, causal, items, bsucc)[0] == 2


def test_schedule_check_rejects_planted_defects():
    cu = np.array([0, 100, 256])
    gold = _load_items("ring_P4_T256_docs100_156_causal.txt")
    # Missing item: a needed key range is no longer covered.
    assert oracle.check_schedule(0, 4, 256, cu, True, gold[:-1])[0] == 9
    # Duplicated item: overlapping key ranges (a pair computed twice).
    dup = np.concatenate([gold, gold[-1:]])
    assert oracle.check_schedule(0, 4, 256, cu, True, dup)[0] == 8
    # An item with no valid pair (pruning violated): rank 0 step 1 chunk 3.
    extra = np.concatenate([gold, np.array([[0, 1, 0, 0, 64, 192, 256, 0]], dtype=np.int32)])
    assert oracle.check_schedule(0, 4, 256, cu, True, extra)[0] == 4
    # A Q range that the rank does not own.
    wrong = gold.copy()
    wrong[0, 0] = 1
    assert oracle.check_schedule(0, 4, 256, cu, True, wrong)[0] == 5
    # Out-of-range tokens.
    oob = gold.copy()
    oob[-1, 6] = 300
    assert oracle.check_schedule(0, 4, 256, cu, True, oob)[0] == 3
    # The brute-force pair count sees a gap inside a kept item.
    shrunk = gold.copy()
    shrunk[1, 6] = 127      # rank 1 step 0 loses key 127
    rc, _ = oracle.check_schedule(0, 4, 256, cu, True, shrunk, brute=True)
    assert rc != 0


def test_cu_seqlens_validation():
    assert oracle.check_cu_seqlens(np.array([0, 5, 9]), 9) == 0
    assert oracle.check_cu_seqlens(np.array([1, 5, 9]), 9) != 0
    assert oracle.check_cu_seqlens(np.array([0, 5, 5, 9]), 9) != 0
    assert oracle.check_cu_seqlens(np.array([0, 5, 8]), 9) != 0
    assert oracle.doc_of(np.array([0, 5, 9]), 4) == 0
    assert oracle.doc_of(np.array([0, 5, 9]), 5) == 1
