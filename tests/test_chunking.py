"""Chunking policies (equal, work-balanced, balanced and moved onto document
starts) and schedules over explicit chunk bounds.

Pins for the oracle's chunk bounds: closed forms on a single document
(causal: the work of the first t rows is t(t+1)/2, so bound r solves a
quadratic; full mask: bound r = ceil(r T / P)), a per-document closed form of
W(t) for packed documents, and the balance invariant the definition implies.
The library must match the oracle exactly; its schedules over balanced bounds
must pass the oracle's schedule check (brute-force pair counting on small T)."""
import math

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl


def _work_prefix(cu, causal, t):
    """W(t) from per-document closed forms (no per-token loop)."""
    w = 0
    for d in range(len(cu) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        if t <= a:
            break
        m = min(t, b) - a
        w += m * (m + 1) // 2 if causal else m * (b - a)
    return w


@pytest.mark.parametrize("T,P", [(32768, 8), (1000, 7), (5, 8), (129, 2), (65536, 16)])
def test_oracle_single_doc_causal_closed_form(T, P):
    cu = np.array([0, T])
    got = [int(x) for x in oracle.chunk_bounds(1, P, T, cu, True)]
    total = T * (T + 1) // 2
    for r in range(1, P):
        # smallest t with P t (t+1) / 2 >= r T (T+1) / 2  <=>  t^2 + t >= r T (T+1) / P
        need = r * T * (T + 1)
        t = max(0, (math.isqrt(4 * need // P + 1) - 1) // 2 - 2)
        while P * t * (t + 1) < need:
            t += 1
        assert got[r] == t, (r, got[r], t)
        assert P * (got[r] * (got[r] + 1) // 2) >= r * total
    assert got[0] == 0 and got[P] == T


@pytest.mark.parametrize("T,P", [(65536, 16), (1000, 7), (3, 5)])
def test_oracle_single_doc_full_mask_closed_form(T, P):
    got = [int(x) for x in oracle.chunk_bounds(1, P, T, np.array([0, T]), False)]
    assert got == [0] + [-(-r * T // P) for r in range(1, P)] + [T]


def _random_cu(rng, T, ndocs):
    cuts = np.sort(rng.choice(np.arange(1, T), size=ndocs - 1, replace=False)) if ndocs > 1 else []
    return np.concatenate([[0], cuts, [T]]).astype(np.int32)


@pytest.mark.parametrize("causal", [True, False])
def test_oracle_packed_balance_invariant(causal):
    rng = np.random.default_rng(3)
    for _ in range(40):
        T = int(rng.integers(2, 3000))
        cu = _random_cu(rng, T, int(rng.integers(1, min(T, 12) + 1)))
        P = int(rng.integers(1, 20))
        b = oracle.chunk_bounds(1, P, T, cu, causal)
        W = _work_prefix(cu, causal, T)
        for r in range(1, P):
            # smallest t: P W(t) >= r W and P W(t-1) < r W
            assert P * _work_prefix(cu, causal, int(b[r])) >= r * W
            assert b[r] == 0 or P * _work_prefix(cu, causal, int(b[r]) - 1) < r * W
        assert np.all(np.diff(b) >= 0)


def test_oracle_doc_snap_rule():
    """Mode 2 restated with the per-document closed form of W: bound r moves to
    the document start nearest in work when that moves at most W(T) / (16P)."""
    rng = np.random.default_rng(8)
    cases = [(np.array([0, 240, 262, 600, 1000]), 1000, 4, False)]
    for _ in range(30):
        T = int(rng.integers(20, 3000))
        cases.append((_random_cu(rng, T, int(rng.integers(2, 15))), T, int(rng.integers(2, 12)),
                      bool(rng.integers(0, 2))))
    moved = 0
    for cu, T, P, causal in cases:
        bal = [int(x) for x in oracle.chunk_bounds(1, P, T, cu, causal)]
        snap = [int(x) for x in oracle.chunk_bounds(2, P, T, cu, causal)]
        W = _work_prefix(cu, causal, T)
        starts = [int(c) for c in cu[1:-1]]
        want = [0]
        for r in range(1, P):
            wb = _work_prefix(cu, causal, bal[r])
            near = min(starts, key=lambda c: (abs(_work_prefix(cu, causal, c) - wb), c))
            if 16 * P * abs(_work_prefix(cu, causal, near) - wb) <= W and near > want[-1]:
                want.append(near)
                moved += near != bal[r]
            else:
                want.append(max(bal[r], want[-1]))
        want.append(T)
        assert snap == want, (cu, P, causal)
    assert moved >= 5
    # One document only: nothing to snap to.
    assert np.array_equal(oracle.chunk_bounds(2, 4, 1000, np.array([0, 1000]), True),
                          oracle.chunk_bounds(1, 4, 1000, np.array([0, 1000]), True))


def test_library_matches_oracle_bounds():
    rng = np.random.default_rng(11)
    for _ in range(150):
        T = int(rng.integers(1, 5000))
        cu = _random_cu(rng, T, int(rng.integers(1, min(T, 30) + 1)))
        P = int(rng.integers(1, 40))
        causal = bool(rng.integers(0, 2))
        for mode in (0, 1, 2):
            assert np.array_equal(sb.sp_chunk_bounds(mode, P, T, cu, causal),
                                  oracle.chunk_bounds(mode, P, T, cu, causal)), (T, P, mode, causal)
    for w in wl.WORKLOADS:
        cu = wl.cu_seqlens(w)
        for mode in (0, 1, 2):
            assert np.array_equal(sb.sp_chunk_bounds(mode, w.P, w.T, cu, w.causal),
                                  oracle.chunk_bounds(mode, w.P, w.T, cu, w.causal))


def _ring_items(P, T, cu, causal, bounds):
    """RING over explicit chunks restated: rank r owns chunk r and at step s
    holds chunk (r - s) mod P; pairless items dropped."""
    out = []
    for r in range(P):
        qa, qb = int(bounds[r]), int(bounds[r + 1])
        for s in range(P):
            src = (r - s) % P
            ka, kb = int(bounds[src]), int(bounds[src + 1])
            if qa < qb and ka < kb and oracle.valid_pairs(cu, causal, qa, qb, ka, kb) > 0:
                out.append([r, s, 0, qa, qb, ka, kb])
    return np.array(out, dtype=np.int32).reshape(-1, 7)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mode", [1, 2])
def test_chunked_schedules_pass_oracle_check(causal, mode):
    rng = np.random.default_rng(5 + mode)
    for P, kind in ((5, sb.SP_SCHED_TASP), (3, sb.SP_SCHED_RING), (7, sb.SP_SCHED_TASP), (4, sb.SP_SCHED_RING)):
        T = 700
        cu = np.array([0, 130, 131, 400, 700], dtype=np.int32)
        bounds = sb.sp_chunk_bounds(mode, P, T, cu, causal)
        items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=1, bounds=bounds)
        succ = sb.sp_tasp_cycles(P, seed=1) if kind == sb.SP_SCHED_TASP else None
        rc, msg = oracle.check_schedule(kind, P, T, cu, causal, items, succ, brute=True, bounds=bounds)
        assert rc == 0, msg
        if kind == sb.SP_SCHED_RING:
            assert np.array_equal(items[:, :7], _ring_items(P, T, cu, causal, bounds))
        # Checked against other bounds the same items fail (ownership or pieces).
        eq = sb.sp_chunk_bounds(0, P, T, cu, causal)
        if not np.array_equal(eq, bounds):
            assert oracle.check_schedule(kind, P, T, cu, causal, items, succ, bounds=eq)[0] != 0
    # Random packings, balanced-doc TASP and RING.
    for _ in range(10):
        T = int(rng.integers(50, 900))
        cu = _random_cu(rng, T, int(rng.integers(1, 9)))
        for P, kind in ((5, sb.SP_SCHED_TASP), (6, sb.SP_SCHED_RING)):
            bounds = sb.sp_chunk_bounds(mode, P, T, cu, causal)
            items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=2, bounds=bounds)
            succ = sb.sp_tasp_cycles(P, seed=2) if kind == sb.SP_SCHED_TASP else None
            rc, msg = oracle.check_schedule(kind, P, T, cu, causal, items, succ, brute=True, bounds=bounds)
            assert rc == 0, msg


def test_equal_bounds_reproduce_default_schedule():
    cu = wl.cu_seqlens(wl.WORKLOADS[2])
    w = wl.WORKLOADS[2]
    a = sb.sp_schedule_build(w.kind, w.P, w.T, cu, True, seed=w.seed)
    b = sb.sp_schedule_build(w.kind, w.P, w.T, cu, True, seed=w.seed,
                             bounds=sb.sp_chunk_bounds(0, w.P, w.T, cu, True))
    assert np.array_equal(a, b)


def _rank_work(items, cu, causal, P):
    work = np.zeros(P)
    for it in items:
        work[it[0]] += oracle.valid_pairs(cu, causal, it[3], it[4], it[5], it[6])
    return work


@pytest.mark.parametrize("idx", [2, 4])
def test_balanced_chunks_even_out_rank_work(idx):
    """Packed causal workloads: equal chunks leave the busiest virtual rank with
    far more attention work than the mean; balanced chunks bring it to the mean
    within one row's work per rank."""
    w = wl.WORKLOADS[idx]
    cu = wl.cu_seqlens(w)
    res = {}
    for mode in (0, 1, 2):
        b = sb.sp_chunk_bounds(mode, w.P, w.T, cu, w.causal)
        items = sb.sp_schedule_build(w.kind, w.P, w.T, cu, w.causal, seed=w.seed, bounds=b)
        work = _rank_work(items, cu, w.causal, w.P)
        res[mode] = work.max() / work.mean()
    assert res[0] > 1.3
    assert res[1] < 1.001
    assert res[2] < 1.0 + 1.0 / 8 + 1e-3


def test_chunking_argument_errors():
    cu = np.array([0, 100, 256], dtype=np.int32)
    with pytest.raises(sb.SpError) as e:
        sb.sp_chunk_bounds(3, 4, 256, cu, True)
    assert e.value.code == 1
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_RING, 4, 256, cu, True, bounds=[0, 10, 5, 100, 256])
    assert e.value.code == 1
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_RING, 4, 256, cu, True, bounds=[0, 10, 20, 100, 255])
    assert e.value.code == 1
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build(sb.SP_SCHED_ZIGZAG, 4, 256, cu, True, bounds=[0, 32, 64, 96, 256])
    assert e.value.code == 2
    # Empty chunks are allowed: the rank has no work.
    items = sb.sp_schedule_build(sb.SP_SCHED_RING, 4, 256, cu, True, bounds=[0, 0, 100, 100, 256])
    rc, msg = oracle.check_schedule(0, 4, 256, cu, True, items, brute=True,
                                    bounds=np.array([0, 0, 100, 100, 256]))
    assert rc == 0, msg
    assert set(items[:, 0]) == {1, 3}
