"""Two-level schedules (Inter-SP schedule between R groups, query heads split
over the U ranks of a group) and the oracle's check for them: the check
reduces the schedule to U head slices, each an R-rank schedule verified by
the pinned single-level check with brute-force pair counting, and rejects
planted defects."""
import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl


def _succ(kind, R, seed):
    return sb.sp_tasp_cycles(R, seed) if kind == sb.SP_SCHED_TASP and R > 1 else None


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind,R,U,Hq", [(sb.SP_SCHED_RING, 2, 8, 16), (sb.SP_SCHED_TASP, 3, 2, 8),
                                         (sb.SP_SCHED_ZIGZAG, 2, 4, 8), (sb.SP_SCHED_TASP, 5, 4, 4),
                                         (sb.SP_SCHED_RING, 1, 4, 32)])
def test_hier_schedule_passes_oracle_check(kind, R, U, Hq, causal):
    T = 720
    cu = np.array([0, 130, 131, 400, 720], dtype=np.int32)
    items, heads = sb.sp_schedule_build_hier(kind, R, U, T, cu, causal, Hq, seed=4)
    flat = sb.sp_schedule_build(kind, R, T, cu, causal, seed=4)
    assert len(items) == U * len(flat)
    rc, msg = oracle.check_hier_schedule(kind, R, U, Hq, T, cu, causal, items, heads, _succ(kind, R, 4),
                                         brute=True)
    assert rc == 0, msg
    # Every rank appears, with its own head slice; order by rank.
    assert np.all(np.diff(items[:, 0]) >= 0)
    for r in np.unique(items[:, 0]):
        hs = heads[items[:, 0] == r]
        u = r % U
        assert np.all(hs[:, 0] == u * Hq // U) and np.all(hs[:, 1] == (u + 1) * Hq // U)


def test_one_rank_per_group_is_the_flat_schedule():
    w = wl.WORKLOADS[2]
    cu = wl.cu_seqlens(w)
    items, heads = sb.sp_schedule_build_hier(w.kind, w.P, 1, w.T, cu, True, w.Hq, seed=w.seed)
    assert np.array_equal(items, sb.sp_schedule_build(w.kind, w.P, w.T, cu, True, seed=w.seed))
    assert np.all(heads[:, 0] == 0) and np.all(heads[:, 1] == w.Hq)


def test_hier_with_balanced_group_chunks():
    w = wl.WORKLOADS[2]
    cu = wl.cu_seqlens(w)
    R, U = 5, 2
    bounds = sb.sp_chunk_bounds(sb.SP_CHUNK_BALANCED, R, w.T, cu, True)
    items, heads = sb.sp_schedule_build_hier(sb.SP_SCHED_TASP, R, U, w.T, cu, True, w.Hq, seed=1,
                                             bounds=bounds)
    rc, msg = oracle.check_hier_schedule(sb.SP_SCHED_TASP, R, U, w.Hq, w.T, cu, True, items, heads,
                                         sb.sp_tasp_cycles(R, 1), bounds=bounds)
    assert rc == 0, msg


def test_hier_check_rejects_planted_defects():
    T, Hq, R, U = 512, 8, 2, 4
    cu = np.array([0, 200, 512], dtype=np.int32)
    items, heads = sb.sp_schedule_build_hier(sb.SP_SCHED_RING, R, U, T, cu, True, Hq)
    ok = oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items, heads, brute=True)
    assert ok[0] == 0, ok[1]
    # A head range that is not the rank's slice.
    bad = heads.copy()
    bad[3] = [0, 2]
    if not np.array_equal(bad[3], heads[3]):
        assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items, bad)[0] == 22
    # One slice loses an item: its keys are no longer covered.
    keep = np.ones(len(items), dtype=bool)
    keep[np.nonzero(items[:, 0] == 1)[0][-1]] = False
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items[keep], heads[keep])[0] == 39
    # A duplicated item in one slice: overlap.
    dup_i = np.concatenate([items, items[-1:]])
    dup_h = np.concatenate([heads, heads[-1:]])
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, dup_i, dup_h)[0] == 38
    # A rank outside R * U.
    big = items.copy()
    big[0, 0] = R * U
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, big, heads)[0] == 21


def test_hier_argument_errors():
    cu = np.array([0, 256], dtype=np.int32)
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build_hier(sb.SP_SCHED_RING, 2, 3, 256, cu, True, 8)  # 8 % 3 != 0
    assert e.value.code == 1
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build_hier(sb.SP_SCHED_TASP, 4, 2, 256, cu, True, 8)  # no decomposition of K4*
    assert e.value.code == 2
    with pytest.raises(sb.SpError) as e:
        sb.sp_schedule_build_hier(sb.SP_SCHED_RING, 0, 2, 256, cu, True, 8)
    assert e.value.code == 1


# ------------------------------------------------------------------ communication

@pytest.mark.parametrize("kind,R,U,Hq,Hkv,causal,needed", [
    (sb.SP_SCHED_RING, 2, 8, 16, 16, False, False), (sb.SP_SCHED_TASP, 3, 2, 8, 2, True, True),
    (sb.SP_SCHED_ZIGZAG, 2, 4, 8, 2, True, False), (sb.SP_SCHED_RING, 4, 2, 8, 8, True, True),
    (sb.SP_SCHED_RING, 1, 4, 8, 8, True, False), (sb.SP_SCHED_TASP, 5, 4, 32, 8, True, False)])
def test_hier_link_bytes_match_oracle(kind, R, U, Hq, Hkv, causal, needed):
    T = 720
    cu = np.array([0, 130, 131, 400, 720], dtype=np.int32)
    succ = _succ(kind, R, 3)
    a = sb.sp_schedule_link_bytes_hier(kind, R, U, T, cu, causal, Hq, Hkv, 64, 2, seed=3, needed_only=needed)
    b = oracle.link_bytes_hier(kind, R, U, T, cu, causal, Hq, Hkv, 64, 2, succ=succ, needed_only=needed)
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(a[1], b[1])


def test_hier_link_bytes_closed_forms():
    """One group: no Inter-SP traffic, and each rank sends its T/U tokens' q and
    k, v of the other slices' heads and gets o back (hand count). One rank per
    group: no all-to-all, Inter-SP equals the flat model."""
    T, U, Hq, Hkv, d = 512, 4, 8, 2, 64
    cu = np.array([0, 512], dtype=np.int32)
    intra, inter = sb.sp_schedule_link_bytes_hier(sb.SP_SCHED_RING, 1, U, T, cu, True, Hq, Hkv, d, 2)
    assert inter.shape[0] == 0
    n = T // U
    hs, kvs = Hq // U, 1      # 2 query heads per slice, inside one KV group of 4
    for u in range(U):
        for v in range(U):
            want = 0 if u == v else n * (hs + 2 * kvs) * d * 2 + n * hs * d * 2
            assert intra[u, v] == want, (u, v)
    R = 4
    intra, inter = sb.sp_schedule_link_bytes_hier(sb.SP_SCHED_RING, R, 1, T, cu, True, Hq, Hkv, d, 2)
    assert not intra.any()
    flat = sb.sp_schedule_link_bytes(sb.SP_SCHED_RING, R, T, cu, True, bytes_per_token=2 * Hkv * d * 2)
    assert np.array_equal(inter, flat)


# ------------------------------------------------------------------ oracle-only pins
# These call the oracle alone: the two-level items are restated here from the
# oracle's flat closed form (pinned by hand-derived lists), and the
# communication counts are written down by hand.

def _restated_hier(kind, R, U, Hq, T, cu, causal):
    """Every item of group g of the flat R-rank schedule, held by the U ranks
    g*U + u, each for query heads [u Hq/U, (u+1) Hq/U)."""
    flat = oracle.closed_form_schedule(kind, R, T, cu, causal)
    hs = Hq // U
    items, heads = [], []
    for it in flat:
        for u in range(U):
            x = it.copy()
            x[0] = it[0] * U + u
            items.append(x)
            heads.append([u * hs, (u + 1) * hs])
    return np.array(items, dtype=np.int32).reshape(-1, 8), np.array(heads, dtype=np.int32).reshape(-1, 2)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kind,R,U,Hq", [(0, 2, 4, 8), (1, 2, 2, 4), (0, 3, 2, 6), (0, 1, 4, 8), (1, 3, 1, 2)])
def test_oracle_hier_check_accepts_restated_schedules(kind, R, U, Hq, causal):
    T = 240
    cu = np.array([0, 50, 51, 180, 240], dtype=np.int32)
    items, heads = _restated_hier(kind, R, U, Hq, T, cu, causal)
    rc, msg = oracle.check_hier_schedule(kind, R, U, Hq, T, cu, causal, items, heads, brute=True)
    assert rc == 0, msg


def test_oracle_hier_check_rejects_defects_on_restated_schedule():
    T, Hq, R, U = 240, 8, 2, 4
    hs = Hq // U
    cu = np.array([0, 100, 240], dtype=np.int32)
    items, heads = _restated_hier(0, R, U, Hq, T, cu, True)
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items, heads, brute=True)[0] == 0
    x = int(np.nonzero(items[:, 0] % U == 1)[0][0])
    bad = heads.copy()
    bad[x] = heads[x] + hs                       # another slice's heads
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items, bad)[0] == 22
    bad = heads.copy()
    bad[x, 1] -= 1                               # right start, one head short
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items, bad)[0] == 22
    keep = np.ones(len(items), dtype=bool)       # slice 1 loses an item
    keep[np.nonzero(items[:, 0] % U == 1)[0][-1]] = False
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, items[keep], heads[keep])[0] == 39
    dup_i = np.concatenate([items, items[x:x + 1]])
    dup_h = np.concatenate([heads, heads[x:x + 1]])
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, dup_i, dup_h)[0] == 38
    big = items.copy()
    big[0, 0] = R * U
    assert oracle.check_hier_schedule(0, R, U, Hq, T, cu, True, big, heads)[0] == 21


def test_oracle_hier_link_bytes_closed_forms():
    """One group over U = 4 ranks of unequal token counts (510 = 128 + 128 +
    127 + 127): rank a sends rank b the q and the k, v of a's tokens for b's
    heads, and returns to b the o of b's tokens for a's heads, so
    intra[a, b] = n_a (hs + 2 kvs) d eb + n_b hs d eb. One rank per group: no
    all-to-all, and the Inter-SP traffic is the flat model's with k and v of
    every key/value head per token."""
    T, U, Hq, Hkv, d, eb = 510, 4, 8, 2, 64, 2
    cu = np.array([0, T], dtype=np.int32)
    intra, inter = oracle.link_bytes_hier(0, 1, U, T, cu, True, Hq, Hkv, d, eb)
    assert inter.shape[0] == 0
    n = [128, 128, 127, 127]
    hs, kvs = Hq // U, 1      # 2 query heads per slice, inside one key/value group of 4
    for a in range(U):
        for b in range(U):
            want = 0 if a == b else n[a] * (hs + 2 * kvs) * d * eb + n[b] * hs * d * eb
            assert intra[a, b] == want, (a, b)
    R = 4
    cu = np.array([0, 200, 512], dtype=np.int32)
    intra, inter = oracle.link_bytes_hier(0, R, 1, 512, cu, True, Hq, Hkv, d, eb)
    assert not intra.any()
    flat = oracle.link_bytes(0, R, 512, cu, True, bytes_per_token=2 * Hkv * d * eb)
    assert np.array_equal(inter, flat)
