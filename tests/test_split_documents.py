"""sp_schedule_split_documents: every schedule item cut at the document
boundaries of the packing. Checked by brute force on small inputs (each valid
(query, key) pair, defined by the oracle's document lookup and the causal
rule, is covered exactly once, as by the uncut schedule), piece by piece (each
piece lies inside one document and is its parent item intersected with that
document, same rank, step and cycle, flags recomputed) and by its ordering
(pieces of one rank, Q range and head range are adjacent; a rank's pieces go in
token order)."""
import ctypes

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl


def _rand_cu(rng, T, max_docs):
    nd = min(int(rng.integers(1, max_docs + 1)), T)
    cuts = np.sort(rng.choice(np.arange(1, T), size=nd - 1, replace=False)) if nd > 1 else []
    return np.concatenate([[0], cuts, [T]]).astype(np.int32)


def _coverage(items, cu, causal, T):
    """Count of items covering each (query, key) pair, the valid-pair mask and
    the same-document mask."""
    doc = np.array([oracle.doc_of(cu, t) for t in range(T)])
    same = doc[:, None] == doc[None, :]
    valid = same.copy()
    if causal:
        valid &= np.arange(T)[None, :] <= np.arange(T)[:, None]
    cnt = np.zeros((T, T), dtype=np.int32)
    for it in items:
        cnt[it[3]:it[4], it[5]:it[6]] += 1
    return cnt, valid, same


def _check_pieces(items, split, cu, causal):
    cu_l = [int(x) for x in cu]
    parent = {}
    for it in items:
        parent.setdefault((int(it[0]), int(it[1]), int(it[2])), []).append(it)
    for p in split:
        qa, qb, ka, kb = (int(x) for x in p[3:7])
        d = oracle.doc_of(cu, qa)
        # One document for the whole piece.
        assert oracle.doc_of(cu, qb - 1) == d and oracle.doc_of(cu, ka) == d and oracle.doc_of(cu, kb - 1) == d
        ds, de = cu_l[d], cu_l[d + 1]
        # Some parent with the same (rank, step, cycle) gives exactly this piece.
        found = False
        for it in parent[(int(p[0]), int(p[1]), int(p[2]))]:
            if (max(int(it[3]), ds), min(int(it[4]), de), max(int(it[5]), ds), min(int(it[6]), de)) == (qa, qb, ka, kb):
                found = True
                break
        assert found, p
        assert oracle.valid_pairs(cu, causal, qa, qb, ka, kb) > 0
        flags = 1 if (causal and kb - 1 > qa) else 0
        assert int(p[7]) == flags


def _check_order(split, heads=None):
    keys = [(int(r[0]), int(r[3]), int(r[4])) + ((int(heads[i][0]), int(heads[i][1])) if heads is not None else ())
            for i, r in enumerate(split)]
    seen = set()
    for i, key in enumerate(keys):
        if i == 0 or key != keys[i - 1]:
            assert key not in seen, key  # one contiguous run per (rank, Q range, heads)
            seen.add(key)
    for i in range(1, len(split)):
        same = split[i][0] == split[i - 1][0] and (heads is None or tuple(heads[i]) == tuple(heads[i - 1]))
        if same:
            assert split[i][3] >= split[i - 1][3]  # a rank's Q pieces in token order


@pytest.mark.parametrize("seed", range(10))
def test_split_covers_the_same_pairs_brute(seed):
    rng = np.random.default_rng(100 + seed)
    P = int(rng.choice([1, 2, 3, 5, 7, 8]))
    T = 2 * P * int(rng.integers(1, 30))
    cu = _rand_cu(rng, T, 7)
    for causal in (True, False):
        for kind in (0, 1, 2):
            items = sb.sp_schedule_build(kind, P, T, cu, causal, seed=seed)
            split = sb.sp_schedule_split_documents(items, cu, causal)
            cnt, valid, same = _coverage(split, cu, causal, T)
            assert (cnt[valid] == 1).all(), (kind, P, T)
            assert (cnt[~same] == 0).all()  # the pieces hold no cross-document pair
            cnt0, _, _ = _coverage(items, cu, causal, T)
            assert np.array_equal(cnt0[valid], cnt[valid])
            _check_pieces(items, split, cu, causal)
            _check_order(split)
            # Cutting again changes nothing.
            assert np.array_equal(sb.sp_schedule_split_documents(split, cu, causal), split)


def test_single_document_is_unchanged():
    for kind, P, T in ((0, 4, 256), (1, 4, 256), (2, 5, 250)):
        items = sb.sp_schedule_build(kind, P, T, [0, T], True)
        assert np.array_equal(sb.sp_schedule_split_documents(items, [0, T], True), items)


def test_worked_example():
    """Two documents [0, 100) and [100, 256), RING over 4 ranks of 64 tokens:
    rank 1 holds Q [64, 128), which meets both documents; its step-0 item (KV
    [64, 128)) becomes Q [64, 100) x KV [64, 100) and Q [100, 128) x KV [100, 128);
    its step-1 item (KV [0, 64)) keeps only the first document's rows."""
    cu = [0, 100, 256]
    items = sb.sp_schedule_build(0, 4, 256, cu, True)
    split = sb.sp_schedule_split_documents(items, cu, True)
    r1 = [tuple(int(x) for x in it[:7]) for it in split if it[0] == 1]
    assert r1 == [(1, 0, 0, 64, 100, 64, 100), (1, 1, 0, 64, 100, 0, 64), (1, 0, 0, 100, 128, 100, 128)]


@pytest.mark.parametrize("causal", [True, False])
def test_split_with_head_ranges(causal):
    rng = np.random.default_rng(7)
    T, R, U, Hq = 240, 3, 2, 8
    cu = _rand_cu(rng, T, 5)
    items, heads = sb.sp_schedule_build_hier(0, R, U, T, cu, causal, Hq)
    split, sh = sb.sp_schedule_split_documents(items, cu, causal, heads=heads)
    assert len(split) == len(sh)
    _check_order(split, sh)
    # Per head range, the same pieces as cutting that head range's items alone.
    for h in {tuple(x) for x in heads.tolist()}:
        sel = (heads[:, 0] == h[0]) & (heads[:, 1] == h[1])
        alone = sb.sp_schedule_split_documents(items[sel], cu, causal)
        ssel = (sh[:, 0] == h[0]) & (sh[:, 1] == h[1])
        assert np.array_equal(split[ssel], alone)
    # Ranks of one group hold the same pieces for different heads.
    rc, msg = oracle.check_hier_schedule(0, R, U, Hq, T, cu, causal, items, heads, brute=True)
    assert rc == 0, msg


def test_workload_splits():
    """The packed workloads: pairs kept, every piece inside one document, the
    single-document workloads unchanged."""
    import bench
    for w in wl.WORKLOADS:
        cu = wl.cu_seqlens(w)
        items = sb.sp_schedule_build(w.kind, w.P, w.T, cu, w.causal, seed=w.seed)
        split = sb.sp_schedule_split_documents(items, cu, w.causal)
        assert sum(bench.valid_pairs_range(cu, w.causal, it) for it in split) == bench.valid_pairs(cu, w.causal)
        if len(cu) == 2:
            assert np.array_equal(split, items)
        d0 = np.searchsorted(cu, split[:, 3], side="right")
        for col in (4, 5, 6):
            off = 1 if col in (4, 6) else 0
            assert np.array_equal(np.searchsorted(cu, split[:, col] - off, side="right"), d0)
        _check_order(split)
        # Every piece is its parent intersected with one document, so the pieces
        # cover each valid pair exactly once when the parents do (the schedule
        # tests check that), and no (parent, document) with a valid pair is lost:
        # the valid pairs add up to the workload's (above).
        _check_pieces(items, split, cu, w.causal)


def test_argument_errors():
    lib = sb.load()
    cu = np.array([0, 10, 20], dtype=np.int32)
    good = np.array([[0, 0, 0, 0, 20, 0, 20, 3]], dtype=np.int32)
    n = ctypes.c_int64(0)
    call = lambda it, c, nd, out, cap, heads=None, out_h=None: lib.sp_schedule_split_documents(
        it.ctypes.data, heads, len(it), c.ctypes.data, nd, 1, out, out_h, ctypes.byref(cap))
    assert call(good, cu, 2, None, n) == 0 and n.value == 2
    small = ctypes.c_int64(1)
    out = np.zeros((2, 8), dtype=np.int32)
    assert call(good, cu, 2, out.ctypes.data, small) == 3 and small.value == 2  # SP_ERR_BUFFER_TOO_SMALL
    for bad_cu in (np.array([0, 20, 10], dtype=np.int32), np.array([1, 10, 20], dtype=np.int32)):
        assert call(good, bad_cu, 2, None, ctypes.c_int64(0)) == 1
    for bad in ([0, 0, 0, 5, 5, 0, 20, 0], [0, 0, 0, 0, 21, 0, 20, 0], [0, 0, 0, 0, 20, -1, 20, 0]):
        assert call(np.array([bad], dtype=np.int32), cu, 2, None, ctypes.c_int64(0)) == 1
    heads = np.array([[0, 4]], dtype=np.int32)
    cap = ctypes.c_int64(2)
    assert call(good, cu, 2, out.ctypes.data, cap, heads.ctypes.data, None) == 1  # out_heads missing
    with pytest.raises(sb.SpError):
        sb.sp_schedule_split_documents(good, [0, 10, 19], True)  # item past the last token
    assert len(sb.sp_schedule_split_documents(np.zeros((0, 8), dtype=np.int32), cu, True)) == 0
    e, eh = sb.sp_schedule_split_documents(np.zeros((0, 8), dtype=np.int32), cu, True,
                                           heads=np.zeros((0, 2), dtype=np.int32))
    assert len(e) == 0 and len(eh) == 0


def test_group_limit_and_fallback():
    """sp_packed_attention takes at most SP_MAX_GROUPS groups; PackedAttention
    keeps the items as built when cutting them would pass that."""
    import os
    import re
    header = os.path.join(os.path.dirname(__file__), "..", "include", "sp_attn.h")
    assert int(re.search(r"#define SP_MAX_GROUPS (\d+)", open(header).read()).group(1)) == sb.SP_MAX_GROUPS
    items = np.array([[0, 0, 0, 0, 4, 0, 4, 0], [0, 1, 0, 0, 4, 4, 8, 0], [1, 0, 0, 4, 8, 4, 8, 0],
                      [0, 2, 0, 0, 4, 8, 9, 0]], dtype=np.int32)
    assert sb.n_groups(items) == 3 and sb.n_groups(items[:0]) == 0
    assert sb.n_groups(items, np.array([[0, 2], [2, 4], [0, 2], [0, 2]])) == 4
    few = wl.cu_from_lengths([300, 212])
    att = sb.PackedAttention(few, True, sb.SP_SCHED_RING, 2, 4, device="cpu")
    assert att.documents_cut and sb.n_groups(att.items) == 3
    many = wl.cu_from_lengths([8] * 10000)  # 10,000 documents: 10,000 groups once cut
    att = sb.PackedAttention(many, True, sb.SP_SCHED_RING, 2, 4, device="cpu")
    assert not att.documents_cut
    assert np.array_equal(att.items, sb.sp_schedule_build(sb.SP_SCHED_RING, 2, 80000, many, True))
    assert sb.n_groups(sb.sp_schedule_split_documents(att.items, many, True)) > sb.SP_MAX_GROUPS
