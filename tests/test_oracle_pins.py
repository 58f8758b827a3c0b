"""Pins for the fp64 attention oracle, against things other than itself.

* brute force: a dense T x T formulation in long double with no max
  subtraction, on tiny inputs;
* closed forms (Q = 0, equal keys, constant V, the first token of a document,
  and the hand-derived three-token fixture in tests/golden);
* a library special case: torch scaled_dot_product_attention in float64;
* invariants: merging partials over any key partition in any order gives the
  full result; perturbing one packed document leaves every other document's
  output bit-identical.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_docs(rng, T, max_docs):
    nd = int(rng.integers(1, max_docs + 1))
    nd = min(nd, T)
    cuts = np.sort(rng.choice(np.arange(1, T), size=nd - 1, replace=False)) if nd > 1 else []
    return np.concatenate([[0], cuts, [T]]).astype(np.int32)


def _brute(q, k, v, cu, causal, scale):
    """Dense masked softmax in long double: exp of raw scores, masked entries 0."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    ld = np.longdouble
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    valid = doc[:, None] == doc[None, :]
    if causal:
        valid &= np.arange(T)[None, :] <= np.arange(T)[:, None]
    O = np.zeros((T, Hq, d), dtype=ld)
    L = np.zeros((T, Hq), dtype=ld)
    for h in range(Hq):
        g = h // G
        S = np.einsum("ic,jc->ij", q[:, h, :].astype(ld), k[:, g, :].astype(ld)) * ld(scale)
        E = np.where(valid, np.exp(S), ld(0))
        Z = E.sum(axis=1)
        L[:, h] = np.log(Z)
        O[:, h, :] = np.einsum("ij,jc->ic", E, v[:, g, :].astype(ld)) / Z[:, None]
    return O.astype(np.float64), L.astype(np.float64)


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_small(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.choice([1, 2, 7, 33, 64]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    Hq = Hkv * G
    d = int(rng.choice([4, 8, 16]))
    causal = bool(seed % 2)
    cu = _rand_docs(rng, T, 5)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attn(q, k, v, cu, causal)
    ob, lb = _brute(q, k, v, cu, causal, scale)
    assert np.max(np.abs(o - ob)) < 1e-12
    assert np.max(np.abs(lse - lb)) < 1e-12


def test_three_token_golden():
    fx = json.load(open(os.path.join(GOLDEN, "three_token_closed_form.json")))
    q = np.array(fx["q"], dtype=np.float64)
    k = np.array([[[float(x) for x in row[0]]] for row in fx["k"]], dtype=np.float64)
    v = np.array(fx["v"], dtype=np.float64)
    ln = {"0": 0.0, "ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4),
          "ln5": math.log(5), "ln6": math.log(6)}

    def num(x):
        if isinstance(x, str) and "/" in x:
            a, b = x.split("/")
            return float(a) / float(b)
        return float(x)

    for case in fx["cases"]:
        o, lse = oracle.attn(q, k, v, np.array(case["cu_seqlens"]), case["causal"])
        exp_o = np.array([[num(x) for x in row] for row in case["O"]])
        exp_l = np.array([ln[x] for x in case["LSE"]])
        assert np.max(np.abs(o[:, 0, :] - exp_o)) < 1e-12, case
        assert np.max(np.abs(lse[:, 0] - exp_l)) < 1e-12, case


def _valid_sets(cu, T, causal):
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    sets = []
    for i in range(T):
        js = [j for j in range(T) if doc[j] == doc[i] and (not causal or j <= i)]
        sets.append(js)
    return sets


@pytest.mark.parametrize("causal", [True, False])
def test_closed_form_zero_query_and_equal_keys(causal):
    rng = np.random.default_rng(7)
    T, Hq, Hkv, d = 40, 4, 2, 8
    cu = np.array([0, 9, 10, 31, 40], dtype=np.int32)
    v = rng.standard_normal((T, Hkv, d))
    sets = _valid_sets(cu, T, causal)
    # Q = 0: all scores 0 -> uniform weights.
    q0 = np.zeros((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    # Equal keys (any Q): all scores of a row are equal -> uniform weights.
    q1 = rng.standard_normal((T, Hq, d))
    keq = np.broadcast_to(rng.standard_normal((1, Hkv, d)), (T, Hkv, d)).copy()
    for q, kk in ((q0, k), (q1, keq)):
        o, lse = oracle.attn(q, kk, v, cu, causal)
        for i in range(T):
            js = sets[i]
            for h in range(Hq):
                g = h // (Hq // Hkv)
                mean = v[js, g, :].mean(axis=0)
                assert np.max(np.abs(o[i, h] - mean)) < 1e-12
                if q is q0:
                    assert abs(lse[i, h] - math.log(len(js))) < 1e-12
                else:
                    s = float(q[i, h] @ kk[0, g]) / math.sqrt(d)
                    assert abs(lse[i, h] - (s + math.log(len(js)))) < 1e-12


def test_constant_values_and_first_token():
    rng = np.random.default_rng(11)
    T, Hq, Hkv, d = 50, 2, 1, 16
    cu = np.array([0, 1, 17, 50], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = np.full((T, Hkv, d), 2.75)
    o, _ = oracle.attn(q, k, v, cu, True)
    assert np.max(np.abs(o - 2.75)) < 1e-12
    v = rng.standard_normal((T, Hkv, d))
    o, lse = oracle.attn(q, k, v, cu, True)
    for D in range(len(cu) - 1):
        t = int(cu[D])
        for h in range(Hq):
            assert np.max(np.abs(o[t, h] - v[t, 0])) < 1e-12
            assert abs(lse[t, h] - float(q[t, h] @ k[t, 0]) / math.sqrt(d)) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_sdpa_single_doc(causal):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    T, Hq, Hkv, d = 96, 8, 2, 32
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    o, _ = oracle.attn(q, k, v, np.array([0, T]), causal)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(o - ref)) < 1e-10


@pytest.mark.parametrize("seed", range(4))
def test_merge_over_random_partitions(seed):
    rng = np.random.default_rng(100 + seed)
    T, Hq, Hkv, d = 80, 4, 2, 8
    causal = bool(seed % 2)
    cu = _rand_docs(rng, T, 4)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    o_full, l_full = oracle.attn(q, k, v, cu, causal)
    nparts = int(rng.integers(2, 9))
    cuts = np.sort(rng.choice(np.arange(1, T), size=nparts - 1, replace=False))
    bounds = np.concatenate([[0], cuts, [T]])
    order = rng.permutation(nparts)
    acc_o = np.zeros((T, Hq, d))
    acc_l = np.full((T, Hq), -np.inf)
    for p in order:
        po, pl = oracle.attn(q, k, v, cu, causal, kv_range=(int(bounds[p]), int(bounds[p + 1])))
        acc_o, acc_l = oracle.lse_merge(acc_o, acc_l, po, pl)
    assert np.max(np.abs(acc_o - o_full)) < 1e-12
    assert np.max(np.abs(acc_l - l_full)) < 1e-12


def test_merge_identity_and_empty():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((6, 3))
    l = rng.standard_normal(6)
    ninf = np.full(6, -np.inf)
    zero = np.zeros((6, 3))
    mo, ml = oracle.lse_merge(o, l, zero, ninf)
    assert np.array_equal(ml, l) and np.max(np.abs(mo - o)) < 1e-15
    mo, ml = oracle.lse_merge(zero, ninf, o, l)
    assert np.array_equal(ml, l) and np.max(np.abs(mo - o)) < 1e-15
    mo, ml = oracle.lse_merge(zero, ninf, zero, ninf)
    assert np.all(ml == -np.inf) and np.all(mo == 0)
    # Two equal partials: LSE grows by ln 2, O unchanged.
    mo, ml = oracle.lse_merge(o, l, o, l)
    assert np.max(np.abs(ml - (l + math.log(2)))) < 1e-14
    assert np.max(np.abs(mo - o)) < 1e-14


def test_partial_without_valid_keys():
    rng = np.random.default_rng(9)
    T, d = 30, 4
    q = rng.standard_normal((T, 1, d))
    k = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    # causal, keys [20, 30) for rows < 20: nothing valid.
    o, lse = oracle.attn(q, k, v, np.array([0, T]), True, kv_range=(20, 30))
    assert np.all(lse[:20] == -np.inf) and np.all(o[:20] == 0)
    assert np.all(np.isfinite(lse[20:]))


@pytest.mark.parametrize("causal", [True, False])
def test_document_isolation(causal):
    rng = np.random.default_rng(21)
    T, Hq, Hkv, d = 64, 4, 1, 8
    cu = np.array([0, 13, 40, 41, 64], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    o1, l1 = oracle.attn(q, k, v, cu, causal)
    a, b = 13, 40
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[a:b] += 3.0 * rng.standard_normal((b - a, Hq, d))
    k2[a:b] *= -1.5
    v2[a:b] += 10.0
    o2, l2 = oracle.attn(q2, k2, v2, cu, causal)
    mask = np.ones(T, dtype=bool)
    mask[a:b] = False
    assert np.array_equal(o1[mask], o2[mask]) and np.array_equal(l1[mask], l2[mask])
    assert not np.array_equal(o1[a:b], o2[a:b])


def test_row_subset_and_dtypes():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    T, Hq, Hkv, d = 70, 2, 2, 8
    cu = np.array([0, 30, 70], dtype=np.int32)
    qf = rng.standard_normal((T, Hq, d)).astype(np.float32)
    kf = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    vf = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    o64, l64 = oracle.attn(qf.astype(np.float64), kf.astype(np.float64), vf.astype(np.float64), cu, True)
    o32, l32 = oracle.attn(qf, kf, vf, cu, True)
    assert np.array_equal(o64, o32) and np.array_equal(l64, l32)
    rows = np.array([69, 0, 31, 29, 30])
    orow, lrow = oracle.attn(qf, kf, vf, cu, True, rows=rows)
    assert np.array_equal(orow, o32[rows]) and np.array_equal(lrow, l32[rows])
    # bf16 bit patterns widen to the same values as their float32 copies.
    tb = [torch.from_numpy(x).to(torch.bfloat16) for x in (qf, kf, vf)]
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in tb]
    wide = [t.float().numpy() for t in tb]
    ob, lb = oracle.attn(*bits, cu, True)
    ow, lw = oracle.attn(*wide, cu, True)
    assert np.array_equal(ob, ow) and np.array_equal(lb, lw)


def test_valid_pair_counts():
    # Closed forms: causal document of length L has L(L+1)/2 pairs, non-causal L^2.
    cu = np.array([0, 100, 256], dtype=np.int32)
    assert oracle.valid_pairs(cu, True, 0, 256, 0, 256) == 100 * 101 // 2 + 156 * 157 // 2
    assert oracle.valid_pairs(cu, False, 0, 256, 0, 256) == 100 * 100 + 156 * 156
    # Sub-rectangles against brute force.
    rng = np.random.default_rng(2)
    T = 60
    cu = _rand_docs(rng, T, 6)
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    for _ in range(30):
        qa, qb = sorted(rng.integers(0, T + 1, size=2))
        ka, kb = sorted(rng.integers(0, T + 1, size=2))
        for causal in (True, False):
            brute = sum(1 for i in range(qa, qb) for j in range(ka, kb)
                        if doc[i] == doc[j] and (not causal or j <= i))
            assert oracle.valid_pairs(cu, causal, int(qa), int(qb), int(ka), int(kb)) == brute


def test_rows_only_query_layout():
    rng = np.random.default_rng(8)
    T, Hq, Hkv, d = 50, 2, 1, 8
    cu = np.array([0, 20, 50], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    rows = np.array([49, 3, 20, 19])
    o1, l1 = oracle.attn(q, k, v, cu, True, rows=rows)
    o2, l2 = oracle.attn(q[rows], k, v, cu, True, rows=rows, q_rows_only=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
