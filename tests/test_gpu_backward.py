"""GPU parity of the backward (sp_packed_attention_backward through the C-ABI)
against the fp64 oracle gradients.

Small cases (the oracle computes every gradient): every element must lie
within a worst-case rounding envelope, and each tensor's relative Frobenius
error must stay below 1e-2.

  Envelope. The kernels round P and dS = P (dP - D) to bf16 before the tensor
  cores read them (relative error <= 2^-9 each), compute D = dO . O from the
  bf16 forward output (|error| <= 2^-9 sum_c |dO_c O_c|), and round the
  outputs to bf16 (2^-9 relative); every other step is fp32 on exact bf16
  inputs. With w_ij = |dS_ij| + P_ij (|dP_ij| + |D_i| + A_i), A_i = sum_c |dO_ic O_ic|:
    |error dQ_i| <= 2^-9 * 3 * scale sum_j w_ij |k_j| + 2^-9 |dQ_i|
    |error dK_j| <= 2^-9 * 3 * scale sum_i w_ij |q_i| + 2^-9 |dK_j|
    |error dV_j| <= 2^-9 * sum_i P_ij |dO_i|          + 2^-9 |dV_j|
  The test allows 2^-7 * M + 2^-8 |ref| (about 1.3-2x the bound). The envelope
  M is computed here in float64 from the definitions, as a bound only: the
  expected values are the oracle's.

  Frobenius. Independent roundings add in quadrature, so the relative error
  of a tensor is a few times 2^-9 / sqrt(3) ~ 1e-3; a dropped key tile or a
  wrong term moves it by far more than 1e-2.

Full-size workloads (the benchmark's launch): dQ at sampled rows and dK, dV
at sampled keys from the oracle's sampled form (rows at document, chunk and
tile edges; keys whose attending queries the oracle can afford). Every sampled
element is held to the same rounding envelope as the small cases, computed for
the sampled positions only, and each sampled tensor to the same Frobenius
bound and max|error| <= 2e-2 max|ref|; plus two identities that hold at any
size, per document and key/value head: sum_j dV_j = sum_i sum_(h in group)
dO_ih (softmax rows sum to one) and sum_j dK_j = 0 (sum_j dS_ij = 0 for every
row). The tolerances are this file's own derivation (the benchmark spec's figures
cover the forward only): the envelope above, 1e-2 relative Frobenius."""
import math

import numpy as np
import pytest

import oracle
import sequence_blockwise_gb300 as sb
from sequence_blockwise_gb300 import workloads as wl
from gpu_util import host_inputs

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
REL_MAX_SAMPLED = 2e-2


def _torch():
    import torch
    return torch


def _inputs(T, Hq, Hkv, d, seed):
    q = wl.random_normal((T, Hq, d), seed, "cuda", "bf16")
    k = wl.random_normal((T, Hkv, d), seed + 1, "cuda", "bf16")
    v = wl.random_normal((T, Hkv, d), seed + 2, "cuda", "bf16")
    do = wl.random_normal((T, Hq, d), seed + 3, "cuda", "bf16")
    return q, k, v, do


def _fwd_bwd(q, k, v, do, cu, causal, kind, P, seed=0):
    att = sb.PackedAttention(cu, causal, kind, P, q.shape[1], seed=seed)
    o, lse = att(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, do)
    sb.sp_check_device_status()
    return o, lse, dq, dk, dv


def _envelopes(q, k, v, do, cu, causal, scale):
    """Worst-case rounding envelopes (M_dq, M_dk, M_dv) in float64 on the CPU."""
    torch = _torch()
    qf, kf, vf, dof = (x.double().cpu() for x in (q, k, v, do))
    T, Hq, d = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    doc = np.searchsorted(np.asarray(cu), np.arange(T), side="right") - 1
    mask = doc[:, None] == doc[None, :]
    if causal:
        mask &= np.arange(T)[None, :] <= np.arange(T)[:, None]
    m = torch.from_numpy(mask)
    kx, vx = kf.repeat_interleave(G, 1), vf.repeat_interleave(G, 1)
    s = torch.einsum("ihc,jhc->hij", qf, kx) * scale
    p = torch.softmax(s.masked_fill(~m, float("-inf")), -1)
    o = torch.einsum("hij,jhc->ihc", p, vx)
    dp = torch.einsum("ihc,jhc->hij", dof, vx)
    D = (dof * o).sum(-1).t()
    A = (dof.abs() * o.abs()).sum(-1).t()
    ds = p * (dp - D[:, :, None])
    w = ds.abs() + p * (dp.abs() + D.abs()[:, :, None] + A[:, :, None])
    m_dq = scale * torch.einsum("hij,jhc->ihc", w, kx.abs())
    m_dk = scale * torch.einsum("hij,ihc->jhc", w, qf.abs()).reshape(T, Hkv, G, d).sum(2)
    m_dv = torch.einsum("hij,ihc->jhc", p, dof.abs()).reshape(T, Hkv, G, d).sum(2)
    return m_dq.numpy(), m_dk.numpy(), m_dv.numpy()


def _rel_fro(got, ref):
    n = float(np.linalg.norm(ref))
    return float(np.linalg.norm(got - ref)) / n if n > 0 else float(np.linalg.norm(got))


CASES = [
    # T, docs, Hq, Hkv, d, causal, kind, P
    (700, [130, 1, 269, 300], 4, 2, 128, True, sb.SP_SCHED_TASP, 5),
    (700, [130, 1, 269, 300], 4, 2, 128, False, sb.SP_SCHED_RING, 3),
    (704, [704], 2, 2, 128, True, sb.SP_SCHED_ZIGZAG, 4),
    (1000, [1, 1, 500, 498], 8, 2, 128, True, sb.SP_SCHED_TASP, 8),
    (640, [333, 307], 4, 4, 64, True, sb.SP_SCHED_RING, 2),
    (640, [333, 307], 4, 1, 64, False, sb.SP_SCHED_TASP, 3),
    (129, [129], 1, 1, 128, True, sb.SP_SCHED_RING, 1),
    (1, [1], 2, 1, 128, True, sb.SP_SCHED_RING, 1),
    (1537, [900, 637], 4, 2, 128, True, sb.SP_SCHED_TASP, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}-H{c[2]}x{c[3]}-d{c[4]}-c{int(c[5])}-k{c[6]}P{c[7]}")
def test_backward_matches_oracle(case):
    T, docs, Hq, Hkv, d, causal, kind, P = case
    cu = wl.cu_from_lengths(docs)
    q, k, v, do = _inputs(T, Hq, Hkv, d, 101 + T)
    _, _, dq, dk, dv = _fwd_bwd(q, k, v, do, cu, causal, kind, P)
    ref = oracle.attn_backward(host_inputs(q), host_inputs(k), host_inputs(v), host_inputs(do), cu,
                               causal)
    env = _envelopes(q, k, v, do, cu, causal, 1.0 / math.sqrt(d))
    for name, got, r, mm in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, env):
        g = got.double().cpu().numpy()
        err = np.abs(g - r)
        bound = 2.0 ** -7 * mm + 2.0 ** -8 * np.abs(r) + 1e-6
        worst = float(np.max(err / bound))
        fro = _rel_fro(g, r)
        print(f"{name}: max|err|={err.max():.3e} max|ref|={np.abs(r).max():.3e} "
              f"rel_fro={fro:.3e} worst err/envelope={worst:.3f}")
        assert worst <= 1.0, (name, worst)
        assert fro <= REL_FRO, (name, fro)


@pytest.mark.parametrize("inter,R,U", [(sb.SP_SCHED_RING, 2, 2), (sb.SP_SCHED_ZIGZAG, 2, 4)])
def test_backward_two_level_schedule(inter, R, U):
    """The backward of a forward run on a two-level schedule (query heads split
    over the U ranks of each group) against the oracle, same envelope."""
    T, docs, Hq, Hkv, d = 704, [300, 404], 8, 2, 128
    cu = wl.cu_from_lengths(docs)
    q, k, v, do = _inputs(T, Hq, Hkv, d, 19 + U)
    att = sb.PackedAttention(cu, True, inter, R * U, Hq, ulysses=U)
    o, lse = att(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, do)
    sb.sp_check_device_status()
    ref = oracle.attn_backward(host_inputs(q), host_inputs(k), host_inputs(v), host_inputs(do), cu, True)
    env = _envelopes(q, k, v, do, cu, True, 1.0 / math.sqrt(d))
    for name, got, r, mm in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, env):
        g = got.double().cpu().numpy()
        worst = float(np.max(np.abs(g - r) / (2.0 ** -7 * mm + 2.0 ** -8 * np.abs(r) + 1e-6)))
        assert worst <= 1.0, (name, worst)
        assert _rel_fro(g, r) <= REL_FRO, name


def test_backward_deterministic_and_schedule_invariant():
    """Two runs give identical dK and dV bits (each is summed in a fixed order)
    and dQ equal up to the rounding of its fp32 reduction order; RING and TASP
    schedules give the same dK and dV (computed over the mask) and dQ within
    rounding."""
    torch = _torch()
    T, docs, Hq, Hkv, d = 1000, [1, 1, 500, 498], 8, 2, 128
    cu = wl.cu_from_lengths(docs)
    q, k, v, do = _inputs(T, Hq, Hkv, d, 7)
    a = _fwd_bwd(q, k, v, do, cu, True, sb.SP_SCHED_TASP, 8)
    b = _fwd_bwd(q, k, v, do, cu, True, sb.SP_SCHED_TASP, 8)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    # One bf16 step of the larger value at most, where fp32 sums in another
    # order round to the other side of a bf16 midpoint.
    gap = (a[2].float() - b[2].float()).abs()
    assert bool((gap <= 2.0 ** -7 * torch.maximum(a[2].float().abs(), b[2].float().abs()) + 1e-30).all())
    c = _fwd_bwd(q, k, v, do, cu, True, sb.SP_SCHED_RING, 2)
    for x, y in zip(a[2:], c[2:]):
        assert float((x.float() - y.float()).abs().max()) <= 2e-2 * float(x.float().abs().max())


def test_backward_first_token_and_isolation():
    """Causal first token of a document attends only itself: P = 1, dS = 0, so
    dQ there is (rounding-)zero and dV of that key from that query is dO.
    A one-token document's dK is zero and its dV is the sum of its heads' dO."""
    torch = _torch()
    T, docs, Hq, Hkv, d = 300, [100, 1, 199], 4, 2, 128
    cu = wl.cu_from_lengths(docs)
    q, k, v, do = _inputs(T, Hq, Hkv, d, 3)
    _, _, dq, dk, dv = _fwd_bwd(q, k, v, do, cu, True, sb.SP_SCHED_RING, 2)
    G = Hq // Hkv
    firsts = torch.tensor(cu[:-1].astype(np.int64), device="cuda")
    assert float(dq[firsts].float().abs().max()) <= 1e-3 * float(dq.float().abs().max())
    lone = 100
    assert float(dk[lone].float().abs().max()) <= 1e-3 * float(dk.float().abs().max())
    want = do[lone].float().reshape(Hkv, G, d).sum(1)
    assert float((dv[lone].float() - want).abs().max()) <= 2.0 ** -7 * float(want.abs().max()) + 1e-3


def test_backward_argument_errors_on_device():
    torch = _torch()
    T, Hq, Hkv, d = 256, 2, 1, 128
    cu = wl.cu_from_lengths([T])
    q, k, v, do = _inputs(T, Hq, Hkv, d, 5)
    att = sb.PackedAttention(cu, True, sb.SP_SCHED_RING, 2, Hq)
    o, lse = att(q, k, v)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(sb.SpError) as e:
        sb.sp_packed_attention_backward(q, k, v, o, do, lse, torch.empty_like(q), torch.empty_like(k),
                                        torch.empty_like(v), att.cu_dev, True, att.items_dev, small)
    assert e.value.code == 3
    qf = q.float()
    with pytest.raises(sb.SpError) as e:
        sb.sp_packed_attention_backward(qf, k.float(), v.float(), o.float(), do.float(), lse,
                                        torch.empty_like(qf), torch.empty_like(k.float()),
                                        torch.empty_like(v.float()), att.cu_dev, True, att.items_dev,
                                        torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 2


# ---------------------------------------------------------------- full size

BUDGET = 3.0e10  # oracle work per workload, in (query, key) pairs x query heads x d


def _chunk_bounds(w):
    if w.kind == sb.SP_SCHED_ZIGZAG:
        c = w.T // (2 * w.P)
        return [i * c for i in range(2 * w.P + 1)]
    base, extra = divmod(w.T, w.P)
    out, s = [0], 0
    for r in range(w.P):
        s += base + (1 if r < extra else 0)
        out.append(s)
    return out


def _pick_samples(w, cu):
    """dQ rows and dK/dV keys whose oracle cost fits the budget. A dQ row costs
    its valid keys; a set of keys costs the queries attending them (each with
    its own LSE and D over its keys): for causal masks the cheap keys sit at
    the end of a document, for full masks only short documents are cheap."""
    rng = np.random.default_rng(w.seed + 11)
    cu = np.asarray(cu, dtype=np.int64)
    unit = float(w.Hq * w.d)
    edges = set()
    for b in list(cu) + _chunk_bounds(w):
        for dlt in (-129, -128, -2, -1, 0, 1, 127, 128):
            if 0 <= b + dlt < w.T:
                edges.add(int(b + dlt))
    cand = np.array(sorted(edges | set(int(x) for x in rng.integers(0, w.T, 2048))), dtype=np.int64)
    doc = np.searchsorted(cu, cand, side="right") - 1
    keys = (cand - cu[doc] + 1) if w.causal else (cu[doc + 1] - cu[doc])
    per_row = keys.astype(np.float64) * unit
    qrows, spent = [], 0.0
    for i in np.argsort(per_row, kind="stable"):
        if spent + per_row[i] > BUDGET / 2 or len(qrows) >= 128:
            break
        qrows.append(int(cand[i]))
        spent += per_row[i]
    krows, spent = [], 0.0
    lens = np.diff(cu)
    for di in np.argsort(lens, kind="stable"):
        a, b = int(cu[di]), int(cu[di + 1])
        n = b - a
        W = min(n, 160) if w.causal else n
        cost = lambda W: (W * n if w.causal else n * n) * unit
        while w.causal and W > 1 and spent + cost(W) > BUDGET / 2:
            W //= 2
        if spent + cost(W) > BUDGET / 2:
            continue
        lo = b - W
        picks = {b - 1, lo} | {x for x in (b - 129, b - 128, b - 127) if lo <= x < b}
        picks |= set(int(x) for x in rng.integers(lo, b, min(8, W)))
        krows.extend(sorted(picks))
        spent += cost(W)
        if len(krows) >= 128:
            break
    return np.array(sorted(qrows), dtype=np.int64), np.array(sorted(set(krows)), dtype=np.int64)


def _row_stats(qr, kd, vd, dor, scale, valid):
    """Full-row quantities of query rows qr, dor [r, Hkv, G, d] (query head
    g G + x) over a document's keys kd, vd [n, Hkv, d], valid [r, n] bool:
    P, dP [r, Hkv, G, n] and D, A [r, Hkv, G], in float64."""
    torch = _torch()
    sc = torch.einsum("rgxc,ngc->rgxn", qr, kd) * scale
    sc = sc.masked_fill(~valid[:, None, None, :], float("-inf"))
    p = torch.softmax(sc, -1)
    o = torch.einsum("rgxn,ngc->rgxc", p, vd)
    D = (dor * o).sum(-1)
    A = (dor.abs() * o.abs()).sum(-1)
    dp = torch.einsum("rgxc,ngc->rgxn", dor, vd)
    return p, dp, D, A


def _weights(p, dp, D, A):
    ds = p * (dp - D[..., None])
    return ds.abs() + p * (dp.abs() + D.abs()[..., None] + A[..., None])


def _sampled_envelopes(q, k, v, do, cu, causal, scale, qrows, krows, block=8):
    """The rounding envelopes of _envelopes at the sampled dQ rows and dK/dV
    keys only, in float64 (on the device, in blocks of `block` query rows)."""
    torch = _torch()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    cu = np.asarray(cu, dtype=np.int64)
    dev = q.device
    grp = lambda x: x.double().reshape(x.shape[0], Hkv, G, d)
    m_dq = np.zeros((len(qrows), Hq, d))
    m_dk = np.zeros((len(krows), Hkv, d))
    m_dv = np.zeros((len(krows), Hkv, d))
    qdoc = np.searchsorted(cu, qrows, side="right") - 1
    kdoc = np.searchsorted(cu, krows, side="right") - 1
    for di in np.unique(np.concatenate([qdoc, kdoc])):
        a, b = int(cu[di]), int(cu[di + 1])
        kd, vd = k[a:b].double(), v[a:b].double()
        keys = torch.arange(a, b, device=dev)
        for n_i in np.nonzero(qdoc == di)[0]:
            i = int(qrows[n_i])
            valid = (keys <= i)[None, :] if causal else torch.ones((1, b - a), dtype=torch.bool, device=dev)
            p, dp, D, A = _row_stats(grp(q[i:i + 1]), kd, vd, grp(do[i:i + 1]), scale, valid)
            w = _weights(p, dp, D, A)
            m_dq[n_i] = (scale * torch.einsum("rgxn,ngc->rgxc", w, kd.abs())).reshape(Hq, d).cpu().numpy()
        sel = np.nonzero(kdoc == di)[0]
        if len(sel) == 0:
            continue
        cols = torch.from_numpy(krows[sel] - a).to(dev)
        r0 = int(krows[sel].min()) if causal else a  # the first query attending these keys
        acc_k = torch.zeros((len(sel), Hkv, d), dtype=torch.float64, device=dev)
        acc_v = torch.zeros((len(sel), Hkv, d), dtype=torch.float64, device=dev)
        for s0 in range(r0, b, block):
            s1 = min(b, s0 + block)
            rows = torch.arange(s0, s1, device=dev)
            valid = (keys[None, :] <= rows[:, None]) if causal else \
                torch.ones((s1 - s0, b - a), dtype=torch.bool, device=dev)
            qr, dor = grp(q[s0:s1]), grp(do[s0:s1])
            p, dp, D, A = _row_stats(qr, kd, vd, dor, scale, valid)
            p, dp = p[..., cols], dp[..., cols]
            w = _weights(p, dp, D, A)
            acc_k += scale * torch.einsum("rgxk,rgxc->kgc", w, qr.abs())
            acc_v += torch.einsum("rgxk,rgxc->kgc", p, dor.abs())
        m_dk[sel] = acc_k.cpu().numpy()
        m_dv[sel] = acc_v.cpu().numpy()
    return m_dq, m_dk, m_dv


BF16_WORKLOADS = [w for w in wl.WORKLOADS if w.dtype == "bf16"]


@pytest.mark.parametrize("w", BF16_WORKLOADS, ids=lambda w: w.name)
def test_backward_workload_parity(w):
    torch = _torch()
    cu = wl.cu_seqlens(w)
    q, k, v = wl.make_qkv(w, "cuda")
    do = wl.random_normal((w.T, w.Hq, w.d), w.seed + 99, "cuda", "bf16")
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed)
    o, lse = att(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, do)
    sb.sp_check_device_status()

    G = w.Hq // w.Hkv
    # Identities per document and key/value head.
    for di in range(len(cu) - 1):
        a, b = int(cu[di]), int(cu[di + 1])
        sdv = dv[a:b].double().sum(0)
        sdo = do[a:b].double().reshape(b - a, w.Hkv, G, w.d).sum((0, 2))
        scale_v = dv[a:b].double().abs().sum(0).max().item() + 1e-30
        assert float((sdv - sdo).abs().max()) <= 1e-2 * scale_v, (di, "sum dV")
        sdk = dk[a:b].double().sum(0)
        scale_k = dk[a:b].double().abs().sum(0).max().item() + 1e-30
        assert float(sdk.abs().max()) <= 1e-2 * scale_k, (di, "sum dK")

    qrows, krows = _pick_samples(w, cu)
    assert len(qrows) > 0
    # A full mask over one 64K document has no affordable key sample: its dK
    # and dV rest on the identities above and the small full-mask cases.
    assert len(krows) > 0 or not w.causal
    rq, rk, rv = oracle.attn_backward_sampled(host_inputs(q), host_inputs(k), host_inputs(v),
                                              host_inputs(do), cu, w.causal, qrows, krows)
    qi = torch.from_numpy(qrows).cuda()
    ki = torch.from_numpy(krows).cuda()
    env = _sampled_envelopes(q, k, v, do, cu, w.causal, 1.0 / math.sqrt(w.d), qrows, krows)
    for name, got, ref, mm in (("dq", dq[qi], rq, env[0]), ("dk", dk[ki], rk, env[1]),
                               ("dv", dv[ki], rv, env[2])):
        if ref.shape[0] == 0:
            continue
        g = got.double().cpu().numpy()
        err = float(np.abs(g - ref).max())
        mx = float(np.abs(ref).max())
        fro = _rel_fro(g, ref)
        worst = float(np.max(np.abs(g - ref) / (2.0 ** -7 * mm + 2.0 ** -8 * np.abs(ref) + 1e-6)))
        print(f"{w.name} {name}: {g.shape[0]} samples max|err|={err:.3e} max|ref|={mx:.3e} "
              f"rel_fro={fro:.3e} worst err/envelope={worst:.3f}")
        assert worst <= 1.0, (name, worst)
        assert err <= REL_MAX_SAMPLED * mx and fro <= REL_FRO, (name, err, mx, fro)
