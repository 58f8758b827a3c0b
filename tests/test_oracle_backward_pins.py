"""Pins for the oracle's attention gradients: central finite differences of the
oracle's own forward (a different computation: only forward evaluations),
torch autograd of scaled_dot_product_attention in float64, and the identity
that dK summed over the keys of a document is zero (softmax rows sum to one)."""
import math

import numpy as np
import pytest

import oracle


def _loss(q, k, v, w, cu, causal):
    o, _ = oracle.attn(q, k, v, cu, causal)
    return float(np.sum(o * w))


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    rng = np.random.default_rng(1)
    T, Hq, Hkv, d = 23, 4, 2, 8
    cu = np.array([0, 9, 10, 23], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    w = rng.standard_normal((T, Hq, d))
    dq, dk, dv = oracle.attn_backward(q, k, v, w, cu, causal)
    eps = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], w, cu, causal)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], w, cu, causal)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_autograd(causal):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    T, Hq, Hkv, d = 40, 4, 2, 16
    G = Hq // Hkv
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    w = rng.standard_normal((T, Hq, d))
    dq, dk, dv = oracle.attn_backward(q, k, v, w, np.array([0, T]), causal)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(G, dim=1).permute(1, 0, 2)[None],
        tv.repeat_interleave(G, dim=1).permute(1, 0, 2)[None], is_causal=causal)
    (o[0].permute(1, 0, 2) * torch.tensor(w)).sum().backward()
    assert np.max(np.abs(tq.grad.numpy() - dq)) < 1e-10
    assert np.max(np.abs(tk.grad.numpy() - dk)) < 1e-10
    assert np.max(np.abs(tv.grad.numpy() - dv)) < 1e-10


def test_dk_sums_to_zero_per_document_and_isolation():
    rng = np.random.default_rng(3)
    T, Hq, Hkv, d = 50, 2, 1, 8
    cu = np.array([0, 17, 50], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    w = rng.standard_normal((T, Hq, d))
    for causal in (True, False):
        dq, dk, dv = oracle.attn_backward(q, k, v, w, cu, causal)
        for a, b in ((0, 17), (17, 50)):
            assert np.max(np.abs(dk[a:b].sum(axis=0))) < 1e-12
        # Output gradient of document 0 does not reach document 1.
        w2 = w.copy()
        w2[:17] = 0
        dq2, dk2, dv2 = oracle.attn_backward(q, k, v, w2, cu, causal)
        assert np.array_equal(dq2[:17], np.zeros_like(dq2[:17]))
        assert np.array_equal(dk2[:17], np.zeros_like(dk2[:17]))
        assert np.array_equal(dq2[17:], dq[17:]) and np.array_equal(dv2[17:], dv[17:])


@pytest.mark.parametrize("causal", [True, False])
def test_sampled_gradients_match_full(causal):
    """The sampled form (chosen dQ rows, chosen dK/dV keys) equals the pinned
    full gradients at those positions, bf16 inputs, GQA, several documents."""
    rng = np.random.default_rng(5)
    T, Hq, Hkv, d = 61, 6, 2, 16
    cu = np.array([0, 1, 20, 21, 61], dtype=np.int32)
    bits = lambda shape: (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q, k, v, w = bits((T, Hq, d)), bits((T, Hkv, d)), bits((T, Hkv, d)), bits((T, Hq, d))
    dq, dk, dv = oracle.attn_backward(q, k, v, w, cu, causal)
    qrows = np.array([0, 1, 5, 19, 20, 21, 40, 60])
    krows = np.array([0, 2, 19, 20, 22, 59, 60])
    sq, sk, sv = oracle.attn_backward_sampled(q, k, v, w, cu, causal, qrows, krows)
    assert np.allclose(sq, dq[qrows], rtol=1e-12, atol=1e-13)
    assert np.allclose(sk, dk[krows], rtol=1e-12, atol=1e-13)
    assert np.allclose(sv, dv[krows], rtol=1e-12, atol=1e-13)
    # Empty selections are allowed; out-of-range rows are rejected.
    e = oracle.attn_backward_sampled(q, k, v, w, cu, causal)
    assert e[0].shape == (0, Hq, d) and e[1].shape == (0, Hkv, d)
    with pytest.raises(ValueError):
        oracle.attn_backward_sampled(q, k, v, w, cu, causal, qrows=[T])
