"""Pins of the backward oracle against things other than its own formulas.

(1) Central finite differences of the forward oracle: the gradient of
    L = sum(O * G) in each input entry, with no use of the backward formulas.
(2) torch.autograd through a float64 torch attention (a foreign library's
    differentiation), including causal and window masks.
(3) Invariants the true gradient has: shifting every key by one vector leaves
    every softmax row unchanged, so sum_j dK_j = 0; shifting every value by c
    shifts every live O row by c, so sum_j dV_j = sum of dO over rows that see
    a key; homogeneity of the scores gives sum q.dQ = sum k.dK; and the
    identity rowsum(P * dP) = rowsum(dO * O) the kernels rely on.
(4) Planted mistakes in a copy of the oracle fail pin (1).
"""

import numpy as np
import pytest

from oracle import (MASK_CAUSAL, MASK_NONE, MASK_WINDOW, attention_backward, attention_backward_grouped,
                    attention_grouped, attention_probs, attention_three_pass)

MASKS = [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 2, 1), (MASK_WINDOW, 0, 0)]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, g, scale, mk, wl, wr, q_offset=0, fwd=attention_three_pass):
    o, _ = fwd(q, k, v, scale, mk, wl, wr, q_offset=q_offset)
    return float((o * g).sum())


def _finite_diff(q, k, v, g, scale, mk, wl, wr, q_offset=0, fwd=attention_three_pass, h=1e-6):
    grads = []
    for which in range(3):
        x = [q.copy(), k.copy(), v.copy()]
        gr = np.zeros_like(x[which])
        for idx in np.ndindex(x[which].shape):
            saved = x[which][idx]
            x[which][idx] = saved + h
            lp = _loss(*x, g, scale, mk, wl, wr, q_offset, fwd)
            x[which][idx] = saved - h
            lm = _loss(*x, g, scale, mk, wl, wr, q_offset, fwd)
            x[which][idx] = saved
            gr[idx] = (lp - lm) / (2 * h)
        grads.append(gr)
    return grads


@pytest.mark.parametrize("mk,wl,wr", MASKS)
@pytest.mark.parametrize("nq,nk,q_offset", [(5, 5, 0), (3, 6, 3)])
def test_matches_finite_differences(mk, wl, wr, nq, nk, q_offset):
    B, H, D = 1, 2, 3
    q = _rand((B, H, nq, D), 1)
    k = _rand((B, H, nk, D), 2)
    v = _rand((B, H, nk, D), 3)
    g = _rand((B, H, nq, D), 4)
    scale = 0.7
    got = attention_backward(q, k, v, g, scale, mk, wl, wr, q_offset)
    want = _finite_diff(q, k, v, g, scale, mk, wl, wr, q_offset)
    for a, b, name in zip(got, want, ("dQ", "dK", "dV")):
        assert np.allclose(a, b, atol=2e-7, rtol=0), (name, np.abs(a - b).max())


def test_grouped_matches_finite_differences():
    B, H, Hkv, N, D = 1, 4, 2, 4, 3
    q = _rand((B, H, N, D), 5)
    k = _rand((B, Hkv, N, D), 6)
    v = _rand((B, Hkv, N, D), 7)
    g = _rand((B, H, N, D), 8)
    got = attention_backward_grouped(q, k, v, g, 0.5, MASK_CAUSAL)
    want = _finite_diff(q, k, v, g, 0.5, MASK_CAUSAL, -1, -1, fwd=attention_grouped)
    for a, b in zip(got, want):
        assert np.allclose(a, b, atol=2e-7, rtol=0)


@pytest.mark.parametrize("mk,wl,wr", [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 16, 3)])
def test_matches_torch_autograd_float64(mk, wl, wr):
    torch = pytest.importorskip("torch")
    from oracle import allowed_mask
    B, H, N, D = 2, 3, 40, 16
    q, k, v, g = (_rand((B, H, N, D), 10 + i) for i in range(4))
    scale = 0.25
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    ok = torch.tensor(allowed_mask(N, N, mk, wl, wr))
    p = torch.softmax(s.masked_fill(~ok, float("-inf")), dim=-1)
    (p @ tv).backward(torch.tensor(g))
    got = attention_backward(q, k, v, g, scale, mk, wl, wr)
    for a, t in zip(got, (tq, tk, tv)):
        assert np.allclose(a, t.grad.numpy(), atol=1e-12, rtol=1e-10)


@pytest.mark.parametrize("mk,wl,wr", MASKS)
def test_invariants(mk, wl, wr):
    B, H, N, D = 2, 2, 33, 8
    q, k, v, g = (_rand((B, H, N, D), 20 + i) for i in range(4))
    scale = 0.4
    dq, dk, dv = attention_backward(q, k, v, g, scale, mk, wl, wr)
    assert np.allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    o, lse = attention_three_pass(q, k, v, scale, mk, wl, wr)
    live = np.isfinite(lse)[..., None]
    assert np.allclose(dv.sum(axis=2), (g * live).sum(axis=2), atol=1e-12)
    assert np.allclose((q * dq).sum(axis=(2, 3)), (k * dk).sum(axis=(2, 3)), atol=1e-12)
    for b in range(B):
        for h in range(H):
            p = attention_probs(q[b, h], k[b, h], scale, mk, wl, wr)
            dp = g[b, h] @ v[b, h].T
            assert np.allclose((p * dp).sum(axis=1), (g[b, h] * o[b, h]).sum(axis=1), atol=1e-12)


def test_rows_that_see_no_key_have_zero_gradient():
    # window (0, 0) with q_offset beyond the keys: queries 0..2 sit at 5..7, keys are 0..4
    q, k, v, g = (_rand((1, 1, 3 if i in (0, 3) else 5, 4), 30 + i) for i in range(4))
    dq, dk, dv = attention_backward(q, k, v, g, 1.0, MASK_WINDOW, 0, 0, q_offset=5)
    assert not dq.any() and not dk.any() and not dv.any()


def _broken(q, k, v, do, scale, mk, wl, wr, q_offset, mistake):
    dq, dk, dv = (np.zeros_like(t) for t in (q, k, v))
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            p = attention_probs(q[b, h], k[b, h], scale, mk, wl, wr, q_offset)
            dp = do[b, h] @ v[b, h].T
            if mistake == "no_rowsum":
                ds = p * dp
            else:
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dv[b, h] = (p.T if mistake != "dv_untransposed" else p) @ do[b, h]
            dq[b, h] = (scale if mistake != "unscaled" else 1.0) * (ds @ k[b, h])
            dk[b, h] = scale * ((ds.T if mistake != "dk_from_dq_side" else ds) @ q[b, h])
    return dq, dk, dv


@pytest.mark.parametrize("mistake", ["no_rowsum", "unscaled", "dv_untransposed", "dk_from_dq_side"])
def test_planted_mistakes_fail_finite_differences(mistake):
    B, H, N, D = 1, 1, 4, 3
    q, k, v, g = (_rand((B, H, N, D), 40 + i) for i in range(4))
    scale = 0.8
    want = _finite_diff(q, k, v, g, scale, MASK_CAUSAL, -1, -1)
    got = _broken(q, k, v, g, scale, MASK_CAUSAL, -1, -1, 0, mistake)
    assert any(not np.allclose(a, b, atol=2e-7) for a, b in zip(got, want))


@pytest.mark.parametrize("mk,wl,wr", MASKS)
def test_sampled_backward_equals_full(mk, wl, wr):
    from oracle import attention_backward_sampled
    N, D = 70, 8
    q, k, v, g = (_rand((1, 1, N, D), 50 + i) for i in range(4))
    dq, dk, dv = attention_backward(q, k, v, g, 0.6, mk, wl, wr)
    rows, keys = [0, 5, 33, 69], [1, 2, 40, 69]
    sq, sk, sv = attention_backward_sampled(q[0, 0], k[0, 0], v[0, 0], g[0, 0], 0.6, mk, wl, wr, rows, keys,
                                            row_chunk=16)
    assert np.allclose(sq, dq[0, 0, rows], atol=1e-13)
    assert np.allclose(sk, dk[0, 0, keys], atol=1e-13)
    assert np.allclose(sv, dv[0, 0, keys], atol=1e-13)
