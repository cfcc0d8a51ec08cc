"""Pins for the float64 oracle (CPU only).

Each check compares the oracle with something other than itself: hand-derived
exact values, exact-arithmetic brute force (mpmath), closed forms, invariants
of softmax attention, and a foreign library (torch's CPU SDPA).  The last
group plants mistakes in the oracle and checks that the pins catch them.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import (MASK_CAUSAL, MASK_NONE, MASK_WINDOW, allowed_mask, attention_bruteforce,
                    attention_online, attention_probs, attention_three_pass, unmasked_pairs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")

MASKS = [
    (MASK_NONE, -1, -1),
    (MASK_CAUSAL, -1, -1),
    (MASK_WINDOW, 3, 0),
    (MASK_WINDOW, 0, 2),
    (MASK_WINDOW, 2, 5),
    (MASK_WINDOW, -1, 1),
    (MASK_WINDOW, 4, -1),
]


def _parse(x):
    if isinstance(x, str) and x.startswith("ln:"):
        return math.log(float(Fraction(x[3:])))
    return float(Fraction(x))


def _arr(nested):
    return np.array([[[[_parse(x) for x in row] for row in h] for h in b] for b in nested])


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _hand_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _check_hand(fn):
    """Run every hand case through fn(q,k,v,scale,mask,wl,wr) -> (O, LSE)."""
    for case in _hand_cases():
        q, k, v = _arr(case["q"]), _arr(case["k"]), _arr(case["v"])
        scale = _parse(case["scale"])
        for e in case["expect"]:
            o, lse = fn(q, k, v, scale, e["mask"], e["win_l"], e["win_r"])
            want_o = np.array([[_parse(x) for x in row] for row in e["o"]])
            want_lse = np.array([math.log(_parse(x)) for x in e["lse_exp"]])
            np.testing.assert_allclose(np.asarray(o)[0, 0], want_o, rtol=0, atol=1e-14,
                                       err_msg=f"{case['name']} mask={e['mask']},{e['win_l']},{e['win_r']}")
            np.testing.assert_allclose(np.asarray(lse)[0, 0], want_lse, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- hand values

def test_hand_cases_three_pass():
    _check_hand(lambda q, k, v, s, m, wl, wr: attention_three_pass(q, k, v, s, m, wl, wr))


def test_hand_cases_online():
    for bk in (1, 2, 3, 64):
        _check_hand(lambda q, k, v, s, m, wl, wr: attention_online(q, k, v, s, m, wl, wr, block_k=bk))


def test_hand_cases_bruteforce():
    _check_hand(lambda q, k, v, s, m, wl, wr: attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), s, m, wl, wr))


# ------------------------------------------------- exact-arithmetic brute force

def _mp_attention(q, k, v, scale, mask, wl, wr, q_offset=0):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    nq, nk = q.shape[0], k.shape[0]
    o = np.zeros((nq, v.shape[1]))
    lse = np.zeros(nq)
    for i in range(nq):
        pos = i + q_offset
        js = [j for j in range(nk)
              if (mask != MASK_CAUSAL or j <= pos)
              and (mask != MASK_WINDOW or ((wl < 0 or j >= pos - wl) and (wr < 0 or j <= pos + wr)))]
        s = {j: mp.mpf(scale) * mp.fsum(mp.mpf(q[i, d]) * mp.mpf(k[j, d]) for d in range(q.shape[1]))
             for j in js}
        z = mp.fsum(mp.e ** s[j] for j in js)
        for d in range(v.shape[1]):
            o[i, d] = float(mp.fsum(mp.e ** s[j] * mp.mpf(v[j, d]) for j in js) / z)
        lse[i] = float(mp.log(z))
    return o, lse


@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_three_pass_vs_exact(mask, wl, wr):
    for seed, (n, d, sc) in enumerate([(7, 3, 0.7), (9, 5, 1.3), (5, 2, 12.0)]):
        q, k, v = _rand((1, 1, n, d), seed), _rand((1, 1, n, d), seed + 10), _rand((1, 1, n, d), seed + 20)
        o, lse = attention_three_pass(q, k, v, sc, mask, wl, wr)
        eo, else_ = _mp_attention(q[0, 0], k[0, 0], v[0, 0], sc, mask, wl, wr)
        np.testing.assert_allclose(o[0, 0], eo, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], else_, rtol=1e-14, atol=1e-13)


def test_three_pass_vs_exact_q_offset():
    q, k, v = _rand((1, 1, 3, 4), 1), _rand((1, 1, 8, 4), 2), _rand((1, 1, 8, 4), 3)
    for mask, wl, wr in MASKS:
        o, lse = attention_three_pass(q, k, v, 0.5, mask, wl, wr, q_offset=5)
        eo, else_ = _mp_attention(q[0, 0], k[0, 0], v[0, 0], 0.5, mask, wl, wr, q_offset=5)
        np.testing.assert_allclose(o[0, 0], eo, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], else_, rtol=1e-14, atol=1e-13)


def test_large_scores_stay_finite_and_exact():
    """Scores in the thousands: the max subtraction must keep everything finite."""
    q, k, v = _rand((1, 1, 6, 4), 5, 30.0), _rand((1, 1, 6, 4), 6, 30.0), _rand((1, 1, 6, 4), 7)
    for mask, wl, wr in MASKS[:3]:
        o, lse = attention_three_pass(q, k, v, 1.0, mask, wl, wr)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        eo, else_ = _mp_attention(q[0, 0], k[0, 0], v[0, 0], 1.0, mask, wl, wr)
        np.testing.assert_allclose(o[0, 0], eo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, 0], else_, rtol=1e-13)


def test_bruteforce_vs_three_pass():
    q, k, v = _rand((2, 2, 11, 4), 1), _rand((2, 2, 11, 4), 2), _rand((2, 2, 11, 3), 3)
    for mask, wl, wr in MASKS:
        o, lse = attention_three_pass(q, k, v, 0.4, mask, wl, wr)
        bo, blse = attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.4, mask, wl, wr)
        np.testing.assert_allclose(o, np.array(bo), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(blse), rtol=0, atol=1e-13)


# ------------------------------------------ the pages' own identity (online)

@pytest.mark.parametrize("mask,wl,wr", MASKS + [(MASK_WINDOW, 17, 0), (MASK_WINDOW, 40, 33)])
def test_online_recurrence_equals_three_pass(mask, wl, wr):
    n = 203
    q, k, v = _rand((1, 2, n, 16), 11), _rand((1, 2, n, 16), 12), _rand((1, 2, n, 16), 13)
    ref_o, ref_lse = attention_three_pass(q, k, v, 0.9, mask, wl, wr, row_chunk=64)
    for bk in (1, 7, 64, n):
        o, lse = attention_online(q, k, v, 0.9, mask, wl, wr, block_k=bk)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_row_chunking_is_invisible():
    q, k, v = _rand((1, 1, 300, 8), 1), _rand((1, 1, 300, 8), 2), _rand((1, 1, 300, 8), 3)
    a = attention_three_pass(q, k, v, 0.3, MASK_WINDOW, 20, 3, row_chunk=1024)
    b = attention_three_pass(q, k, v, 0.3, MASK_WINDOW, 20, 3, row_chunk=17)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ----------------------------------------------------------------- invariants

@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_probs_rows_sum_to_one_and_masked_are_zero(mask, wl, wr):
    q, k = _rand((13, 6), 1), _rand((13, 6), 2)
    p = attention_probs(q, k, 0.8, mask, wl, wr)
    ok = allowed_mask(13, 13, mask, wl, wr)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (p[~ok] == 0.0).all()
    assert (p[ok] > 0.0).all()


@pytest.mark.parametrize("c", [0.0, 1.5, -3.0])
@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_constant_v_gives_constant_o(c, mask, wl, wr):
    q, k = _rand((1, 2, 37, 8), 3), _rand((1, 2, 37, 8), 4)
    v = np.full((1, 2, 37, 8), c)
    o, _ = attention_three_pass(q, k, v, 0.5, mask, wl, wr)
    np.testing.assert_allclose(o, c, rtol=0, atol=1e-14)


def test_single_key():
    q, k, v = _rand((2, 3, 1, 5), 1), _rand((2, 3, 1, 5), 2), _rand((2, 3, 1, 5), 3)
    for mask, wl, wr in MASKS:
        o, lse = attention_three_pass(q, k, v, 0.7, mask, wl, wr)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(lse, 0.7 * np.einsum("bhnd,bhnd->bhn", q, k), rtol=0, atol=1e-15)


def test_causal_row_zero_sees_only_key_zero():
    q, k, v = _rand((1, 2, 50, 8), 1), _rand((1, 2, 50, 8), 2), _rand((1, 2, 50, 8), 3)
    o, lse = attention_three_pass(q, k, v, 0.25, MASK_CAUSAL)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.25 * (q[:, :, 0] * k[:, :, 0]).sum(-1), rtol=0, atol=1e-15)


@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_zero_scale_is_mean_of_visible_values(mask, wl, wr):
    n = 23
    q, k, v = _rand((1, 1, n, 4), 1), _rand((1, 1, n, 4), 2), _rand((1, 1, n, 4), 3)
    o, lse = attention_three_pass(q, k, v, 0.0, mask, wl, wr)
    ok = allowed_mask(n, n, mask, wl, wr)
    for i in range(n):
        sel = v[0, 0][ok[i]]
        np.testing.assert_allclose(o[0, 0, i], sel.mean(axis=0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(len(sel))) < 1e-14


def test_mask_reductions():
    n = 31
    q, k, v = _rand((1, 2, n, 8), 1), _rand((1, 2, n, 8), 2), _rand((1, 2, n, 8), 3)
    full = attention_three_pass(q, k, v, 0.6, MASK_NONE)
    causal = attention_three_pass(q, k, v, 0.6, MASK_CAUSAL)
    for got, want in [
        (attention_three_pass(q, k, v, 0.6, MASK_WINDOW, -1, -1), full),
        (attention_three_pass(q, k, v, 0.6, MASK_WINDOW, n - 1, n - 1), full),
        (attention_three_pass(q, k, v, 0.6, MASK_WINDOW, 5 * n, -1), full),
        (attention_three_pass(q, k, v, 0.6, MASK_WINDOW, -1, 0), causal),
        (attention_three_pass(q, k, v, 0.6, MASK_WINDOW, n - 1, 0), causal),
    ]:
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1], want[1])
    o, _ = attention_three_pass(q, k, v, 0.6, MASK_WINDOW, 0, 0)
    np.testing.assert_array_equal(o, v)


def test_window_band_edges_exact():
    """Row i of window (wl, wr) equals full attention over keys [i-wl, i+wr] only."""
    n, wl, wr = 40, 6, 3
    q, k, v = _rand((1, 1, n, 4), 1), _rand((1, 1, n, 4), 2), _rand((1, 1, n, 4), 3)
    o, lse = attention_three_pass(q, k, v, 1.1, MASK_WINDOW, wl, wr)
    for i in range(n):
        lo, hi = max(0, i - wl), min(n - 1, i + wr)
        so, slse = attention_three_pass(q[:, :, i:i + 1], k[:, :, lo:hi + 1], v[:, :, lo:hi + 1], 1.1)
        np.testing.assert_allclose(o[0, 0, i], so[0, 0, 0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[0, 0, i], slse[0, 0, 0], rtol=0, atol=1e-14)


def test_permutation_equivariance():
    n = 29
    q, k, v = _rand((1, 1, n, 8), 1), _rand((1, 1, n, 8), 2), _rand((1, 1, n, 8), 3)
    o, lse = attention_three_pass(q, k, v, 0.5, MASK_NONE)
    perm = np.random.default_rng(0).permutation(n)
    o2, lse2 = attention_three_pass(q, k[:, :, perm], v[:, :, perm], 0.5, MASK_NONE)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)
    o3, lse3 = attention_three_pass(q[:, :, perm], k, v, 0.5, MASK_NONE)
    np.testing.assert_allclose(o3, o[:, :, perm], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse3, lse[:, :, perm], rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_per_row_shift_invariance(mask, wl, wr):
    """Adding u to every key adds scale*q_i.u to row i of S: O is unchanged and
    LSE_i moves by exactly that amount (softmax is over keys, per query row)."""
    n = 21
    q, k, v = _rand((1, 1, n, 6), 1), _rand((1, 1, n, 6), 2), _rand((1, 1, n, 6), 3)
    u = _rand((6,), 9, 2.0)
    o, lse = attention_three_pass(q, k, v, 0.7, mask, wl, wr)
    o2, lse2 = attention_three_pass(q, k + u, v, 0.7, mask, wl, wr)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse + 0.7 * (q @ u), rtol=0, atol=1e-12)


# ------------------------------------------------------------ foreign library

@pytest.mark.parametrize("mask,wl,wr", MASKS)
def test_against_torch_sdpa_float64(mask, wl, wr):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    n = 45
    q, k, v = _rand((2, 3, n, 16), 1), _rand((2, 3, n, 16), 2), _rand((2, 3, n, 16), 3)
    o, lse = attention_three_pass(q, k, v, 0.3, mask, wl, wr)
    ok = torch.from_numpy(allowed_mask(n, n, mask, wl, wr))
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    to = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=ok, scale=0.3)
    np.testing.assert_allclose(o, to.numpy(), rtol=0, atol=1e-12)
    s = (tq @ tk.transpose(-1, -2)) * 0.3
    tlse = torch.logsumexp(s.masked_fill(~ok, float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, tlse.numpy(), rtol=0, atol=1e-12)


# -------------------------------------------------------------- pair counting

def test_unmasked_pairs_closed_forms():
    for n in (1, 2, 7, 128, 1000):
        assert unmasked_pairs(n, MASK_NONE) == n * n
        assert unmasked_pairs(n, MASK_CAUSAL) == n * (n + 1) // 2
        for wl in (0, 1, 5, 300):
            assert unmasked_pairs(n, MASK_WINDOW, wl, 0) == sum(min(i, wl) + 1 for i in range(n))
    # the 16k sliding-window workload: rows i < 1024 see i+1 keys, the rest 1025
    assert unmasked_pairs(16384, MASK_WINDOW, 1024, 0) == sum(range(1, 1025)) + (16384 - 1024) * 1025


# ------------------------------------------------- planted mistakes get caught

def _planted(kind):
    def fn(q, k, v, s, m, wl, wr):
        if kind == "transposed":
            return attention_three_pass(k, q, v, s, m, wl, wr)
        if kind == "no_scale":
            return attention_three_pass(q, k, v, 1.0, m, wl, wr)
        if kind == "causal_off_by_one":
            if m == MASK_CAUSAL:
                return attention_three_pass(q, k, v, s, MASK_WINDOW, -1, 1)
            return attention_three_pass(q, k, v, s, m, wl, wr)
        if kind == "window_exclusive":
            if m == MASK_WINDOW:
                return attention_three_pass(q, k, v, s, m, max(wl - 1, 0) if wl > 0 else wl, wr)
            return attention_three_pass(q, k, v, s, m, wl, wr)
        if kind == "v_transposed":
            vt = np.swapaxes(v, -1, -2).copy() if v.shape[-1] == v.shape[-2] else v[..., ::-1, :]
            return attention_three_pass(q, k, vt, s, m, wl, wr)
        raise AssertionError(kind)
    return fn


@pytest.mark.parametrize("kind", ["transposed", "no_scale", "causal_off_by_one", "window_exclusive", "v_transposed"])
def test_pins_catch_planted_mistakes(kind):
    with pytest.raises(AssertionError):
        _check_hand(_planted(kind))


# ------------------------------------------------------- grouped K/V heads

def test_grouped_equals_plain_with_repeated_kv_heads():
    from oracle import attention_grouped
    q = _rand((2, 6, 19, 8), 1)
    k, v = _rand((2, 2, 19, 8), 2), _rand((2, 2, 19, 8), 3)
    for mask, wl, wr in MASKS[:4]:
        o, lse = attention_grouped(q, k, v, 0.4, mask, wl, wr)
        ro, rlse = attention_three_pass(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.4, mask, wl, wr)
        np.testing.assert_array_equal(o, ro)
        np.testing.assert_array_equal(lse, rlse)
    with pytest.raises(ValueError):
        attention_grouped(q, k[:, :1].repeat(4, axis=1), v[:, :1].repeat(4, axis=1), 0.4)


def test_grouped_head_mapping_is_contiguous_groups():
    """Query heads 0..G-1 share K/V head 0 (not heads 0, Hkv, 2 Hkv, ...)."""
    from oracle import attention_grouped
    q = _rand((1, 4, 5, 3), 4)
    k = np.stack([np.full((5, 3), 0.0), np.full((5, 3), 0.0)])[None]
    v = np.stack([np.full((5, 3), 1.0), np.full((5, 3), 2.0)])[None]
    o, _ = attention_grouped(q, k, v, 1.0)
    np.testing.assert_array_equal(o[0, :, 0, 0], [1.0, 1.0, 2.0, 2.0])
