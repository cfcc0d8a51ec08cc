"""Pins of the paged-cache decode oracle.

(1) A hand-built table: the gathered rows are exactly the cache rows the
    table names, position by position.
(2) With pages in order the result equals the plain grouped decode on the
    contiguous cache (query i at position n - Nq + i).
(3) Moving pages in memory and the table with them changes nothing.
(4) Cache contents past a sequence's length, and in pages it does not use,
    change nothing.
(5) A planted off-by-one in the query position fails pin (2) for causal.
"""

import numpy as np
import pytest

from oracle import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, attention_grouped, attention_paged, gather_pages


def _rng(s):
    return np.random.default_rng(s)


def test_gather_hand_table():
    cache = np.arange(4 * 2 * 1 * 1, dtype=np.float64).reshape(4, 2, 1, 1)   # page p row r holds 2p + r
    rows = gather_pages(cache, [3, 0, 2], 5, 2)
    assert rows[:, 0, 0].tolist() == [6, 7, 0, 1, 4]


def _contiguous_case(B, H, Hkv, Nq, n, D, ps, seed):
    r = _rng(seed)
    q = r.standard_normal((B, H, Nq, D))
    k = r.standard_normal((B, Hkv, n, D))
    v = r.standard_normal((B, Hkv, n, D))
    pages = -(-n // ps)
    # page (b, p) at physical index b * pages + p, rows padded with garbage past n
    kc = r.standard_normal((B * pages, ps, Hkv, D))
    vc = r.standard_normal((B * pages, ps, Hkv, D))
    for b in range(B):
        for j in range(n):
            kc[b * pages + j // ps, j % ps] = k[b, :, j]
            vc[b * pages + j // ps, j % ps] = v[b, :, j]
    table = np.arange(B * pages).reshape(B, pages)
    return q, k, v, kc, vc, table


@pytest.mark.parametrize("mk,wl,wr", [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 5, 0)])
def test_in_order_pages_equal_contiguous_decode(mk, wl, wr):
    B, H, Hkv, Nq, n, D, ps = 2, 4, 2, 3, 37, 8, 8
    q, k, v, kc, vc, table = _contiguous_case(B, H, Hkv, Nq, n, D, ps, 1)
    o, lse = attention_paged(q, kc, vc, table, [n] * B, ps, 0.3, mk, wl, wr)
    ro, rl = attention_grouped(q, k, v, 0.3, mk, wl, wr, q_offset=n - Nq)
    assert np.allclose(o, ro, atol=1e-13) and np.allclose(lse, rl, atol=1e-13)


def test_moving_pages_changes_nothing_and_tails_are_ignored():
    B, H, Hkv, Nq, n, D, ps = 3, 2, 1, 1, 50, 4, 16
    q, k, v, kc, vc, table = _contiguous_case(B, H, Hkv, Nq, n, D, ps, 2)
    lens = [50, 17, 33]
    o0, l0 = attention_paged(q, kc, vc, table, lens, ps, 0.5, MASK_CAUSAL)
    perm = _rng(3).permutation(kc.shape[0])
    inv = np.argsort(perm)
    o1, l1 = attention_paged(q, kc[perm], vc[perm], inv[table], lens, ps, 0.5, MASK_CAUSAL)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    kc2, vc2 = kc.copy(), vc.copy()
    for b, n_b in enumerate(lens):
        for j in range(n_b, table.shape[1] * ps):
            kc2[table[b, j // ps], j % ps] = 1e3
            vc2[table[b, j // ps], j % ps] = -1e3
    o2, l2 = attention_paged(q, kc2, vc2, table, lens, ps, 0.5, MASK_CAUSAL)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_planted_off_by_one_position_is_caught():
    B, H, Hkv, Nq, n, D, ps = 1, 2, 2, 4, 20, 8, 4
    q, k, v, kc, vc, table = _contiguous_case(B, H, Hkv, Nq, n, D, ps, 4)
    o, _ = attention_paged(q, kc, vc, table, [n], ps, 0.3, MASK_CAUSAL)
    wrong, _ = attention_grouped(q, k, v, 0.3, MASK_CAUSAL, -1, -1, q_offset=n - Nq + 1)
    assert not np.allclose(o, wrong, atol=1e-6)
