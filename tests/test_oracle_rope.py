"""Pins of the RoPE oracle against constructions other than its own formula.

The rotation is checked against (1) complex multiplication by e^{i p theta},
(2) the matrix exponential of the skew-symmetric generator (scipy ``expm``),
(3) closed-form table entries, and (4) the invariants a rotary embedding must
have: orthogonality, the identity at position 0, composition of positions,
and dot products that depend only on the position difference.  The last
tests plant mistakes in the oracle's inputs and show that the pins catch
them.
"""

import math

import numpy as np
import pytest

from oracle import (MASK_CAUSAL, MASK_NONE, STYLE_HALF, STYLE_INTERLEAVED, apply_rope, attention_grouped,
                    attention_rope, pair_index, rope_tables)

STYLES = [STYLE_HALF, STYLE_INTERLEAVED]


def _rng(seed):
    return np.random.default_rng(seed)


def test_table_closed_forms():
    cos, sin = rope_tables(200, 128, base=10000.0)
    # column 0 turns by exactly one radian per position
    for p in (0, 1, 7, 199):
        assert cos[p, 0] == pytest.approx(math.cos(p), abs=1e-15)
        assert sin[p, 0] == pytest.approx(math.sin(p), abs=1e-15)
    # column D/4 of a base-10000 table: theta = 10000^(-1/2) = 0.01
    for p in (1, 100, 157):
        assert cos[p, 32] == pytest.approx(math.cos(0.01 * p), abs=1e-14)
        assert sin[p, 32] == pytest.approx(math.sin(0.01 * p), abs=1e-14)
    assert np.allclose(cos ** 2 + sin ** 2, 1.0, atol=1e-15)
    # angles add: e^{i(p+r)theta} = e^{i p theta} e^{i r theta}
    z = cos + 1j * sin
    assert np.allclose(z[37] * z[55], z[92], atol=1e-13)
    # the angle falls as the pair index grows (theta_i decreasing, all positive)
    ang = np.unwrap(np.angle(z[1]))
    assert np.all(np.diff(ang) < 0) and np.all(ang > 0)


@pytest.mark.parametrize("style", STYLES)
def test_complex_multiplication_form(style):
    D, N = 64, 9
    cos, sin = rope_tables(N + 5, D, base=500.0)
    x = _rng(1).standard_normal((2, 3, N, D))
    got = apply_rope(x, cos, sin, style, pos0=5)
    a, b = pair_index(D, style)
    z = (x[..., a] + 1j * x[..., b]) * (cos[5:5 + N] + 1j * sin[5:5 + N])
    want = np.empty_like(x)
    want[..., a] = z.real
    want[..., b] = z.imag
    assert np.allclose(got, want, atol=1e-14)


@pytest.mark.parametrize("style", STYLES)
def test_matrix_exponential_of_generator(style):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    D, base = 16, 10000.0
    theta = base ** (-np.arange(D // 2) * 2.0 / D)
    a, b = pair_index(D, style)
    G = np.zeros((D, D))
    G[b, a] = theta
    G[a, b] = -theta
    cos, sin = rope_tables(64, D, base)
    x = _rng(2).standard_normal((1, 1, 1, D))
    for p in (0, 1, 13, 63):
        R = scipy_linalg.expm(p * G)
        got = apply_rope(x, cos, sin, style, pos0=p)[0, 0, 0]
        assert np.allclose(got, R @ x[0, 0, 0], atol=1e-12), p


@pytest.mark.parametrize("style", STYLES)
def test_invariants(style):
    D, N = 32, 40
    cos, sin = rope_tables(2 * N + 10, D, base=10000.0)
    x = _rng(3).standard_normal((2, 2, N, D))
    y = apply_rope(x, cos, sin, style)
    # a rotation keeps every row's norm, and row 0 (position 0) is untouched
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.array_equal(y[:, :, 0], x[:, :, 0])
    # positions compose: turning by p1 then by p2 is turning by p1 + p2
    one = x[:, :, :1]
    twice = apply_rope(apply_rope(one, cos, sin, style, pos0=11), cos, sin, style, pos0=23)
    assert np.allclose(twice, apply_rope(one, cos, sin, style, pos0=34), atol=1e-12)
    # q.k depends only on the position difference
    q = x[0, 0, :1]
    k = x[1, 1, :1]
    d0 = np.dot(apply_rope(q, cos, sin, style, pos0=7, seq_axis=-2)[0],
                apply_rope(k, cos, sin, style, pos0=3, seq_axis=-2)[0])
    d1 = np.dot(apply_rope(q, cos, sin, style, pos0=47, seq_axis=-2)[0],
                apply_rope(k, cos, sin, style, pos0=43, seq_axis=-2)[0])
    assert d0 == pytest.approx(d1, abs=1e-12)


def test_half_and_interleaved_differ_by_a_permutation():
    D, N = 32, 12
    cos, sin = rope_tables(N, D)
    x = _rng(4).standard_normal((1, 2, N, D))
    perm = np.empty(D, dtype=np.int64)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2
    half = apply_rope(x, cos, sin, STYLE_HALF)
    inter = apply_rope(x[..., perm], cos, sin, STYLE_INTERLEAVED)
    back = np.empty_like(inter)
    back[..., perm] = inter
    assert np.allclose(half, back, atol=1e-14)


def test_bnhd_axis_matches_bhnd():
    D, N = 16, 10
    cos, sin = rope_tables(N + 3, D)
    x = _rng(5).standard_normal((2, 3, N, D))
    y = apply_rope(x, cos, sin, STYLE_HALF, pos0=3)
    yt = apply_rope(x.transpose(0, 2, 1, 3), cos, sin, STYLE_HALF, pos0=3, seq_axis=-3)
    assert np.allclose(yt.transpose(0, 2, 1, 3), y, atol=0)


def test_attention_rope_identity_table_and_shift_invariance():
    B, H, N, D = 1, 2, 24, 16
    r = _rng(6)
    q, k, v = (r.standard_normal((B, H, N, D)) for _ in range(3))
    one = np.ones((64, D // 2))
    zero = np.zeros((64, D // 2))
    o_id, l_id = attention_rope(q, k, v, 0.25, one, zero)
    o_ref, l_ref = attention_grouped(q, k, v, 0.25)
    assert np.allclose(o_id, o_ref, atol=0) and np.allclose(l_id, l_ref, atol=0)
    cos, sin = rope_tables(64, D)
    for mk in (MASK_NONE, MASK_CAUSAL):
        o0, l0 = attention_rope(q, k, v, 0.25, cos, sin, STYLE_HALF, mk)
        o1, l1 = attention_rope(q, k, v, 0.25, cos, sin, STYLE_HALF, mk, q_pos0=30, k_pos0=30)
        assert np.allclose(o0, o1, atol=1e-12) and np.allclose(l0, l1, atol=1e-12)
        # moving only the keys changes the result
        o2, _ = attention_rope(q, k, v, 0.25, cos, sin, STYLE_HALF, mk, q_pos0=0, k_pos0=30)
        assert np.abs(o2 - o0).max() > 1e-3


@pytest.mark.parametrize("mistake", ["sin_sign", "swapped_pairs", "shifted_table"])
def test_planted_mistakes_are_caught(mistake):
    """A plausible slip in the rotation fails the generator pin."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    D = 8
    theta = 10000.0 ** (-np.arange(D // 2) * 2.0 / D)
    a, b = pair_index(D, STYLE_HALF)
    G = np.zeros((D, D))
    G[b, a] = theta
    G[a, b] = -theta
    cos, sin = rope_tables(16, D)
    x = _rng(7).standard_normal((1, 1, 1, D))
    p = 5
    want = scipy_linalg.expm(p * G) @ x[0, 0, 0]
    if mistake == "sin_sign":
        got = apply_rope(x, cos, -sin, STYLE_HALF, pos0=p)
    elif mistake == "swapped_pairs":
        got = apply_rope(x, cos, sin, STYLE_INTERLEAVED, pos0=p)
    else:
        got = apply_rope(x, cos, sin, STYLE_HALF, pos0=p + 1)
    assert not np.allclose(got[0, 0, 0], want, atol=1e-6)
