"""Rotary position embedding (RoPE) of Q and K ahead of attention, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[AscendC FA-2] section 9 ("Extensions: integration with RoPE and a paged KV
cache") names RoPE fusion: the rotation is applied to the Q and K blocks as
they are loaded, from a table of cosines and sines.  The page gives no
formula, so this module writes out the standard rotary embedding:

    a row x at sequence position p is split into D/2 pairs (x_a, x_b); pair i
    turns by the angle p * theta_i, theta_i = base ** (-2 i / D):
        x_a' = x_a cos(p theta_i) - x_b sin(p theta_i)
        x_b' = x_b cos(p theta_i) + x_a sin(p theta_i)

Readings where the page is silent:
  * pairing.  STYLE_HALF pairs element i with i + D/2 (the form of the code
    shipped with the LLaMA, Qwen and Baichuan models the page's introduction
    names); STYLE_INTERLEAVED pairs 2i with 2i + 1 (the form of the original
    rotary-embedding paper).  Both are offered.
  * the table.  cos/sin are [n_pos, D/2] (row p, column i = angle p theta_i);
    the caller owns it, as the page's "needs a cos/sin table" suggests.
    ``rope_tables`` builds one from ``base``.
  * positions.  Row n of Q sits at position q_pos0 + n, row n of K at
    k_pos0 + n; only K and Q turn, V does not.
"""

import numpy as np

from .attention import MASK_NONE, attention_grouped

STYLE_HALF = 0
STYLE_INTERLEAVED = 1


def rope_tables(n_pos, D, base=10000.0):
    """cos, sin [n_pos, D/2] float64: entry (p, i) at the angle p * base^(-2i/D)."""
    if D % 2:
        raise ValueError("D must be even")
    i = np.arange(D // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / D)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def pair_index(D, style):
    """(a, b) index arrays of the D/2 rotated pairs for a pairing style."""
    h = D // 2
    if style == STYLE_HALF:
        return np.arange(h), np.arange(h) + h
    if style == STYLE_INTERLEAVED:
        return 2 * np.arange(h), 2 * np.arange(h) + 1
    raise ValueError(f"unknown RoPE style {style}")


def apply_rope(x, cos, sin, style=STYLE_HALF, pos0=0, seq_axis=-2):
    """Rotate every row of x (float64 result).

    x has its sequence on ``seq_axis`` and D on the last axis ([B, H, N, D]:
    seq_axis=-2; [B, N, H, D]: seq_axis=-3).  Row n turns by the table row
    pos0 + n, which must exist.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    n = x.shape[seq_axis]
    cos = np.asarray(cos, dtype=np.float64)
    sin = np.asarray(sin, dtype=np.float64)
    if cos.shape[-1] != D // 2 or pos0 < 0 or pos0 + n > cos.shape[0]:
        raise ValueError("table does not cover the rows")
    c = cos[pos0:pos0 + n]
    s = sin[pos0:pos0 + n]
    # broadcast the [n, D/2] table rows along every other axis of x
    shape = [1] * x.ndim
    shape[seq_axis] = n
    shape[-1] = D // 2
    c = c.reshape(shape)
    s = s.reshape(shape)
    a, b = pair_index(D, style)
    xa = x[..., a]
    xb = x[..., b]
    out = np.empty_like(x)
    out[..., a] = xa * c - xb * s
    out[..., b] = xb * c + xa * s
    return out


def attention_rope(q, k, v, scale, cos, sin, style=STYLE_HALF, mask_kind=MASK_NONE, win_l=-1, win_r=-1,
                   q_pos0=0, k_pos0=0, q_offset=0):
    """Attention of the rotated Q and K with V, [B, H, N, D] / [B, H_kv, N, D].

    The definition of [AscendC FA-2] section 1.1 applied to apply_rope(Q) and
    apply_rope(K); ``q_offset`` places the queries against the keys for the
    mask, as in ``attention_three_pass``.
    """
    qr = apply_rope(q, cos, sin, style, q_pos0)
    kr = apply_rope(k, cos, sin, style, k_pos0)
    return attention_grouped(qr, kr, v, scale, mask_kind, win_l, win_r, q_offset)
