"""Gradients of attention with respect to Q, K and V, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The second page ([ops-transformer] walk-through, closing remarks) notes that
the operator also has a backward pass, and the first page's section 9 lists
training support as an extension; neither writes it out.  This module takes
the plainest reading: the gradient of the three-pass definition of
[AscendC FA-2] section 1.1,

    S  = scale * Q K^T + mask         P = softmax_rows(S)       O = P V

for an upstream gradient dO of O, by the chain rule:

    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - rowsum(P * dP))         (softmax Jacobian, row by row)
    dQ = scale * dS K
    dK = scale * dS^T Q

Masked entries have P = 0 and so dS = 0; a row that sees no key has P = 0 and
contributes nothing.  The LSE output of the forward is not differentiated
(its gradient is taken as zero).  The fused kernels use the identity
rowsum(P * dP) = rowsum(dO * O), which ``tests/test_oracle_backward.py``
checks rather than assumes.
"""

import numpy as np

from .attention import MASK_NONE, attention_probs


def attention_backward(q, k, v, do, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1, q_offset=0):
    """(dQ, dK, dV) for [B, H, N, D] inputs (float64), the chain rule above."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            p = attention_probs(q[b, h], k[b, h], scale, mask_kind, win_l, win_r, q_offset)   # [Nq, Nk]
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def attention_backward_grouped(q, k, v, do, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1, q_offset=0):
    """The same for grouped K/V heads: query head h reads K/V head h // (H / H_kv),
    so a K/V head's gradient is the sum over the query heads that read it."""
    H, Hkv = q.shape[1], k.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    g = H // Hkv
    ke = np.repeat(np.asarray(k, dtype=np.float64), g, axis=1)
    ve = np.repeat(np.asarray(v, dtype=np.float64), g, axis=1)
    dq, dke, dve = attention_backward(q, ke, ve, do, scale, mask_kind, win_l, win_r, q_offset)
    B, _, Nk, D = ke.shape
    dk = dke.reshape(B, Hkv, g, Nk, D).sum(axis=2)
    dv = dve.reshape(B, Hkv, g, Nk, D).sum(axis=2)
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1, rows=(), keys=(),
                               row_chunk=1024):
    """dQ for the query rows `rows` and dK, dV for the keys `keys` of ONE (batch,
    head) ([N, D] arrays), by the same chain rule, for sequences too long for the
    whole N x N probability matrix: P's rows are formed a chunk at a time with
    the row max and sum of the definition, and only the requested rows and
    columns of dS are kept.  Returns (dq [len(rows), D], dk, dv [len(keys), D])."""
    from .attention import allowed_mask
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    n = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    dq = np.zeros((len(rows), q.shape[1]))
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    for c0 in range(0, n, row_chunk):
        c1 = min(n, c0 + row_chunk)
        p = attention_probs(q[c0:c1], k, scale, mask_kind, win_l, win_r, q_offset=c0)   # [chunk, Nk]
        dp = do[c0:c1] @ v.T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        if len(keys):
            dv += p[:, keys].T @ do[c0:c1]
            dk += scale * (ds[:, keys].T @ q[c0:c1])
        sel = (rows >= c0) & (rows < c1)
        if sel.any():
            dq[sel] = scale * (ds[rows[sel] - c0] @ k)
    return dq, dk, dv
