"""Plain float64 attention, written from the pages' definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Slow and obviously
correct; no blocking, fusion or reordering beyond what each definition states.

Page names used below (full titles in the package docstring):
  [AscendC FA-2]    "Ascend C advanced practice: high-performance
                     FlashAttention-2-style tile-level fused attention"
  [ops-transformer] the hwcomputing.csdn.net walk-through of the
                     ops-transformer FlashAttention operator
  [catlass]         "FlashAttention under the catlass template" (lnwmold)
  [Ascend practice] "FlashAttention extreme optimisation on Ascend NPUs:
                     from principle to practice"

Conventions (readings of places where the pages are silent or disagree):
  * layout [B, H, N, D] ([ops-transformer] "the traditional attention flow",
    [catlass] "Usage", [Ascend practice] ``standard_attention``);
  * the scale multiplies Q K^T before masking and softmax ([AscendC FA-2]
    section 4.2 kernel: ``qk *= scale``), so the row max and the LSE are
    over scaled, masked scores, LSE in natural log;
  * causal: key j is visible to query i iff j <= i ([AscendC FA-2] section
    4.2 masks ``k > q``);
  * window (win_l, win_r): key j is visible iff i - win_l <= j <= i + win_r,
    both ends inclusive, a negative bound meaning "unbounded on that side"
    ([catlass] "Usage": a (window_left, window_right) tuple selects the
    sliding-window variant; the pages give no inclusivity or sign rule);
  * ``q_offset`` places query row i at key position i + q_offset (0 when
    queries and keys are the same sequence);
  * a row that sees no key at all has O = 0 and LSE = -inf.
"""

import math

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2


def allowed_mask(n_q, n_k, mask_kind, win_l=-1, win_r=-1, q_offset=0):
    """Boolean [n_q, n_k]: True where query i may attend to key j.

    Causal follows [AscendC FA-2] section 4.2 (a key after the query is set
    to -inf); the sliding window follows [catlass] "Usage" with the inclusive
    band reading stated in the module docstring.
    """
    i = np.arange(n_q, dtype=np.int64)[:, None] + int(q_offset)
    j = np.arange(n_k, dtype=np.int64)[None, :]
    if mask_kind == MASK_NONE:
        return np.ones((n_q, n_k), dtype=bool)
    if mask_kind == MASK_CAUSAL:
        return j <= i
    if mask_kind == MASK_WINDOW:
        ok = np.ones((n_q, n_k), dtype=bool)
        if win_l >= 0:
            ok &= j >= i - int(win_l)
        if win_r >= 0:
            ok &= j <= i + int(win_r)
        return ok
    raise ValueError(f"unknown mask kind {mask_kind}")


def unmasked_pairs(n, mask_kind, win_l=-1, win_r=-1):
    """Number of visible (i, j) pairs for one (batch, head) of length n,
    counted by materialising the mask row block by row block."""
    total = 0
    for r0 in range(0, n, 2048):
        r1 = min(n, r0 + 2048)
        total += int(allowed_mask(r1 - r0, n, mask_kind, win_l, win_r, q_offset=r0).sum())
    return total


def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def attention_probs(q, k, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1, q_offset=0):
    """Softmax probabilities P [n_q, n_k] for ONE (batch, head).

    [AscendC FA-2] section 1.1: P = Q K^T, S = softmax(P * scale) row-wise;
    masked scores are -inf so their probability is exactly 0.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    s = float(scale) * (q @ k.T)
    ok = allowed_mask(q.shape[0], k.shape[0], mask_kind, win_l, win_r, q_offset)
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])
    z = e.sum(axis=1)
    z_safe = np.where(empty, 1.0, z)
    return e / z_safe[:, None]


def attention_three_pass(q, k, v, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1,
                         q_offset=0, row_chunk=1024):
    """Standard three-pass attention in float64.

    For every (b, h): S = scale * Q K^T (materialised, one block of query rows
    at a time so the whole N x N matrix never exists at once; each block
    still holds complete rows of S), mask, M = row max, P = exp(S - M) / sum,
    O = P V, LSE = M + ln(sum exp(S - M)).

    Follows [AscendC FA-2] section 1.1, [ops-transformer] "the traditional
    attention flow" (S = Q K^T, P = softmax(S), O = P V) and
    [Ascend practice] ``standard_attention``.

    q: [B, H, Nq, D]; k, v: [B, H, Nk, D] (any float dtype; upcast exactly).
    Returns (O [B, H, Nq, D] float64, LSE [B, H, Nq] float64).
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, v.shape[3]), dtype=np.float64)
    lse = np.full((B, H, Nq), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            kk = k[b, h]
            vv = v[b, h]
            for r0 in range(0, Nq, row_chunk):
                r1 = min(Nq, r0 + row_chunk)
                s = float(scale) * (q[b, h, r0:r1] @ kk.T)
                ok = allowed_mask(r1 - r0, Nk, mask_kind, win_l, win_r, q_offset + r0)
                s = np.where(ok, s, -np.inf)
                m = s.max(axis=1)
                live = np.isfinite(m)
                m_safe = np.where(live, m, 0.0)
                e = np.exp(s - m_safe[:, None])
                z = e.sum(axis=1)
                z_safe = np.where(live, z, 1.0)
                p = e / z_safe[:, None]
                o[b, h, r0:r1] = p @ vv
                lse[b, h, r0:r1] = np.where(live, m_safe + np.log(z_safe), -np.inf)
    return o, lse


def attention_grouped(q, k, v, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1, q_offset=0):
    """Grouped-query attention: q [B, H, Nq, D], k and v [B, H_kv, Nk, D] with
    H a multiple of H_kv; query head h uses key/value head h // (H // H_kv).
    Each head is the plain definition of :func:`attention_three_pass`."""
    H, Hkv = q.shape[1], k.shape[1]
    if Hkv < 1 or H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    G = H // Hkv
    outs_o, outs_l = [], []
    for h in range(H):
        o, lse = attention_three_pass(q[:, h:h + 1], k[:, h // G:h // G + 1], v[:, h // G:h // G + 1], scale,
                                      mask_kind, win_l, win_r, q_offset)
        outs_o.append(o)
        outs_l.append(lse)
    return np.concatenate(outs_o, axis=1), np.concatenate(outs_l, axis=1)


def attention_online(q, k, v, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1,
                     q_offset=0, block_k=64):
    """The online-softmax recurrence over blocks of keys, in float64.

    [AscendC FA-2] section 1.2 and [ops-transformer] "online softmax:
    incremental update" keep a running row max m and a running sum l and
    divide by l once at the end.  The printed update steps are garbled (one
    adds the accumulator to itself, one divides by the new sum inside the
    loop, one subtracts the block max instead of the running max); this is
    the consistent textbook form of the same identity:

        m' = max(m, max_j S_j)
        l' = e^{m - m'} l + sum_j e^{S_j - m'}
        A' = e^{m - m'} A + sum_j e^{S_j - m'} V_j
        O  = A / l,   LSE = m + ln l

    with e^{-inf - (-inf)} taken as 0 while a row has seen no visible key.
    Returns (O, LSE) like :func:`attention_three_pass`.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, v.shape[3]), dtype=np.float64)
    lse = np.full((B, H, Nq), -np.inf, dtype=np.float64)
    ok_full = allowed_mask(Nq, Nk, mask_kind, win_l, win_r, q_offset)
    for b in range(B):
        for h in range(H):
            m = np.full(Nq, -np.inf)
            l = np.zeros(Nq)
            acc = np.zeros((Nq, v.shape[3]))
            for k0 in range(0, Nk, block_k):
                k1 = min(Nk, k0 + block_k)
                s = float(scale) * (q[b, h] @ k[b, h, k0:k1].T)
                s = np.where(ok_full[:, k0:k1], s, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)
                p = np.exp(s - m_use[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ v[b, h, k0:k1]
                m = m_new
            live = l > 0
            o[b, h] = np.where(live[:, None], acc / np.where(live, l, 1.0)[:, None], 0.0)
            lse[b, h] = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


def attention_bruteforce(q, k, v, scale, mask_kind=MASK_NONE, win_l=-1, win_r=-1,
                         q_offset=0):
    """Pure-Python triple loop over (i, j, d) for tiny inputs (no numpy
    arithmetic).  Same definition as :func:`attention_three_pass`, evaluated
    one scalar at a time; returns nested lists O[b][h][i][d], LSE[b][h][i]."""
    B, H, Nq, D = (len(q), len(q[0]), len(q[0][0]), len(q[0][0][0]))
    Nk = len(k[0][0])
    Dv = len(v[0][0][0])
    out_o, out_lse = [], []
    for b in range(B):
        ob, lb = [], []
        for h in range(H):
            oh, lh = [], []
            for i in range(Nq):
                pos = i + q_offset
                scores = []
                for j in range(Nk):
                    if mask_kind == MASK_CAUSAL and j > pos:
                        continue
                    if mask_kind == MASK_WINDOW:
                        if win_l >= 0 and j < pos - win_l:
                            continue
                        if win_r >= 0 and j > pos + win_r:
                            continue
                    dot = 0.0
                    for d in range(D):
                        dot += float(q[b][h][i][d]) * float(k[b][h][j][d])
                    scores.append((j, float(scale) * dot))
                if not scores:
                    oh.append([0.0] * Dv)
                    lh.append(-math.inf)
                    continue
                mx = max(s for _, s in scores)
                z = 0.0
                for _, s in scores:
                    z += math.exp(s - mx)
                row = []
                for d in range(Dv):
                    acc = 0.0
                    for j, s in scores:
                        acc += math.exp(s - mx) / z * float(v[b][h][j][d])
                    row.append(acc)
                oh.append(row)
                lh.append(mx + math.log(z))
            ob.append(oh)
            lb.append(lh)
        out_o.append(ob)
        out_lse.append(lb)
    return out_o, out_lse
