"""Work and traffic accounting for the attention forward (host logic).

FLOPs follow the usual count for attention: 2 D flops for the score q_i.k_j
and 2 D for the weighted add p_ij v_j, i.e. 4 D per visible (i, j) pair
(4 B H N^2 D without a mask).  Masked pairs are not counted.

Algorithmic HBM bytes are the compulsory traffic: read Q, K, V once, write O
once and LSE once -- the IO lower bound the pages contrast with the naive
path's materialised N x N scores ("FlashAttention under the catlass
template", section "Principle", IO complexity; "FlashAttention extreme
optimisation on Ascend NPUs", "read once, write once").
"""

import numpy as np

MASK_NONE, MASK_CAUSAL, MASK_WINDOW = 0, 1, 2

_ELEM = {"f16": 2, "bf16": 2, "f32": 4}


def visible_keys_per_row(N, mask_kind, win_l=-1, win_r=-1):
    """int64 [N]: how many keys row i may attend to (closed form per row)."""
    i = np.arange(N, dtype=np.int64)
    if mask_kind == MASK_NONE:
        return np.full(N, N, dtype=np.int64)
    if mask_kind == MASK_CAUSAL:
        return i + 1
    if mask_kind != MASK_WINDOW:
        raise ValueError(mask_kind)
    lo = np.zeros(N, dtype=np.int64) if win_l < 0 else np.maximum(0, i - win_l)
    hi = np.full(N, N - 1, dtype=np.int64) if win_r < 0 else np.minimum(N - 1, i + win_r)
    return np.maximum(0, hi - lo + 1)


def unmasked_pairs(N, mask_kind, win_l=-1, win_r=-1):
    return int(visible_keys_per_row(N, mask_kind, win_l, win_r).sum())


def attention_flops(B, H, N, D, mask_kind, win_l=-1, win_r=-1):
    return 4 * D * B * H * unmasked_pairs(N, mask_kind, win_l, win_r)


def algorithmic_bytes(B, H, N, D, dtype, o_dtype=None, with_lse=True):
    e = _ELEM[dtype]
    eo = _ELEM[o_dtype or dtype]
    return B * H * N * D * (3 * e + eo) + (B * H * N * 4 if with_lse else 0)


def rope_bytes(w, tensors=1):
    """Compulsory bytes of the rotary embedding pass of workload ``w`` over
    ``tensors`` of Q and K (1: K alone, the pass the fused forward leaves;
    2: both): each read and its rotated copy written, plus the cos/sin table
    read once."""
    esize = {"f16": 2, "bf16": 2, "f32": 4}[w.dtype]
    x = tensors * w.B * w.H * w.N * w.D * esize
    return 2 * x + 2 * w.N * (w.D // 2) * 4
