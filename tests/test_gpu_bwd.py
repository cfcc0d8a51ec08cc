"""Backward pass on the GPU (fa_bwd) against the float64 oracle.

The kernels' arithmetic fixes the bound.  Each gradient entry is a sum of
products X = sum_t a_t b_t whose 16-bit factor (P for dV, dS for dK and dQ)
enters the tensor core rounded to the input type (unit roundoff u = 2^-11
fp16, 2^-8 bf16), the other factor exactly, with fp32 accumulation; so
    |dX| <= 1.05 u sum_t |a_t b_t|  +  2^-16 sum_t |a_t b_t|   (fp32 sums, P's ex2)
          + (the Dsum term, dK and dQ only) + half an ulp of X (16-bit output).
dS = P (dP - Dsum) uses Dsum = rowsum(dO * O) with O as the forward wrote it
(16-bit), so Dsum is off by up to sum_d |dO_d| halfulp(O_d); that error times
P, summed against |Q| (dK) or |K| (dQ) and the scale, is the Dsum term.
"""

import math

import numpy as np
import pytest
import torch

import attention_forward_16_gb300 as fa
from attention_forward_16_gb300.inputs import make_qkv
from oracle import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, attention_backward_grouped, attention_probs

pytestmark = pytest.mark.gpu

U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
MASKS = [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 100, 0), (MASK_WINDOW, 5, 2)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_16_gb300.build import build
    build()
    fa.load()


def _half_ulp(x, dtype):
    mant = {"f16": 10, "bf16": 7}[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - mant)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _run(q, k, v, do, mk, wl, wr, layout="bhnd"):
    """GPU forward (for O and LSE) and backward on host tensors ([B,H,N,D] order)."""
    perm = (lambda t: t.permute(0, 2, 1, 3).contiguous()) if layout == "bnhd" else (lambda t: t)
    dq_, dk_, dv_, ddo = (perm(t).cuda() for t in (q, k, v, do))
    window = (wl, wr) if mk == MASK_WINDOW else None
    o, lse = fa.attention_fwd(dq_, dk_, dv_, causal=mk == MASK_CAUSAL, window=window, layout=layout)
    gq, gk, gv = fa.attention_bwd(dq_, dk_, dv_, o, lse, ddo, causal=mk == MASK_CAUSAL, window=window,
                                  layout=layout)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    back = (lambda t: t.permute(0, 2, 1, 3)) if layout == "bnhd" else (lambda t: t)
    return tuple(back(t.cpu()) for t in (gq, gk, gv, o))


def _bounds(q, k, v, do, o16, scale, mk, wl, wr, dtype):
    """Per-entry bounds for dQ, dK, dV (see the module docstring)."""
    q, k, v, do = (_f64(t) for t in (q, k, v, do))
    B, H, N, D = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    u = U[dtype]
    bq = np.zeros_like(q)
    bk = np.zeros_like(k)
    bv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = h // g
            p = attention_probs(q[b, h], k[b, hk], scale, mk, wl, wr)
            dp = do[b, h] @ v[b, hk].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dsum_err = (np.abs(do[b, h]) * _half_ulp(o16[b, h], dtype)).sum(axis=1) + 1e-6
            pd = p * dsum_err[:, None]
            rel = 1.05 * u + 2.0 ** -16
            bv[b, hk] += rel * (p.T @ np.abs(do[b, h]))
            bk[b, hk] += abs(scale) * (rel * (np.abs(ds).T @ np.abs(q[b, h])) + pd.T @ np.abs(q[b, h]))
            bq[b, h] = abs(scale) * (rel * (np.abs(ds) @ np.abs(k[b, hk])) + pd @ np.abs(k[b, hk]))
    return bq, bk, bv


def _check(got, ref, bound, dtype, what):
    err = np.abs(got - ref)
    lim = bound + _half_ulp(ref, dtype) * 1.0001 + 1e-6
    worst = (err - lim).max()
    assert worst <= 0, f"{what}: worst excess {worst:.3e} (max err {err.max():.3e})"


def _inputs(B, H, Hkv, N, D, dtype, seed):
    q, _, _ = make_qkv(B, H, N, D, dtype, seed=seed, n_k=1)
    _, k, v = make_qkv(B, Hkv, 1, D, dtype, seed=seed + 1, n_k=N)
    do, _, _ = make_qkv(B, H, N, D, dtype, seed=seed + 2, n_k=1)
    return q, k, v, do


def _compare(q, k, v, do, mk, wl, wr, dtype, what, layout="bhnd"):
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D)
    gq, gk, gv, o16 = (_f64(t) for t in _run(q, k, v, do, mk, wl, wr, layout))
    rq, rk, rv = attention_backward_grouped(_f64(q), _f64(k), _f64(v), _f64(do), scale, mk, wl, wr)
    bq, bk, bv = _bounds(q, k, v, do, o16, scale, mk, wl, wr, dtype)
    _check(gv, rv, bv, dtype, "dV " + what)
    _check(gk, rk, bk, dtype, "dK " + what)
    _check(gq, rq, bq, dtype, "dQ " + what)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [128, 200, 384, 512])
def test_backward_matches_oracle(dtype, D, N):
    q, k, v, do = _inputs(1, 2, 2, N, D, dtype, seed=N + D)
    for mk, wl, wr in MASKS:
        _compare(q, k, v, do, mk, wl, wr, dtype, f"{dtype} D={D} N={N} mask=({mk},{wl},{wr})")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
def test_backward_grouped_heads_and_layouts(dtype, layout):
    q, k, v, do = _inputs(2, 4, 2, 300, 128, dtype, seed=77)
    for mk, wl, wr in [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1)]:
        _compare(q, k, v, do, mk, wl, wr, dtype, f"{dtype} {layout} GQA 4/2 mask={mk}", layout)


def test_backward_tiny_and_single_key():
    for N in (1, 2, 17):
        q, k, v, do = _inputs(1, 1, 1, N, 64, "f16", seed=N)
        _compare(q, k, v, do, MASK_CAUSAL, -1, -1, "f16", f"N={N} causal")
    # one row, one key: P = 1, so dV = dO and dQ = dK = 0 exactly
    q, k, v, do = _inputs(1, 1, 1, 1, 64, "bf16", seed=5)
    gq, gk, gv, _ = (_f64(t) for t in _run(q, k, v, do, MASK_NONE, -1, -1))
    assert np.array_equal(gv, _f64(do)) and not gq.any() and not gk.any()


def test_backward_is_deterministic():
    q, k, v, do = _inputs(1, 4, 4, 1000, 128, "bf16", seed=8)
    a = _run(q, k, v, do, MASK_CAUSAL, -1, -1)
    b = _run(q, k, v, do, MASK_CAUSAL, -1, -1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_rejects():
    t = [torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda") for _ in range(8)]
    q, k, v, o, do, dq, dk, dv = (x.data_ptr() for x in t)
    lse = torch.zeros(1, 1, 128, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 1, 128), dtype=torch.uint8, device="cuda")
    args = [q, k, v, o, do, lse.data_ptr(), dq, dk, dv, 1, 1, 1, 128, 64, 0.1, 0, -1, -1, 0, 0, ws.data_ptr(),
            ws.numel(), None]
    assert fa.fa_bwd(*args) == 0
    torch.cuda.synchronize()
    for idx, val, code in [(18, 2, fa.binding.FA_ERR_UNSUPPORTED),      # fp32
                           (13, 96, fa.binding.FA_ERR_UNSUPPORTED),     # D
                           (21, ws.numel() - 1, fa.binding.FA_ERR_ARG),  # workspace too small
                           (20, ws.data_ptr() + 16, fa.binding.FA_ERR_ALIGN),
                           (11, 3, fa.binding.FA_ERR_ARG),               # H_kv does not divide H
                           (5, None, fa.binding.FA_ERR_ARG)]:            # no LSE
        bad = list(args)
        bad[idx] = val
        assert fa.fa_bwd(*bad) == code, (idx, val)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
def test_unmasked_build_equals_masked_build(dtype, layout):
    """With no mask, whole key tiles and N >= 512 the backward kernels run
    their build without mask code; a window wider than the sequence selects
    the full build with every key visible.  Same sums in the same order:
    bit-equal gradients, and the no-mask ones match the oracle."""
    N, D = 512, 128
    q, k, v, do = _inputs(1, 4, 2, N, D, dtype, seed=77)
    plain = _run(q, k, v, do, MASK_NONE, -1, -1, layout)
    wide = _run(q, k, v, do, MASK_WINDOW, N, N, layout)
    for a, b in zip(plain, wide):
        assert torch.equal(a, b)
    _compare(q, k, v, do, MASK_NONE, -1, -1, dtype, f"unmasked build {dtype} {layout}", layout)


FULL = [("f16", MASK_CAUSAL), ("bf16", MASK_NONE)]


@pytest.mark.parametrize("dtype,mk", FULL)
def test_backward_full_size_sampled_heads(dtype, mk):
    """The benchmark shape B=4 H=32 N=4096 D=128: two whole heads against the oracle."""
    B, H, N, D = 4, 32, 4096, 128
    q, k, v, do = _inputs(B, H, H, N, D, dtype, seed=99)
    scale = 1.0 / math.sqrt(D)
    gq, gk, gv, o16 = _run(q, k, v, do, mk, -1, -1)
    for b, h in ((0, 0), (3, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        hq, hk, hv, hdo = (t[sl] for t in (q, k, v, do))
        rq, rk, rv = attention_backward_grouped(_f64(hq), _f64(hk), _f64(hv), _f64(hdo), scale, mk)
        bq, bk, bv = _bounds(hq, hk, hv, hdo, _f64(o16[sl]), scale, mk, -1, -1, dtype)
        _check(_f64(gv[sl]), rv, bv, dtype, f"dV full ({b},{h})")
        _check(_f64(gk[sl]), rk, bk, dtype, f"dK full ({b},{h})")
        _check(_f64(gq[sl]), rq, bq, dtype, f"dQ full ({b},{h})")


def _sampled_bounds(q, k, v, do, o16, scale, mk, wl, wr, dtype, rows, keys, chunk=1024):
    """The module's per-entry bounds for sampled dQ rows and dK, dV keys of one
    head ([N, D] float64 arrays), formed a chunk of query rows at a time."""
    from oracle import attention_probs
    u = U[dtype]
    rel = 1.05 * u + 2.0 ** -16
    rows, keys = np.asarray(rows), np.asarray(keys)
    bq = np.zeros((len(rows), q.shape[1]))
    bk = np.zeros((len(keys), q.shape[1]))
    bv = np.zeros((len(keys), q.shape[1]))
    for c0 in range(0, q.shape[0], chunk):
        c1 = min(q.shape[0], c0 + chunk)
        p = attention_probs(q[c0:c1], k, scale, mk, wl, wr, q_offset=c0)
        dp = do[c0:c1] @ v.T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dsum_err = (np.abs(do[c0:c1]) * _half_ulp(o16[c0:c1], dtype)).sum(axis=1) + 1e-6
        pd = p * dsum_err[:, None]
        bv += rel * (p[:, keys].T @ np.abs(do[c0:c1]))
        bk += abs(scale) * (rel * (np.abs(ds[:, keys]).T @ np.abs(q[c0:c1])) + pd[:, keys].T @ np.abs(q[c0:c1]))
        sel = (rows >= c0) & (rows < c1)
        if sel.any():
            r = rows[sel] - c0
            bq[sel] = abs(scale) * (rel * (np.abs(ds[r]) @ np.abs(k)) + pd[r] @ np.abs(k))
    return bq, bk, bv


@pytest.mark.parametrize("dtype,N,mk,wl,wr", [("bf16", 16384, MASK_CAUSAL, -1, -1),
                                              ("f16", 16384, MASK_WINDOW, 2048, 0)])
def test_backward_long_sequences_sampled(dtype, N, mk, wl, wr):
    """A long sequence: sampled query rows (dQ) and keys (dK, dV) against the
    oracle's chunked backward, within the module's bound (the oracle forms
    whole 16,384-key rows, seconds of host time per head)."""
    from oracle import attention_backward_sampled
    B, H, D = 1, 1, 128
    q, k, v, do = _inputs(B, H, H, N, D, dtype, seed=N)
    scale = 1.0 / math.sqrt(D)
    gq, gk, gv, o16 = _run(q, k, v, do, mk, wl, wr)
    rows = [0, 1, 4097, N // 2 + 3, N - 1]
    keys = [0, 130, N // 2, N - 200, N - 1]
    for h in range(H):
        hq, hk, hv, hdo = (_f64(t[0, h]) for t in (q, k, v, do))
        rq, rk, rv = attention_backward_sampled(hq, hk, hv, hdo, scale, mk, wl, wr, rows, keys)
        bq, bk, bv = _sampled_bounds(hq, hk, hv, hdo, _f64(o16[0, h]), scale, mk, wl, wr, dtype, rows, keys)
        _check(_f64(gq[0, h])[rows], rq, bq, dtype, f"dQ N={N} head {h}")
        _check(_f64(gk[0, h])[keys], rk, bk, dtype, f"dK N={N} head {h}")
        _check(_f64(gv[0, h])[keys], rv, bv, dtype, f"dV N={N} head {h}")
