"""Split-K decode against a K/V cache, checked against the float64 oracle (GPU).

Query i sits at cache position Nk - Nq + i, so the oracle is the plain
three-pass attention with q_offset = Nk - Nq.  Decode computes in fp32 with
no 16-bit probabilities, so its error is the output rounding plus fp32
accumulation: |dO| - half an ulp of O <= 5e-5 for 16-bit outputs,
|dO| <= 1e-5 for fp32, |dLSE| <= 1e-5.
"""

import math

import numpy as np
import pytest
import torch

import attention_forward_16_gb300 as fa
from attention_forward_16_gb300 import binding as fb
from attention_forward_16_gb300.inputs import make_qkv
from oracle import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, attention_three_pass

pytestmark = pytest.mark.gpu

MASKS = [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 100, 0), (MASK_WINDOW, 5, 2)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_16_gb300.build import build
    build()
    fb.load()


def _half_ulp(x, dtype):
    mant = {"f16": 10, "bf16": 7}[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - mant)


def _cache(B, H, Nq, Nk, D, dtype, seed):
    q, _, _ = make_qkv(B, H, Nq, D, dtype, seed=seed, n_k=1)
    _, k, v = make_qkv(B, H, 1, D, dtype, seed=seed + 1, n_k=Nk)
    return q, k, v


def _decode(q, k, v, scale, mk, wl, wr, n_splits=0):
    window = (wl, wr) if mk == MASK_WINDOW else None
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=mk == MASK_CAUSAL,
                                 window=window, n_splits=n_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(o, lse, q, k, v, scale, mk, wl, wr, dtype, what):
    Nq, Nk = q.shape[2], k.shape[2]
    ro, rlse = attention_three_pass(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, mk, wl, wr,
                                    q_offset=Nk - Nq)
    live = np.isfinite(rlse)
    assert np.array_equal(np.isfinite(lse), live), what
    err = np.abs(o - ro)
    if dtype == "f32":
        assert err.max() <= 1e-5, f"{what}: max|dO| {err.max():.3e}"
    else:
        beyond = err - _half_ulp(ro, dtype)
        assert beyond.max() <= 5e-5, f"{what}: max(|dO| - ulp/2) {beyond.max():.3e}"
    if live.any():
        assert np.abs(lse[live] - rlse[live]).max() <= 1e-5, f"{what}: max|dLSE| {np.abs(lse[live] - rlse[live]).max():.3e}"


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 7), (1, 1000), (3, 255), (4, 4097), (16, 600), (16, 16)])
def test_decode_matches_oracle(dtype, D, Nq, Nk):
    q, k, v = _cache(2, 3, Nq, Nk, D, dtype, seed=Nq * 100 + Nk)
    scale = 1.0 / math.sqrt(D)
    for mk, wl, wr in MASKS:
        for ns in (0, 1, 5):
            o, lse = _decode(q, k, v, scale, mk, wl, wr, ns)
            _check(o, lse, q, k, v, scale, mk, wl, wr, dtype, f"{dtype} D={D} Nq={Nq} Nk={Nk} mask={mk} splits={ns}")


def test_decode_long_cache_many_splits():
    q, k, v = _cache(1, 8, 1, 65536, 128, "bf16", seed=7)
    for ns in (0, 64, 300):
        o, lse = _decode(q, k, v, 0.088, MASK_NONE, -1, -1, ns)
        _check(o, lse, q, k, v, 0.088, MASK_NONE, -1, -1, "bf16", f"65536 keys, {ns} splits")


def test_decode_split_count_does_not_change_result():
    q, k, v = _cache(2, 4, 2, 3000, 128, "f32", seed=8)
    base, lbase = _decode(q, k, v, 0.1, MASK_CAUSAL, -1, -1, 1)
    for ns in (2, 3, 16, 100):
        o, lse = _decode(q, k, v, 0.1, MASK_CAUSAL, -1, -1, ns)
        assert np.abs(o - base).max() <= 2e-6 and np.abs(lse - lbase).max() <= 2e-6, ns


def test_decode_equals_full_attention_rows():
    """The last Nq rows of the fused forward on the whole sequence are a decode."""
    B, H, N, D = 1, 4, 700, 128
    q, k, v = make_qkv(B, H, N, D, "f16", seed=9)
    ofull, lfull = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, o_dtype=torch.float32)
    od, ld = fa.attention_decode(q[:, :, -5:].contiguous().cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    # the fused forward rounds P to fp16 (relative 2^-11); decode keeps P in fp32
    assert (od.float() - ofull[:, :, -5:]).abs().max().item() <= 2e-3
    assert (ld - lfull[:, :, -5:]).abs().max().item() <= 1e-3


def test_decode_workspace_errors():
    q, k, v = (t.cuda() for t in _cache(1, 2, 1, 5000, 64, "f16", seed=10))
    o = torch.empty_like(q)
    ns, wb = fb.fa_decode_plan(1, 2, 1, 5000, 64, 4)
    assert ns == 4 and wb > 0
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, 1, 2, 1, 5000, 64, 0.1, 0, -1, -1,
            fb.FA_F16, 4)
    s = torch.cuda.current_stream().cuda_stream
    assert fb.fa_decode(*args, None, 0, s) == fb.FA_ERR_ARG
    assert fb.fa_decode(*args, ws.data_ptr(), wb - 1, s) == fb.FA_ERR_ARG
    assert fb.fa_decode(*args, ws.data_ptr() + 16, wb, s) == fb.FA_ERR_ALIGN
    assert fb.fa_decode(*args, ws.data_ptr(), wb, s) == fb.FA_OK
    torch.cuda.synchronize()
    ns1, wb1 = fb.fa_decode_plan(1, 2, 1, 5000, 64, 1)
    assert ns1 == 1 and wb1 == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
@pytest.mark.parametrize("H,Hkv,Nq", [(8, 8, 2), (8, 2, 2), (8, 1, 1), (16, 1, 1)])
@pytest.mark.parametrize("Nk", [999, 3000])
def test_decode_grouped_heads_and_layouts(dtype, layout, H, Hkv, Nq, Nk):
    from oracle import attention_grouped
    B, D = 2, 128
    q, _, _ = make_qkv(B, H, Nq, D, dtype, seed=900 + Hkv, n_k=1)
    _, k, v = make_qkv(B, Hkv, 1, D, dtype, seed=901 + Hkv, n_k=Nk)
    perm = (lambda t: t.permute(0, 2, 1, 3).contiguous()) if layout == "bnhd" else (lambda t: t)
    for mk, wl, wr in MASKS:
        for ns in (0, 1, 7):
            window = (wl, wr) if mk == MASK_WINDOW else None
            o, lse = fa.attention_decode(perm(q).cuda(), perm(k).cuda(), perm(v).cuda(), scale=0.1,
                                         causal=mk == MASK_CAUSAL, window=window, n_splits=ns, layout=layout)
            torch.cuda.synchronize()
            o = perm(o.cpu()).float().numpy().astype(np.float64)
            ro, rlse = attention_grouped(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.1, mk, wl, wr,
                                         q_offset=Nk - Nq)
            err = np.abs(o - ro)
            what = f"{dtype} {layout} H={H} Hkv={Hkv} Nq={Nq} Nk={Nk} mask={mk} splits={ns}"
            if dtype == "f32":
                assert err.max() <= 1e-5, what
            else:
                assert (err - _half_ulp(ro, dtype)).max() <= 5e-5, what
            assert np.abs(lse.cpu().numpy() - rlse).max() <= 1e-5, what


def test_decode_grouped_rejects_too_many_rows():
    q = torch.zeros(1, 32, 1, 128, dtype=torch.float16, device="cuda")
    p = q.data_ptr()
    # 32 query heads on one K/V head: 32 rows per group > 16
    assert fb.fa_decode_gqa(p, p, p, p, None, 1, 32, 1, 1, 64, 128, 0.1, 0, -1, -1, fb.FA_F16, 0, 1, None, 0,
                            None) == fb.FA_ERR_UNSUPPORTED
    assert fb.fa_decode_gqa(p, p, p, p, None, 1, 32, 5, 1, 64, 128, 0.1, 0, -1, -1, fb.FA_F16, 0, 1, None, 0,
                            None) == fb.FA_ERR_ARG


# ------------------------------------------------------------- paged cache

def _paged_case(B, H, Hkv, Nq, lens, D, ps, dtype, seed):
    """Q, a page-shuffled cache holding each sequence's K/V, its table and lengths."""
    rng = np.random.default_rng(seed)
    max_pages = -(-max(lens) // ps)
    num_pages = B * max_pages + 3
    q, _, _ = make_qkv(B, H, Nq, D, dtype, seed=seed, n_k=1)
    _, kc, vc = make_qkv(1, num_pages, 1, D * Hkv, dtype, seed=seed + 1, n_k=ps)   # [1, pages, ps, Hkv*D]
    kc = kc.reshape(num_pages, ps, Hkv, D).contiguous()
    vc = vc.reshape(num_pages, ps, Hkv, D).contiguous()
    table = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    return q, kc, vc, table, np.array(lens, dtype=np.int32)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("H,Hkv,Nq", [(4, 4, 1), (8, 2, 1), (8, 2, 3)])
@pytest.mark.parametrize("ps", [16, 64])
def test_paged_decode_matches_oracle(dtype, H, Hkv, Nq, ps):
    from oracle import attention_paged
    B, D = 3, 128
    lens = [1000, 37, 2 * ps + 1]
    q, kc, vc, table, sl = _paged_case(B, H, Hkv, Nq, lens, D, ps, dtype, seed=ps + H + Nq)
    for mk, wl, wr in MASKS:
        window = (wl, wr) if mk == MASK_WINDOW else None
        for ns in (0, 1, 5):
            o, lse = fa.attention_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(table).cuda(),
                                               torch.from_numpy(sl).cuda(), scale=0.1, causal=mk == MASK_CAUSAL,
                                               window=window, n_splits=ns)
            torch.cuda.synchronize()
            ro, rlse = attention_paged(q.double().numpy(), kc.double().numpy(), vc.double().numpy(), table, sl, ps,
                                       0.1, mk, wl, wr)
            o = o.float().cpu().numpy().astype(np.float64)
            lse = lse.cpu().numpy().astype(np.float64)
            what = f"paged {dtype} H={H} Hkv={Hkv} Nq={Nq} ps={ps} mask={mk} splits={ns}"
            live = np.isfinite(rlse)
            assert np.array_equal(np.isfinite(lse), live), what
            err = np.abs(o - ro)
            if dtype == "f32":
                assert err.max() <= 1e-5, what
            else:
                assert (err - _half_ulp(ro, dtype)).max() <= 5e-5, what
            assert np.abs(lse[live] - rlse[live]).max() <= 1e-5, what


def test_paged_in_order_equals_contiguous_decode():
    B, H, Hkv, Nq, Nk, D, ps = 2, 8, 2, 1, 4096, 128, 256
    q, _, _ = make_qkv(B, H, Nq, D, "bf16", seed=31, n_k=1)
    _, k, v = make_qkv(B, Hkv, 1, D, "bf16", seed=32, n_k=Nk)
    kb, vb = (t.permute(0, 2, 1, 3).contiguous() for t in (k, v))   # [B, Nk, Hkv, D]
    kc = kb.reshape(B * (Nk // ps), ps, Hkv, D).contiguous()
    vc = vb.reshape(B * (Nk // ps), ps, Hkv, D).contiguous()
    table = torch.arange(B * (Nk // ps), dtype=torch.int32).reshape(B, Nk // ps)
    sl = torch.full((B,), Nk, dtype=torch.int32)
    qc = q.cuda()
    o1, l1 = fa.attention_decode_paged(qc, kc.cuda(), vc.cuda(), table.cuda(), sl.cuda(), causal=True)
    o2, l2 = fa.attention_decode(qc.permute(0, 2, 1, 3).contiguous(), kb.cuda(), vb.cuda(), causal=True,
                                 layout="bnhd")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2.permute(0, 2, 1, 3)) and torch.equal(l1, l2)


def test_paged_short_sequences_see_no_key():
    # a sequence shorter than its query count: its early queries sit at negative positions
    q, kc, vc, table, sl = _paged_case(2, 4, 4, 3, [1, 50], 64, 16, "f16", seed=40)
    o, lse = fa.attention_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(table).cuda(),
                                       torch.from_numpy(sl).cuda(), causal=True)
    torch.cuda.synchronize()
    lse = lse.cpu()
    assert torch.isinf(lse[0, :, :2]).all() and torch.isfinite(lse[0, :, 2]).all() and torch.isfinite(lse[1]).all()
    assert (o.cpu()[0, :, :2] == 0).all()
