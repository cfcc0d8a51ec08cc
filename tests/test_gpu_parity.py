"""Parity of the CUDA path against the float64 oracle (GPU).

Tolerances (fixed by the method's targets; derivation for 16-bit O below):
  * fp32 inputs (FFMA kernel): max|dO| <= 1e-5, max|dLSE| <= 1e-5.
  * fp16/bf16 inputs, O written in fp32: max|dO| <= 2e-3, max|dLSE| <= 1e-3.
  * fp16/bf16 inputs, O written in the input type: the output rounding alone
    is up to half an ulp of |O| (bf16: 3.9e-3 for |O| in [1, 2)), so the bound
    is applied to |dO| minus half an ulp of the oracle value: <= 2e-3.
Inputs come from the seeded generator; the oracle sees the same rounded
values upcast to float64.
"""

import math

import numpy as np
import pytest
import torch

import attention_forward_16_gb300 as fa
from attention_forward_16_gb300 import binding as fb
from attention_forward_16_gb300.inputs import WORKLOADS, make_qkv, make_workload, torch_dtype
from oracle import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, attention_three_pass

pytestmark = pytest.mark.gpu

TOL_O_F32 = 1e-5
TOL_O_16 = 2e-3
TOL_LSE_16 = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_16_gb300.build import build
    build()
    fb.load()


def _half_ulp(x, dtype):
    """Half a unit in the last place of |x| in the 16-bit type (normal range)."""
    mant = {"f16": 10, "bf16": 7}[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - mant)


def _run(q, k, v, scale, mk, wl, wr, o_f32=False):
    window = None
    causal = False
    if mk == MASK_CAUSAL:
        causal = True
    elif mk == MASK_WINDOW:
        window = (wl, wr)
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, window=window,
                              o_dtype=torch.float32 if o_f32 else None)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _ref(q, k, v, scale, mk, wl, wr, heads=None):
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    if heads is not None:
        b, h = heads
        qd, kd, vd = qd[b:b + 1, h:h + 1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1]
    return attention_three_pass(qd, kd, vd, scale, mk, wl, wr)


def _check(o, lse, ro, rlse, dtype, o_f32, what):
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    err = np.abs(o - ro)
    if dtype == "f32":
        assert err.max() <= TOL_O_F32, f"{what}: max|dO| {err.max():.3e}"
        assert np.abs(lse - rlse).max() <= 1e-5, f"{what}: max|dLSE| {np.abs(lse - rlse).max():.3e}"
        return
    if o_f32:
        worst = np.unravel_index(np.argmax(err), err.shape)
        assert err.max() <= TOL_O_16, f"{what}: max|dO| {err.max():.3e} at {worst}"
    else:
        beyond = err - _half_ulp(ro, dtype)
        worst = np.unravel_index(np.argmax(beyond), beyond.shape)
        assert beyond.max() <= TOL_O_16, f"{what}: max(|dO| - ulp/2) {beyond.max():.3e} at {worst}"
    lerr = np.abs(lse - rlse)
    assert lerr.max() <= TOL_LSE_16, f"{what}: max|dLSE| {lerr.max():.3e}"


# --------------------------------------------------------- the small configs

@pytest.mark.parametrize("name", ["tiny_f32_full", "tiny_f32_causal"])
def test_tiny_fp32(name):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o, lse = _run(q, k, v, w.scale, w.mask, w.win_l, w.win_r)
    ro, rlse = _ref(q, k, v, w.scale, w.mask, w.win_l, w.win_r)
    _check(o, lse, ro, rlse, "f32", True, name)


@pytest.mark.parametrize("o_f32", [False, True])
def test_f16_causal_1k(o_f32):
    w = WORKLOADS["f16_causal_1k"]
    q, k, v = make_workload(w)
    o, lse = _run(q, k, v, w.scale, w.mask, w.win_l, w.win_r, o_f32)
    ro, rlse = _ref(q, k, v, w.scale, w.mask, w.win_l, w.win_r)
    _check(o, lse, ro, rlse, "f16", o_f32, "f16_causal_1k")


# ------------------------------------------------- ragged sizes and all masks

MASK_SET = [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 37, 5), (MASK_WINDOW, 200, 0),
            (MASK_WINDOW, 0, 0), (MASK_WINDOW, -1, 3), (MASK_WINDOW, 130, -1)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 256, 257, 640, 1000])
def test_ragged_all_masks(dtype, D, N):
    q, k, v = make_qkv(1, 2, N, D, dtype, seed=7000 + N + D)
    scale = 1.0 / math.sqrt(D)
    for mk, wl, wr in MASK_SET:
        for o_f32 in (True, False):
            o, lse = _run(q, k, v, scale, mk, wl, wr, o_f32)
            ro, rlse = _ref(q, k, v, scale, mk, wl, wr)
            _check(o, lse, ro, rlse, dtype, o_f32, f"{dtype} D={D} N={N} mask={mk},{wl},{wr} o_f32={o_f32}")


@pytest.mark.parametrize("N", [1, 5, 33, 64, 100, 257])
@pytest.mark.parametrize("D", [1, 16, 40, 64, 128])
def test_fp32_ragged(N, D):
    q, k, v = make_qkv(2, 1, N, D, "f32", seed=8000 + N + D)
    for mk, wl, wr in MASK_SET:
        o, lse = _run(q, k, v, 0.3, mk, wl, wr)
        ro, rlse = _ref(q, k, v, 0.3, mk, wl, wr)
        _check(o, lse, ro, rlse, "f32", True, f"f32 N={N} D={D} mask={mk},{wl},{wr}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_many_heads_several_units_per_cta(dtype):
    """More units than SMs: every persistent CTA runs several units, so the
    barrier phases, the K/V ring and TMEM reuse cross unit boundaries."""
    q, k, v = make_qkv(3, 70, 300, 64, dtype, seed=99)
    for mk, wl, wr in [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 100, 20)]:
        o, lse = _run(q, k, v, 0.125, mk, wl, wr, True)
        ro, rlse = _ref(q, k, v, 0.125, mk, wl, wr)
        _check(o, lse, ro, rlse, dtype, True, f"many heads {dtype} mask={mk}")


# ------------------------------------------------------------- special cases

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("c", [0.0, 1.5, -3.0])
def test_constant_v(dtype, c):
    q, k, _ = make_qkv(1, 2, 300, 128, dtype, seed=5)
    v = torch.full_like(q, c)
    # O = c * sum(P rounded) / sum(p): off from c by at most the unit
    # roundoff of P (2^-11 for fp16; for bf16 2^-8, or about 2^-16 where P is split).
    u_p = 2.0 ** -11 if dtype == "f16" else 2.0 ** -8
    for mk, wl, wr in MASK_SET[:4]:
        o, _ = _run(q, k, v, 0.09, mk, wl, wr, True)
        assert np.abs(o - c).max() <= abs(c) * u_p + 1e-6, (mk, np.abs(o - c).max())


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_causal_row_zero_is_v0_bit_exact(dtype):
    q, k, v = make_qkv(2, 3, 200, 64, dtype, seed=6)
    o, lse = _run(q, k, v, 0.125, MASK_CAUSAL, -1, -1)
    v0 = v[:, :, 0].double().numpy()
    assert np.array_equal(o[:, :, 0], v0)
    ref_lse = 0.125 * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy()
    assert np.abs(lse[:, :, 0] - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_zero_and_negative_scale(dtype):
    q, k, v = make_qkv(1, 2, 333, 64, dtype, seed=8)
    for scale in (0.0, -0.2):
        for mk, wl, wr in MASK_SET:
            o, lse = _run(q, k, v, scale, mk, wl, wr, True)
            ro, rlse = _ref(q, k, v, scale, mk, wl, wr)
            _check(o, lse, ro, rlse, dtype, True, f"scale={scale} mask={mk},{wl},{wr}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_large_scores_exercise_lazy_rescale(dtype):
    """scale=1 at D=64 gives scores with std 8: the running max moves by more
    than the lazy-rescale threshold many times along a row, and rows put
    their mass on a few keys.  There the rounding of P to the 16-bit type
    (unit roundoff u_P = 2^-11 fp16, 2^-8 bf16) no longer averages out; with O
    normalised by the exact fp32 row sum the first-order error is
    |dO_id| <= u_P * sum_j P_ij |V_jd|, which is what is asserted (plus fp32
    accumulation slack).  LSE keeps its 1e-3 bound."""
    from oracle import attention_probs
    q, k, v = make_qkv(1, 2, 700, 64, dtype, seed=9)
    u_p = 2.0 ** -11 if dtype == "f16" else 2.0 ** -8
    for mk, wl, wr in MASK_SET[:3]:
        o, lse = _run(q, k, v, 1.0, mk, wl, wr, True)
        ro, rlse = _ref(q, k, v, 1.0, mk, wl, wr)
        for h in range(2):
            P = attention_probs(q[0, h].double().numpy(), k[0, h].double().numpy(), 1.0, mk, wl, wr)
            bound = u_p * (P @ np.abs(v[0, h].double().numpy())) * 1.01 + 2e-5
            err = np.abs(o[0, h] - ro[0, h])
            assert (err <= bound).all(), (mk, h, float((err - bound).max()))
        assert np.abs(lse - rlse).max() <= TOL_LSE_16


def test_increasing_scores_force_rescale_every_tile():
    """Keys grow along the sequence so each new key tile raises every row's
    max well past the threshold: the O rescale runs on every tile."""
    N, D = 1024, 64
    q = torch.ones(1, 1, N, D)
    k = (torch.arange(N, dtype=torch.float32) / 16.0)[None, None, :, None].expand(1, 1, N, D).contiguous()
    v = torch.randn(1, 1, N, D, generator=torch.Generator().manual_seed(3))
    q, k, v = q.half(), k.half(), v.half()
    o, lse = _run(q, k, v, 1.0 / D, MASK_NONE, -1, -1, True)
    ro, rlse = _ref(q, k, v, 1.0 / D, MASK_NONE, -1, -1)
    _check(o, lse, ro, rlse, "f16", True, "monotone keys")


def test_deterministic():
    q, k, v = make_qkv(2, 4, 1000, 128, "bf16", seed=10)
    a = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    b = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------- C ABI called with pointers

@pytest.mark.parametrize("fn,dtype", [("fa_fwd_f16", "f16"), ("fa_fwd_bf16", "bf16"), ("fa_fwd_f32", "f32")])
def test_typed_c_abi_entry_points(fn, dtype):
    q, k, v = make_qkv(1, 3, 200, 64, dtype, seed=11)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(1, 3, 200, device="cuda", dtype=torch.float32)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    rc = getattr(fb, fn)(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         1, 3, 200, 64, 0.125, fb.FA_MASK_WINDOW, 50, 10, stream.cuda_stream)
    assert rc == 0
    assert fb.fa_device_status(stream.cuda_stream) == 0
    ro, rlse = _ref(q, k, v, 0.125, MASK_WINDOW, 50, 10)
    _check(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rlse, dtype,
           dtype == "f32", fn)


def test_lse_pointer_may_be_null():
    q, k, v = make_qkv(1, 1, 100, 64, "f16", seed=12)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    rc = fb.fa_fwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), None, 1, 1, 100, 64, 0.125,
                   fb.FA_MASK_CAUSAL, -1, -1, fb.FA_F16, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ro, _ = _ref(q, k, v, 0.125, MASK_CAUSAL, -1, -1)
    beyond = np.abs(o.float().cpu().numpy() - ro) - _half_ulp(ro, "f16")
    assert beyond.max() <= TOL_O_16


def test_misaligned_device_pointer_rejected():
    buf = torch.empty(4096, dtype=torch.float16, device="cuda")
    p = buf.data_ptr() + 2
    assert fb.fa_fwd(p, p, p, buf.data_ptr(), None, 1, 1, 16, 64, 0.1, 0, -1, -1, fb.FA_F16, None) == fb.FA_ERR_ALIGN


def test_host_buffers_round_trip():
    q, k, v = make_qkv(1, 2, 300, 128, "bf16", seed=13)
    o, lse = fa.attention_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True)
    ro, rlse = _ref(q, k, v, 1.0 / math.sqrt(128), MASK_CAUSAL, -1, -1)
    _check(o.float().numpy().astype(np.float64), lse.numpy().astype(np.float64), ro, rlse, "bf16", False, "host")


# ------------------------------------------------------------------ watchdog

def test_watchdog_reports_timeout_and_context_survives():
    assert fb.fa_device_status(None) == 0
    assert fb.fa_selftest_wait_timeout(20_000_000, None) == 0      # 20 ms wait nobody ends
    assert fb.fa_device_status(None) == fb.FA_ERR_TIMEOUT
    assert fb.fa_device_status(None) == 0                           # cleared
    q, k, v = make_qkv(1, 2, 256, 64, "f16", seed=14)
    o, lse = _run(q, k, v, 0.125, MASK_CAUSAL, -1, -1, True)
    ro, rlse = _ref(q, k, v, 0.125, MASK_CAUSAL, -1, -1)
    _check(o, lse, ro, rlse, "f16", True, "after watchdog")


@pytest.mark.parametrize("kernel", ["one_cta", "cta_pair"])
@pytest.mark.parametrize("dtype,mk", [("f16", MASK_NONE), ("bf16", MASK_CAUSAL)])
def test_forward_kernel_waits_run_out_and_context_survives(dtype, mk, kernel):
    """The attention kernel's own bounded waits, not a separate probe: with the
    limit at its 1 us floor, the first wait for a Q or K/V tile from HBM (or
    for the first S) outlasts it, so every CTA records a timeout, stops, lets
    the copies and products it issued land (the exit drain keeps its own 1 s
    bound), frees TMEM and returns; in the 2-CTA kernel a timeout in either
    CTA stops both, and the pair frees TMEM together once the first CTA's
    products have drained.  The host reads FA_ERR_TIMEOUT; with the limit
    restored, the next call on the same context passes parity."""
    q, k, v = make_qkv(2, 16, 2048, 128, dtype, seed=16)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    causal = mk == MASK_CAUSAL
    assert fb.fa_device_status(None) == 0
    sel = fb.fa_select_fwd_kernel(fb.FA_FWD_CTA_PAIR if kernel == "cta_pair" else fb.FA_FWD_ONE_CTA)
    prev = fb.fa_set_wait_limit_ns(1)          # raised to the 1 us floor
    try:
        fa.attention_fwd(dq, dk, dv, causal=causal)   # outputs undefined: the launch is cut short
        torch.cuda.synchronize()
        rc = fb.fa_device_status(None)
    finally:
        assert fb.fa_set_wait_limit_ns(prev) == 1000
        fb.fa_select_fwd_kernel(sel)
    assert rc == fb.FA_ERR_TIMEOUT
    assert fb.fa_device_status(None) == 0       # cleared by the read
    q2, k2, v2 = (t[:, :2].contiguous() for t in (q, k, v))
    o, lse = _run(q2, k2, v2, 1.0 / math.sqrt(128), mk, -1, -1, True)
    ro, rlse = _ref(q2, k2, v2, 1.0 / math.sqrt(128), mk, -1, -1)
    _check(o, lse, ro, rlse, dtype, True, "after the kernel's own timeout")


# --------------------------------------------- full-size benchmark workloads

FULL = ["f16_full_4k", "f16_causal_4k", "bf16_causal_4k", "bf16_full_4k", "bf16_window_16k"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_heads(name):
    """The benchmark shapes in the benchmark's launch configuration; the
    oracle checks whole heads (first, middle, last) and, for the others, a
    strided sample of rows computed one block at a time."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    window = (w.win_l, w.win_r) if w.mask == MASK_WINDOW else None
    o, lse = fa.attention_fwd(dq, dk, dv, scale=w.scale, causal=w.mask == MASK_CAUSAL, window=window)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    heads = [(0, 0), (w.B // 2, w.H // 2), (w.B - 1, w.H - 1)]
    for b, h in heads:
        ro, rlse = _ref(q, k, v, w.scale, w.mask, w.win_l, w.win_r, heads=(b, h))
        _check(o[b:b + 1, h:h + 1].astype(np.float64), lse[b:b + 1, h:h + 1].astype(np.float64), ro, rlse,
               w.dtype, False, f"{name} head {(b, h)}")
    rng = np.random.default_rng(0)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    for _ in range(6):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        r0 = int(rng.integers(0, w.N - 64))
        ro, rlse = attention_three_pass(qd[b:b + 1, h:h + 1, r0:r0 + 64], kd[b:b + 1, h:h + 1],
                                        vd[b:b + 1, h:h + 1], w.scale, w.mask, w.win_l, w.win_r, q_offset=r0)
        _check(o[b:b + 1, h:h + 1, r0:r0 + 64].astype(np.float64), lse[b:b + 1, h:h + 1, r0:r0 + 64].astype(np.float64),
               ro, rlse, w.dtype, False, f"{name} rows {r0}.. of head {(b, h)}")


@pytest.mark.parametrize("name", FULL)
def test_full_size_raw_bound_with_fp32_o(name):
    """The raw bounds, max|dO| <= 2e-3 and max|dLSE| <= 1e-3, with no allowance
    for the rounding of O: the same kernel writes O in fp32 (only the store
    type of the epilogue differs from the 16-bit run).  Every (b, h) of the
    4,096-key workloads is compared in full; the 16,384-key window workload
    compares four whole heads (first, two inside, last) and the first rows
    of every other head, where rows see the fewest keys and |O| is largest.
    The worst (b, h, i) of each quantity is printed."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    window = (w.win_l, w.win_r) if w.mask == MASK_WINDOW else None
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.mask == MASK_CAUSAL,
                              window=window, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o = o.cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    if w.N <= 4096:
        blocks = [(b, h, 0, w.N) for b in range(w.B) for h in range(w.H)]
    else:
        whole = {(0, 0), (0, w.H // 3), (0, 2 * w.H // 3), (w.B - 1, w.H - 1)}
        blocks = [(b, h, 0, w.N) for b, h in sorted(whole)]
        blocks += [(b, h, 0, 512) for b in range(w.B) for h in range(w.H) if (b, h) not in whole]
    worst_o = (0.0, None)
    worst_l = (0.0, None)
    for b, h, r0, r1 in blocks:
        ro, rlse = attention_three_pass(qd[b:b + 1, h:h + 1, r0:r1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                        w.scale, w.mask, w.win_l, w.win_r, q_offset=r0)
        eo = np.abs(o[b, h, r0:r1] - ro[0, 0])
        el = np.abs(lse[b, h, r0:r1] - rlse[0, 0])
        i, d = np.unravel_index(np.argmax(eo), eo.shape)
        if eo[i, d] > worst_o[0]:
            worst_o = (float(eo[i, d]), (b, h, r0 + int(i), int(d)))
        il = int(np.argmax(el))
        if el[il] > worst_l[0]:
            worst_l = (float(el[il]), (b, h, r0 + il))
    print(f"{name} fp32 O: max|dO| = {worst_o[0]:.3e} at (b, h, i, d) = {worst_o[1]}; "
          f"max|dLSE| = {worst_l[0]:.3e} at (b, h, i) = {worst_l[1]}; {len(blocks)} row blocks")
    assert worst_o[0] <= TOL_O_16, f"{name}: max|dO| {worst_o[0]:.3e} at {worst_o[1]}"
    assert worst_l[0] <= TOL_LSE_16, f"{name}: max|dLSE| {worst_l[0]:.3e} at {worst_l[1]}"


# ------------------------------------------- layouts and grouped K/V heads

def _to_bhnd(x, layout):
    return x if layout == "bhnd" else x.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
@pytest.mark.parametrize("Hkv", [6, 3, 1])
@pytest.mark.parametrize("D,N", [(64, 300), (128, 129), (128, 512)])
def test_layouts_and_grouped_heads(dtype, layout, Hkv, D, N):
    from oracle import attention_grouped
    B, H = 2, 6
    q, _, _ = make_qkv(B, H, N, D, dtype, seed=500 + Hkv)
    _, k, v = make_qkv(B, Hkv, N, D, dtype, seed=600 + Hkv)
    if layout == "bnhd":
        q, k, v = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))
    for mk, wl, wr in [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 70, 3)]:
        window = (wl, wr) if mk == MASK_WINDOW else None
        o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=0.1, causal=mk == MASK_CAUSAL, window=window,
                                  o_dtype=torch.float32, layout=layout)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        assert o.shape == q.shape and lse.shape == (B, H, N)
        ro, rlse = attention_grouped(_to_bhnd(q, layout).double().numpy(), _to_bhnd(k, layout).double().numpy(),
                                     _to_bhnd(v, layout).double().numpy(), 0.1, mk, wl, wr)
        _check(_to_bhnd(o.cpu(), layout).numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rlse,
               dtype, True, f"{layout} Hkv={Hkv} D={D} N={N} mask={mk}")


def test_bnhd_benchmark_shape_sampled():
    """[B, N, H, D] input at the benchmark size (no transposing copy) with
    GQA 32 -> 8, checked on sampled heads."""
    from oracle import attention_grouped
    B, N, H, Hkv, D = 4, 4096, 32, 8, 128
    q, _, _ = make_qkv(B, H, N, D, "f16", seed=700)
    _, k, v = make_qkv(B, Hkv, N, D, "f16", seed=701)
    qb, kb, vb = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))
    o, lse = fa.attention_fwd(qb.cuda(), kb.cuda(), vb.cuda(), causal=True, layout="bnhd")
    torch.cuda.synchronize()
    o = o.float().cpu().permute(0, 2, 1, 3).numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    for b, h in [(0, 0), (1, 13), (3, 31)]:
        ro, rlse = attention_grouped(q[b:b + 1, h:h + 1].double().numpy(),
                                     k[b:b + 1, h // 4:h // 4 + 1].double().numpy(),
                                     v[b:b + 1, h // 4:h // 4 + 1].double().numpy(), 1 / math.sqrt(D), MASK_CAUSAL)
        _check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ro, rlse, "f16", False, f"bnhd gqa head {(b, h)}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,N", [(64, 512), (128, 640)])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
def test_unmasked_build_equals_masked_build(dtype, D, N, layout):
    """A problem with no mask, whole key tiles and N >= 512 runs the kernel
    build without mask and split-P code; a window wider than the sequence
    selects the full build yet leaves every key visible and every row with
    N keys.  Both compute the same sums in the same order: bit-equal O and
    LSE, and both match the oracle."""
    from oracle import attention_grouped
    q, k, v = make_qkv(2, 6, N, D, dtype, seed=N + D)
    k, v = k[:, ::2].contiguous(), v[:, ::2].contiguous()  # grouped heads, 6 -> 3
    perm = (lambda t: t.permute(0, 2, 1, 3).contiguous()) if layout == "bnhd" else (lambda t: t)
    outs = []
    for window in (None, (N, N)):
        o, lse = fa.attention_fwd(perm(q).cuda(), perm(k).cuda(), perm(v).cuda(), scale=1.0 / math.sqrt(D),
                                  window=window, layout=layout)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        outs.append((o.cpu(), lse.cpu()))
    assert fb.fa_geom_needs_masks(N, MASK_NONE, -1, -1) == 0
    assert fb.fa_geom_needs_masks(N, MASK_WINDOW, N, N) == 1
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    back = (lambda t: t.permute(0, 2, 1, 3)) if layout == "bnhd" else (lambda t: t)
    o = back(outs[0][0]).float().numpy().astype(np.float64)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    ro, rlse = attention_grouped(qd, kd, vd, 1.0 / math.sqrt(D), MASK_NONE, -1, -1)
    _check(o, outs[0][1].numpy().astype(np.float64), ro, rlse, dtype, False, f"unmasked build {dtype} D={D}")


def test_gqa_rejects_bad_head_counts():
    q = torch.zeros(1, 6, 64, 64, dtype=torch.float16, device="cuda")
    p = q.data_ptr()
    assert fb.fa_fwd_gqa(p, p, p, p, None, 1, 6, 4, 64, 64, 0.1, 0, -1, -1, fb.FA_F16, fb.FA_F16, 0, None) == fb.FA_ERR_ARG
    assert fb.fa_fwd_gqa(p, p, p, p, None, 1, 6, 7, 64, 64, 0.1, 0, -1, -1, fb.FA_F16, fb.FA_F16, 0, None) == fb.FA_ERR_ARG
    assert fb.fa_fwd_gqa(p, p, p, p, None, 1, 6, 3, 64, 64, 0.1, 0, -1, -1, fb.FA_F16, fb.FA_F16, 2, None) == fb.FA_ERR_ARG


@pytest.mark.parametrize("name", ["f16_full_4k", "bf16_causal_4k"])
def test_full_size_every_head(name):
    """The benchmark shape compared in full: every (b, h) of O and LSE against
    the oracle, one head at a time (about 0.35 s of float64 work per head on
    16 host cores).  The 16k-key window configuration keeps the sampled test
    above: its oracle materialises whole 16,384-key score rows, minutes of
    host time per pass."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    window = (w.win_l, w.win_r) if w.mask == MASK_WINDOW else None
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.mask == MASK_CAUSAL,
                              window=window)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    for b in range(w.B):
        for h in range(w.H):
            ro, rlse = attention_three_pass(qd[b:b + 1, h:h + 1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                            w.scale, w.mask, w.win_l, w.win_r)
            _check(o[b:b + 1, h:h + 1].astype(np.float64), lse[b:b + 1, h:h + 1].astype(np.float64), ro, rlse,
                   w.dtype, False, f"{name} head {(b, h)}")


@pytest.mark.parametrize("dtype,D,N,mk,wl,wr", [
    ("bf16", 128, 65536, MASK_CAUSAL, -1, -1),
    ("f16", 128, 65536, MASK_WINDOW, 4096, 0),
    ("f16", 64, 32768, MASK_NONE, -1, -1),
])
def test_long_sequences_sampled_rows(dtype, D, N, mk, wl, wr):
    """Long sequences (row and tile indices far past 2^16): the first, last and
    strided rows of two heads against the oracle computed row block by row block."""
    B, H = 1, 2
    q, k, v = make_qkv(B, H, N, D, dtype, seed=N + D)
    scale = 1.0 / math.sqrt(D)
    window = (wl, wr) if mk == MASK_WINDOW else None
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=mk == MASK_CAUSAL, window=window)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    for h in range(H):
        for r0 in (0, 13 * 1021, N // 2 + 7, N - 64):
            ro, rlse = attention_three_pass(qd[:, h:h + 1, r0:r0 + 64], kd[:, h:h + 1], vd[:, h:h + 1], scale, mk,
                                            wl, wr, q_offset=r0)
            _check(o[:, h:h + 1, r0:r0 + 64].astype(np.float64), lse[:, h:h + 1, r0:r0 + 64].astype(np.float64),
                   ro, rlse, dtype, False, f"N={N} head {h} rows {r0}..")


# ------------------------------------------------- the CTA-pair forward kernel

@pytest.fixture
def pair_kernel():
    prev = fb.fa_select_fwd_kernel(fb.FA_FWD_CTA_PAIR)
    yield
    fb.fa_select_fwd_kernel(prev)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 255, 256, 640, 1000])
def test_pair_kernel_ragged_all_masks(pair_kernel, dtype, N):
    """The 2-CTA kernel (M = 256 products over an SM pair, each CTA holding
    half of every K and V tile, three S buffers) meets the same bounds on
    ragged lengths and every mask, with O in fp32 and in the input type."""
    q, k, v = make_qkv(2, 3, N, 128, dtype, seed=9000 + N)
    for mk, wl, wr in MASK_SET:
        for o_f32 in (True, False):
            o, lse = _run(q, k, v, 0.088, mk, wl, wr, o_f32)
            ro, rlse = _ref(q, k, v, 0.088, mk, wl, wr)
            _check(o, lse, ro, rlse, dtype, o_f32, f"pair {dtype} N={N} mask={mk},{wl},{wr} o_f32={o_f32}")


@pytest.mark.parametrize("name", ["f16_full_4k", "bf16_causal_4k", "bf16_window_16k"])
def test_pair_kernel_full_size_raw_bound(pair_kernel, name):
    """Benchmark shapes on the 2-CTA kernel, fp32 O, raw bounds on sampled
    heads and row blocks (the first rows, where |O| is largest, included)."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    window = (w.win_l, w.win_r) if w.mask == MASK_WINDOW else None
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.mask == MASK_CAUSAL,
                              window=window, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o = o.cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    for b, h, r0, r1 in ((0, 0, 0, 512), (w.B - 1, w.H - 1, w.N - 512, w.N), (w.B // 2, w.H // 2, 1000, 1512)):
        ro, rlse = attention_three_pass(qd[b:b + 1, h:h + 1, r0:r1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                        w.scale, w.mask, w.win_l, w.win_r, q_offset=r0)
        assert np.abs(o[b, h, r0:r1] - ro[0, 0]).max() <= TOL_O_16, (name, b, h, r0)
        assert np.abs(lse[b, h, r0:r1] - rlse[0, 0]).max() <= TOL_LSE_16, (name, b, h, r0)


def test_pair_kernel_layouts_gqa_and_rope(pair_kernel):
    """[B, N, H, D] input and grouped K/V heads on the 2-CTA kernel against the
    oracle, and the rotary embedding of Q (rotated by that kernel's Q-release
    warps) bit-equal to the two-pass path."""
    from oracle import attention_grouped
    B, H, Hkv, N, D = 2, 4, 2, 300, 128
    q, _, _ = make_qkv(B, H, N, D, "bf16", seed=77)
    _, k, v = make_qkv(B, Hkv, N, D, "bf16", seed=78)
    qb, kb, vb = (t.permute(0, 2, 1, 3).contiguous().cuda() for t in (q, k, v))
    o, lse = fa.attention_fwd(qb, kb, vb, causal=True, layout="bnhd", o_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rlse = attention_grouped(q.double().numpy(), k.double().numpy(), v.double().numpy(), 1 / math.sqrt(D),
                                 MASK_CAUSAL)
    _check(o.cpu().permute(0, 2, 1, 3).numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rlse,
           "bf16", True, "pair bnhd gqa")
    cos, sin = fa.rope_tables(N + 9, D, 10000.0)
    _, kr = fa.apply_rope(None, kb, cos, sin, k_pos0=9, layout="bnhd")
    qr, _ = fa.apply_rope(qb, None, cos, sin, q_pos0=9, layout="bnhd")
    o1, l1 = fa.attention_fwd(qb, kr, vb, layout="bnhd", rope=(cos, sin), rope_pos0=9)
    o2, l2 = fa.attention_fwd(qr, kr, vb, layout="bnhd")
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_kernel_selector_rejects_unknown_values():
    assert fb.fa_select_fwd_kernel(7) == fb.FA_ERR_ARG
    prev = fb.fa_select_fwd_kernel(fb.FA_FWD_AUTO)
    assert fb.fa_select_fwd_kernel(prev) == fb.FA_FWD_AUTO
