"""Host-side checks that need no GPU: the library builds, loads and exports
every symbol of include/fa.h; argument validation; the tile planner and the
mask-free-tile predicate against the oracle's mask; the FLOP count against
the oracle's pair count."""

import ctypes
import os
import re

import numpy as np
import pytest

from attention_forward_16_gb300 import binding as fb
from attention_forward_16_gb300 import flops
from oracle import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, allowed_mask, unmasked_pairs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_16_gb300.build import build
    build()
    return fb.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_ ]+\**\s*\**(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_method_entry_points():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_fwd_f16", "fa_fwd_bf16", "fa_fwd_f32", "fa_fwd_ex", "fa_device_status",
              "fa_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"libfa.so does not export {n}"
    assert set(names) == set(fb.SIGNATURES), "binding signatures out of sync with include/fa.h"


def test_version_and_strerror(lib):
    assert lib.fa_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6, 7):
        assert lib.fa_strerror(code)


# ----------------------------------------------------- validation, no launch

def _call(lib, q=16, k=16, v=16, o=16, lse=None, B=1, H=1, N=8, D=64, scale=0.1, mk=0, wl=-1, wr=-1, dt=0, odt=None):
    return lib.fa_fwd_ex(q, k, v, o, lse, B, H, N, D, scale, mk, wl, wr, dt, dt if odt is None else odt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fb.FA_ERR_ARG),
    (dict(o=None), fb.FA_ERR_ARG),
    (dict(B=0), fb.FA_ERR_ARG),
    (dict(H=-1), fb.FA_ERR_ARG),
    (dict(N=0), fb.FA_ERR_ARG),
    (dict(scale=float("nan")), fb.FA_ERR_ARG),
    (dict(scale=float("inf")), fb.FA_ERR_ARG),
    (dict(mk=3), fb.FA_ERR_ARG),
    (dict(mk=2, wl=-2), fb.FA_ERR_ARG),
    (dict(mk=2, wr=-5), fb.FA_ERR_ARG),
    (dict(B=1 << 20, H=1 << 12), fb.FA_ERR_ARG),
    (dict(D=96), fb.FA_ERR_UNSUPPORTED),
    (dict(D=256, dt=1), fb.FA_ERR_UNSUPPORTED),
    (dict(D=129, dt=2), fb.FA_ERR_UNSUPPORTED),
    (dict(dt=5), fb.FA_ERR_UNSUPPORTED),
    (dict(dt=0, odt=1), fb.FA_ERR_UNSUPPORTED),
    (dict(dt=2, odt=0), fb.FA_ERR_UNSUPPORTED),
    (dict(q=24), fb.FA_ERR_ALIGN),
    (dict(o=8), fb.FA_ERR_ALIGN),
    (dict(lse=2), fb.FA_ERR_ALIGN),
])
def test_validation_rejects_before_any_launch(lib, kw, code):
    assert _call(lib, **kw) == code


# ----------------------------------------------------------- tile planning

PLAN_CASES = [
    (1, 300, MASK_NONE, -1, -1),
    (2, 513, MASK_CAUSAL, -1, -1),
    (1, 1, MASK_CAUSAL, -1, -1),
    (1, 129, MASK_WINDOW, 37, 5),
    (1, 1000, MASK_WINDOW, 200, 0),
    (1, 700, MASK_WINDOW, 0, 0),
    (1, 640, MASK_WINDOW, -1, 3),
    (1, 650, MASK_WINDOW, 130, -1),
    (1, 2048, MASK_WINDOW, 1024, 0),
]


@pytest.mark.parametrize("BH,N,mk,wl,wr", PLAN_CASES)
def test_plan_covers_exactly_the_visible_pairs(lib, BH, N, mk, wl, wr):
    units = fb.fa_plan_units(1, BH, N, mk, wl, wr)
    ok = allowed_mask(N, N, mk, wl, wr)
    seen_rows = {}
    for (bh, q0, lo0, hi0, lo1, hi1) in units:
        for t, (lo, hi) in enumerate(((lo0, hi0), (lo1, hi1))):
            r0 = q0 + 128 * t
            if r0 >= N:
                assert lo == hi
                continue
            r1 = min(N, r0 + 128)
            assert 0 <= lo < hi <= (N + 127) // 128
            for r in range(r0, r1):
                seen_rows[(bh, r)] = seen_rows.get((bh, r), 0) + 1
            rows = ok[r0:r1]
            # every visible key of these rows lies in a visited tile ...
            cols = np.nonzero(rows.any(axis=0))[0]
            assert cols.min() >= lo * 128 and cols.max() < hi * 128
            # ... and the first and last visited tiles hold at least one
            assert rows[:, lo * 128:(lo + 1) * 128].any() and rows[:, (hi - 1) * 128:hi * 128].any()
    assert len(seen_rows) == BH * N and set(seen_rows.values()) == {1}


@pytest.mark.parametrize("BH,N,mk,wl,wr", PLAN_CASES)
def test_tiles_without_mask_are_fully_visible(lib, BH, N, mk, wl, wr):
    ok = allowed_mask(N, N, mk, wl, wr)
    nt = (N + 127) // 128
    for r0 in range(0, N, 128):
        r1 = min(N, r0 + 128)
        for j in range(nt):
            block = ok[r0:r1, j * 128:min(N, (j + 1) * 128)]
            need = fb.fa_tile_needs_mask(N, mk, wl, wr, r0, j)
            assert need in (0, 1)
            if not need:
                assert block.all() and (j + 1) * 128 <= N


@pytest.mark.parametrize("N,mk,wl,wr,expect", [
    (512, MASK_NONE, -1, -1, 0), (4096, MASK_NONE, -1, -1, 0), (1024, MASK_WINDOW, -1, -1, 0),
    (384, MASK_NONE, -1, -1, 1),      # rows see fewer than 512 keys: bf16 split P
    (640 + 5, MASK_NONE, -1, -1, 1),  # ragged last key tile
    (1024, MASK_CAUSAL, -1, -1, 1), (1024, MASK_WINDOW, 100, -1, 1), (1024, MASK_WINDOW, -1, 0, 1),
    (1024, MASK_WINDOW, 2000, 2000, 1),
])
def test_unmasked_build_only_for_problems_without_masks(lib, N, mk, wl, wr, expect):
    # The forward kernel's build without mask and split-P paths is taken only
    # where every tile is fully visible and every row sees at least 512 keys.
    got = fb.fa_geom_needs_masks(N, mk, wl, wr)
    assert got == expect
    if got == 0:
        ok = allowed_mask(N, N, mk, wl, wr)
        assert ok.all() and N % 128 == 0 and N >= 512
        nt = N // 128
        for r0 in range(0, N, 128):
            for j in range(nt):
                assert fb.fa_tile_needs_mask(N, mk, wl, wr, r0, j) == 0
    assert fb.fa_geom_needs_masks(N, 7, wl, wr) < 0  # bad mask kind


def test_unit_order_is_longest_first_for_causal(lib):
    units = fb.fa_plan_units(2, 3, 1024, MASK_CAUSAL)
    work = [(hi0 - lo0) + (hi1 - lo1) for (_, _, lo0, hi0, lo1, hi1) in units]
    assert work == sorted(work, reverse=True)


def test_causal_units_come_in_head_groups(lib):
    # N = 4096: groups of 32 heads (a group's K/V, 2 MB a head, fits half of
    # L2), each group longest first; 4 x 32 = 128 heads make four groups, the
    # last one short when the heads do not divide evenly
    for B, H in ((4, 32), (3, 25)):
        units = fb.fa_plan_units(B, H, 4096, MASK_CAUSAL)
        BH, per_head = B * H, 16
        assert len(units) == BH * per_head
        start = 0
        for g0 in range(0, BH, 32):
            gh = min(32, BH - g0)
            grp = units[start:start + gh * per_head]
            start += gh * per_head
            assert {u[0] for u in grp} == set(range(g0, g0 + gh))
            work = [(hi0 - lo0) + (hi1 - lo1) for (_, _, lo0, hi0, lo1, hi1) in grp]
            assert work == sorted(work, reverse=True)
        assert start == len(units)


# ------------------------------------------------------------- FLOP count

@pytest.mark.parametrize("N", [1, 2, 7, 128, 129, 1000])
@pytest.mark.parametrize("mk,wl,wr", [(MASK_NONE, -1, -1), (MASK_CAUSAL, -1, -1), (MASK_WINDOW, 5, 0),
                                      (MASK_WINDOW, 0, 3), (MASK_WINDOW, 40, 17), (MASK_WINDOW, -1, 2),
                                      (MASK_WINDOW, 3, -1), (MASK_WINDOW, 0, 0)])
def test_pair_count_matches_oracle_mask(N, mk, wl, wr):
    assert flops.unmasked_pairs(N, mk, wl, wr) == unmasked_pairs(N, mk, wl, wr)


def test_flops_of_the_benchmark_shapes():
    assert flops.attention_flops(4, 32, 4096, 128, MASK_NONE) == 2 ** 40
    assert flops.attention_flops(4, 32, 4096, 128, MASK_CAUSAL) == 549_890_031_616
    assert flops.attention_flops(1, 64, 16384, 128, MASK_WINDOW, 1024, 0) == 533_096_038_400
    assert flops.attention_flops(2, 8, 1024, 64, MASK_CAUSAL) == 2_149_580_800
    assert flops.algorithmic_bytes(4, 32, 4096, 128, "f16") == 538_968_064


# ------------------------------------------------------ decode: host checks

def _dec(lib, q=16, k=16, v=16, o=16, B=1, H=1, Nq=1, Nk=8, D=64, scale=0.1, mk=0, wl=-1, wr=-1, dt=0, ns=0,
         ws=None, wb=0):
    return lib.fa_decode(q, k, v, o, None, B, H, Nq, Nk, D, scale, mk, wl, wr, dt, ns, ws, wb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fb.FA_ERR_ARG),
    (dict(Nq=0), fb.FA_ERR_ARG),
    (dict(Nq=9, Nk=8), fb.FA_ERR_ARG),
    (dict(scale=float("nan")), fb.FA_ERR_ARG),
    (dict(mk=2, wl=-3), fb.FA_ERR_ARG),
    (dict(Nq=17, Nk=40), fb.FA_ERR_UNSUPPORTED),
    (dict(D=96), fb.FA_ERR_UNSUPPORTED),
    (dict(dt=3), fb.FA_ERR_UNSUPPORTED),
    (dict(k=24), fb.FA_ERR_ALIGN),
])
def test_decode_validation_rejects_before_any_launch(lib, kw, code):
    assert _dec(lib, **kw) == code


def test_decode_plan_arithmetic():
    """The split plan covers every key exactly once with chunks of 4-key groups."""
    # a Python restatement of the plan, checked against its coverage contract
    for BH, Nk, sms, req in [(1, 1, 152, 0), (8, 32768, 152, 0), (256, 4096, 152, 0), (1, 5000, 152, 4),
                             (2, 3000, 148, 100), (1, 65536, 152, 300), (4, 7, 152, 5)]:
        ns, chunk = _plan(BH, Nk, sms, req)
        assert chunk % 4 == 0 and ns >= 1
        assert (ns - 1) * chunk < Nk <= ns * chunk
        if req <= 0 and Nk >= 256:
            assert chunk >= 256 or ns == 1 or BH * ns >= 8 * sms


def _plan(BH, Nk, sms, req):
    s = req if req > 0 else -(-8 * sms // BH)
    cap = -(-Nk // 256)
    if req <= 0 and s > cap:
        s = cap
    s = max(1, min(s, Nk, 1024))
    c = -(-Nk // s)
    c = -(-c // 4) * 4
    return -(-Nk // c), c


# --------------------------------------------------------- RoPE: host checks

def _rope(lib, q=16, k=32, qo=48, ko=64, cos=80, sin=96, B=1, H=2, Hkv=1, Nq=4, Nk=4, D=64, qp=0, kp=0, n_pos=8,
          st=0, dt=0, lay=0):
    return lib.fa_rope(q, k, qo, ko, cos, sin, B, H, Hkv, Nq, Nk, D, qp, kp, n_pos, st, dt, lay, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None, k=None, qo=None, ko=None), fb.FA_ERR_ARG),
    (dict(q=None), fb.FA_ERR_ARG),              # out given without its input
    (dict(ko=None), fb.FA_ERR_ARG),
    (dict(cos=None), fb.FA_ERR_ARG),
    (dict(B=0), fb.FA_ERR_ARG),
    (dict(D=40), fb.FA_ERR_ARG),                 # not a multiple of 16
    (dict(D=2048), fb.FA_ERR_ARG),
    (dict(st=2), fb.FA_ERR_ARG),
    (dict(lay=3), fb.FA_ERR_ARG),
    (dict(qp=5), fb.FA_ERR_ARG),                 # rows 5..8 leave an 8-row table
    (dict(kp=-1), fb.FA_ERR_ARG),
    (dict(Nk=9), fb.FA_ERR_ARG),
    (dict(Hkv=0), fb.FA_ERR_ARG),
    (dict(dt=3), fb.FA_ERR_UNSUPPORTED),
    (dict(q=24), fb.FA_ERR_ALIGN),
    (dict(ko=8), fb.FA_ERR_ALIGN),
    (dict(sin=100), fb.FA_ERR_ALIGN),
])
def test_rope_validation_rejects_before_any_launch(lib, kw, code):
    assert _rope(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(n_pos=0), fb.FA_ERR_ARG),
    (dict(D=7), fb.FA_ERR_ARG),
    (dict(base=0.0), fb.FA_ERR_ARG),
    (dict(base=float("inf")), fb.FA_ERR_ARG),
    (dict(cos=None), fb.FA_ERR_ARG),
    (dict(cos=20), fb.FA_ERR_ALIGN),
])
def test_rope_tables_validation(lib, kw, code):
    a = dict(cos=16, sin=32, n_pos=4, D=8, base=10000.0)
    a.update(kw)
    assert lib.fa_rope_tables(a["cos"], a["sin"], a["n_pos"], a["D"], a["base"], None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), fb.FA_ERR_ARG),
    (dict(ps=24), fb.FA_ERR_ARG),              # not a power of two
    (dict(max_pages=1), fb.FA_ERR_ARG),        # 1 x 16 < max_seq_len 64
    (dict(num_pages=0), fb.FA_ERR_ARG),
    (dict(Hkv=3), fb.FA_ERR_ARG),
    (dict(D=96), fb.FA_ERR_UNSUPPORTED),
    (dict(table=18), fb.FA_ERR_ALIGN),
    (dict(k=24), fb.FA_ERR_ALIGN),
])
def test_paged_decode_validation(lib, kw, code):
    a = dict(q=16, k=32, v=48, table=64, lens=80, o=96, B=1, H=2, Hkv=1, Nq=1, max_seq=64, ps=16, max_pages=4,
             num_pages=8, D=64, dt=0)
    a.update(kw)
    rc = lib.fa_decode_paged(a["q"], a["k"], a["v"], a["table"], a["lens"], a["o"], None, a["B"], a["H"], a["Hkv"],
                             a["Nq"], a["max_seq"], a["ps"], a["max_pages"], a["num_pages"], a["D"], 0.1, 0, -1, -1,
                             a["dt"], 0, 0, None, 0, None)
    assert rc == code


def test_wait_limit_setter_floor_and_round_trip(lib):
    """The setter raises values below FA_MIN_WAIT_LIMIT_NS (1 us) to it and
    returns the previous limit; it only stores a host value, so this needs
    no GPU.  The kernels' final drain keeps its own 1 s bound whatever is set."""
    floor = 1000
    text = open(HEADER).read()
    assert re.search(r"#define\s+FA_MIN_WAIT_LIMIT_NS\s+1000ull", text)
    before = lib.fa_set_wait_limit_ns(0)
    try:
        assert lib.fa_set_wait_limit_ns(1) == floor          # 0 was raised to the floor
        assert lib.fa_set_wait_limit_ns(floor - 1) == floor  # so was 1
        assert lib.fa_set_wait_limit_ns(5_000_000) == floor
        assert lib.fa_set_wait_limit_ns(7) == 5_000_000      # values at or above the floor are kept
    finally:
        lib.fa_set_wait_limit_ns(before)
    assert lib.fa_set_wait_limit_ns(before) == before


def test_fwd_rope_rejections_before_any_launch(lib):
    """fa_fwd_rope validates its table arguments before touching a device."""
    def call(cos=16, sin=16, n_pos=100, pos0=0, style=0, N=8, dt=0, q=16):
        return lib.fa_fwd_rope(q, 16, 16, 16, None, cos, sin, n_pos, pos0, style, 1, 1, 1, N, 64, 0.1, 0, -1, -1,
                               dt, dt, 0, None)
    assert call(cos=None) == fb.FA_ERR_ARG
    assert call(sin=None) == fb.FA_ERR_ARG
    assert call(n_pos=0) == fb.FA_ERR_ARG
    assert call(pos0=-1) == fb.FA_ERR_ARG
    assert call(pos0=95, N=8) == fb.FA_ERR_ARG          # rows 95 .. 102 run past the 100-entry table
    assert call(style=2) == fb.FA_ERR_ARG
    assert call(cos=8) == fb.FA_ERR_ALIGN
    assert call(dt=2) == fb.FA_ERR_UNSUPPORTED          # the fp32 kernel has no in-kernel rotation
    assert call(q=None) == fb.FA_ERR_ARG                # then the forward's own checks


def test_forward_kernel_selector_is_host_only(lib):
    """fa_select_fwd_kernel only records the choice (no device needed) and
    refuses values that name no kernel."""
    prev = lib.fa_select_fwd_kernel(fb.FA_FWD_CTA_PAIR)
    try:
        assert lib.fa_select_fwd_kernel(fb.FA_FWD_ONE_CTA) == fb.FA_FWD_CTA_PAIR
        assert lib.fa_select_fwd_kernel(3) == fb.FA_ERR_ARG
        assert lib.fa_select_fwd_kernel(-1) == fb.FA_ERR_ARG
        assert lib.fa_select_fwd_kernel(fb.FA_FWD_AUTO) == fb.FA_FWD_ONE_CTA
    finally:
        lib.fa_select_fwd_kernel(prev)
