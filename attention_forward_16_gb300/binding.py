"""ctypes binding over libfa.so: argument marshalling only.

The functions named like the C ABI (``fa_fwd``, ``fa_fwd_f16`` ...) take raw
pointers and sizes exactly as ``include/fa.h`` declares them.
:func:`attention_fwd` is the tensor-level convenience: it checks shapes,
allocates O and LSE with torch on the inputs' device and calls ``fa_fwd_ex``
on the current stream.  Every step of the computation runs in libfa's CUDA
kernels; there is no other implementation to fall back to, and a missing
library raises.
"""

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_MASK_NONE, FA_MASK_CAUSAL, FA_MASK_WINDOW = 0, 1, 2
FA_LAYOUT_BHND, FA_LAYOUT_BNHD = 0, 1
_LAYOUT_CODE = {"bhnd": FA_LAYOUT_BHND, "bnhd": FA_LAYOUT_BNHD}
FA_F16, FA_BF16, FA_F32 = 0, 1, 2
FA_OK, FA_ERR_ARG, FA_ERR_UNSUPPORTED, FA_ERR_ALIGN, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6
FA_ERR_SCRATCH = -7
FA_ROPE_HALF, FA_ROPE_INTERLEAVED = 0, 1
_ROPE_STYLE = {"half": FA_ROPE_HALF, "interleaved": FA_ROPE_INTERLEAVED}

_DTYPE_CODE = {torch.float16: FA_F16, torch.bfloat16: FA_BF16, torch.float32: FA_F32}

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

# name -> (restype, argtypes), mirroring include/fa.h
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _I, _P]),
    "fa_fwd_f16": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_fwd_bf16": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_fwd_f32": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _I, _P]),
    "fa_decode_plan": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _P, ctypes.c_ulonglong, _P]),
    "fa_decode_plan_gqa": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_decode_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _I, _P,
                           ctypes.c_ulonglong, _P]),
    "fa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I,
                             _I, _I, _P, ctypes.c_ulonglong, _P]),
    "fa_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _P]),
    "fa_decode_noalloc_scratch_bytes": (ctypes.c_ulonglong, []),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _P,
                    ctypes.c_ulonglong, _P]),
    "fa_bwd_workspace_bytes": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_rope": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "fa_rope_tables": (_I, [_P, _P, _I, _I, ctypes.c_double, _P]),
    "fa_fwd_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _I,
                         _P]),
    "fa_device_status": (_I, [_P]),
    "fa_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "fa_select_fwd_kernel": (_I, [_I]),
    "fa_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "fa_plan_units": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), _I]),
    "fa_tile_needs_mask": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_geom_needs_masks": (_I, [_I, _I, _I, _I]),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_last_cuda_error": (ctypes.c_char_p, []),
    "fa_version": (_I, []),
}

_lib = None


class FaError(RuntimeError):
    def __init__(self, code, where):
        lib = load()
        msg = lib.fa_strerror(code).decode()
        if code == FA_ERR_CUDA:
            msg += ": " + lib.fa_last_cuda_error().decode()
        super().__init__(f"{where} returned {code} ({msg})")
        self.code = code


def load(path=None):
    """Load libfa.so (built by ``attention_forward_16_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libfa.so is not built ({p}); run attention_forward_16_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc, where):
    if rc != FA_OK:
        raise FaError(rc, where)
    return rc


# ---------------------------------------------------------------- raw C ABI

def fa_fwd(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, stream):
    return load().fa_fwd(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, stream)


def fa_fwd_f16(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream):
    return load().fa_fwd_f16(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream)


def fa_fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream):
    return load().fa_fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream)


def fa_fwd_f32(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream):
    return load().fa_fwd_f32(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, stream)


def fa_fwd_ex(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, stream):
    return load().fa_fwd_ex(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, stream)


def fa_decode_plan(B, H, Nq, Nk, D, n_splits=0):
    """(n_splits, workspace_bytes) the decode of this shape uses on the current device."""
    ns = ctypes.c_int(0)
    wb = ctypes.c_ulonglong(0)
    _check(load().fa_decode_plan(B, H, Nq, Nk, D, n_splits, ctypes.byref(ns), ctypes.byref(wb)), "fa_decode_plan")
    return ns.value, wb.value


def fa_decode_plan_gqa(B, H, H_kv, Nq, Nk, D, n_splits=0):
    ns = ctypes.c_int(0)
    wb = ctypes.c_ulonglong(0)
    _check(load().fa_decode_plan_gqa(B, H, H_kv, Nq, Nk, D, n_splits, ctypes.byref(ns), ctypes.byref(wb)),
           "fa_decode_plan_gqa")
    return ns.value, wb.value


def fa_decode_gqa(q, k, v, o, lse, B, H, H_kv, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype, layout, n_splits,
                  workspace, workspace_bytes, stream):
    return load().fa_decode_gqa(q, k, v, o, lse, B, H, H_kv, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype,
                                layout, n_splits, workspace, workspace_bytes, stream)


def fa_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype, n_splits, workspace,
              workspace_bytes, stream):
    return load().fa_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype, n_splits,
                            workspace, workspace_bytes, stream)


def fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, H, H_kv, Nq, max_seq_len, page_size,
                    max_pages, num_pages, D, scale, mask_kind, win_l, win_r, dtype, layout, n_splits, workspace,
                    workspace_bytes, stream):
    return load().fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, H, H_kv, Nq, max_seq_len,
                                  page_size, max_pages, num_pages, D, scale, mask_kind, win_l, win_r, dtype, layout,
                                  n_splits, workspace, workspace_bytes, stream)


def fa_decode_noalloc(q, k, v, o, lse, B, H, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype, n_splits, stream):
    """fa_decode with the partial results in the library's fixed scratch array
    (for callers that must not allocate device memory)."""
    return load().fa_decode_noalloc(q, k, v, o, lse, B, H, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype,
                                    n_splits, stream)


def fa_decode_noalloc_scratch_bytes():
    return load().fa_decode_noalloc_scratch_bytes()


def fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, layout, stream):
    return load().fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype,
                             layout, stream)


def fa_bwd(q, k, v, o, d_o, lse, dq, dk, dv, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype, layout,
           workspace, workspace_bytes, stream):
    return load().fa_bwd(q, k, v, o, d_o, lse, dq, dk, dv, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype,
                         layout, workspace, workspace_bytes, stream)


def fa_bwd_workspace_bytes(B, H, N):
    """Workspace bytes fa_bwd needs; raises on bad sizes."""
    out = ctypes.c_ulonglong(0)
    _check(load().fa_bwd_workspace_bytes(B, H, N, ctypes.byref(out)), "fa_bwd_workspace_bytes")
    return out.value


def fa_rope(q, k, q_out, k_out, cos_tab, sin_tab, B, H, H_kv, Nq, Nk, D, q_pos0, k_pos0, n_pos, style, dtype,
            layout, stream):
    return load().fa_rope(q, k, q_out, k_out, cos_tab, sin_tab, B, H, H_kv, Nq, Nk, D, q_pos0, k_pos0, n_pos,
                          style, dtype, layout, stream)


def fa_fwd_rope(q, k, v, o, lse, cos_tab, sin_tab, n_pos, q_pos0, style, B, H, H_kv, N, D, scale, mask_kind, win_l,
                win_r, dtype, o_dtype, layout, stream):
    return load().fa_fwd_rope(q, k, v, o, lse, cos_tab, sin_tab, n_pos, q_pos0, style, B, H, H_kv, N, D, scale,
                              mask_kind, win_l, win_r, dtype, o_dtype, layout, stream)


def fa_rope_tables(cos_tab, sin_tab, n_pos, D, base, stream):
    return load().fa_rope_tables(cos_tab, sin_tab, n_pos, D, base, stream)


def fa_device_status(stream=None):
    return load().fa_device_status(stream)


FA_FWD_AUTO, FA_FWD_ONE_CTA, FA_FWD_CTA_PAIR = 0, 1, 2


def fa_select_fwd_kernel(which):
    return load().fa_select_fwd_kernel(which)


def fa_set_wait_limit_ns(ns):
    return load().fa_set_wait_limit_ns(ns)


def fa_selftest_wait_timeout(limit_ns, stream=None):
    return load().fa_selftest_wait_timeout(limit_ns, stream)


def fa_plan_units(B, H, N, mask_kind, win_l=-1, win_r=-1):
    """All work units as a list of (bh, q0, lo0, hi0, lo1, hi1)."""
    lib = load()
    n = lib.fa_plan_units(B, H, N, mask_kind, win_l, win_r, None, 0)
    _check(n if n < 0 else 0, "fa_plan_units")
    buf = (ctypes.c_int * (6 * n))()
    lib.fa_plan_units(B, H, N, mask_kind, win_l, win_r, buf, n)
    return [tuple(buf[6 * u:6 * u + 6]) for u in range(n)]


def fa_tile_needs_mask(N, mask_kind, win_l, win_r, r0, j):
    return load().fa_tile_needs_mask(N, mask_kind, win_l, win_r, r0, j)


def fa_geom_needs_masks(N, mask_kind, win_l, win_r):
    return load().fa_geom_needs_masks(N, mask_kind, win_l, win_r)


# ------------------------------------------------------------ tensor level

def mask_args(causal=False, window=None):
    """(mask_kind, win_l, win_r) from the user-level mask options."""
    if window is not None:
        if causal:
            raise ValueError("give either causal=True or window=(left, right), not both")
        wl, wr = window
        return FA_MASK_WINDOW, -1 if wl is None else int(wl), -1 if wr is None else int(wr)
    return (FA_MASK_CAUSAL, -1, -1) if causal else (FA_MASK_NONE, -1, -1)


def attention_fwd(q, k, v, scale=None, causal=False, window=None, o_dtype=None, out=None, lse=None,
                  stream=None, layout="bhnd", rope=None, rope_style="half", rope_pos0=0):
    """O, LSE = softmax(scale * Q K^T + mask) V for CUDA tensors.

    ``layout="bhnd"``: q [B, H, N, D], k and v [B, H_kv, N, D];
    ``layout="bnhd"``: q [B, N, H, D], k and v [B, N, H_kv, D].  H must be a
    multiple of H_kv (grouped-query attention when smaller).  O has q's shape,
    LSE is [B, H, N].  ``window=(left, right)`` selects the sliding window
    (None or -1 for an unbounded side); ``scale`` defaults to 1/sqrt(D);
    ``o_dtype=torch.float32`` returns O in fp32 for 16-bit inputs.  Runs on
    the current CUDA stream unless ``stream`` (a torch.cuda.Stream) is given.

    ``rope=(cos, sin)`` (fp32 [n_pos, D/2] tables, ``rope_tables``) rotates Q
    inside the kernel (``fa_fwd_rope``): query row i at position
    ``rope_pos0 + i``, pairing ``rope_style``.  K must already be rotated.
    """
    if layout not in _LAYOUT_CODE:
        raise ValueError(f"layout must be one of {sorted(_LAYOUT_CODE)}")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError(f"q, k, v must be 4-D with k and v alike, got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)}")
    if layout == "bhnd":
        B, H, N, D = q.shape
        Hkv = k.shape[1]
        ok_shape = k.shape[0] == B and k.shape[2] == N and k.shape[3] == D
    else:
        B, N, H, D = q.shape
        Hkv = k.shape[2]
        ok_shape = k.shape[0] == B and k.shape[1] == N and k.shape[3] == D
    if not ok_shape or Hkv < 1 or H % Hkv:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)} for layout {layout}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPE_CODE:
        raise ValueError("q, k, v must share one dtype among float16, bfloat16, float32")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    mk, wl, wr = mask_args(causal, window)
    od = q.dtype if o_dtype is None else o_dtype
    if out is None:
        out = torch.empty(q.shape, dtype=od, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    s = (stream or torch.cuda.current_stream(q.device)).cuda_stream
    if rope is not None:
        cos, sin = rope
        if rope_style not in _ROPE_STYLE:
            raise ValueError(f"rope_style must be one of {sorted(_ROPE_STYLE)}")
        if (cos.dtype != torch.float32 or sin.shape != cos.shape or cos.dim() != 2 or cos.shape[1] != D // 2
                or not (cos.is_cuda and sin.is_cuda and cos.is_contiguous() and sin.is_contiguous())):
            raise ValueError("rope tables must be contiguous fp32 CUDA tensors [n_pos, D/2] of one shape")
        with torch.cuda.device(q.device):
            rc = fa_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                             cos.data_ptr(), sin.data_ptr(), cos.shape[0], int(rope_pos0), _ROPE_STYLE[rope_style],
                             B, H, Hkv, N, D, float(scale), mk, wl, wr, _DTYPE_CODE[q.dtype], _DTYPE_CODE[od],
                             _LAYOUT_CODE[layout], s)
        _check(rc, "fa_fwd_rope")
        return out, lse
    with torch.cuda.device(q.device):
        rc = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, H, Hkv, N, D, float(scale), mk, wl, wr, _DTYPE_CODE[q.dtype], _DTYPE_CODE[od],
                        _LAYOUT_CODE[layout], s)
    _check(rc, "fa_fwd_gqa")
    return out, lse


def attention_decode(q, k, v, scale=None, causal=False, window=None, n_splits=0, out=None, lse=None,
                     workspace=None, stream=None, layout="bhnd"):
    """Decode: queries against a K/V cache.

    ``layout="bhnd"``: q [B, H, Nq, D], k and v [B, H_kv, Nk, D];
    ``layout="bnhd"``: q [B, Nq, H, D], k and v [B, Nk, H_kv, D].  H must be a
    multiple of H_kv and (H / H_kv) * Nq <= 16.  Query i sits at cache
    position Nk - Nq + i.  The split-K workspace is allocated with torch
    unless ``workspace`` (a CUDA uint8 tensor of at least the planned size) is
    given.  Returns (O, LSE), LSE [B, H, Nq]."""
    if layout not in _LAYOUT_CODE:
        raise ValueError(f"layout must be one of {sorted(_LAYOUT_CODE)}")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q, k, v must be 4-D with k and v alike")
    if layout == "bhnd":
        B, H, Nq, D = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
    else:
        B, Nq, H, D = q.shape
        Nk, Hkv = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != D or Hkv < 1 or H % Hkv:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)} for layout {layout}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPE_CODE:
        raise ValueError("q, k, v must share one dtype among float16, bfloat16, float32")
    if not (q.is_cuda and k.is_cuda and v.is_cuda and q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    mk, wl, wr = mask_args(causal, window)
    with torch.cuda.device(q.device):
        ns, wb = fa_decode_plan_gqa(B, H, Hkv, Nq, Nk, D, n_splits)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        if workspace is None and wb > 0:
            workspace = torch.empty(wb, dtype=torch.uint8, device=q.device)
        s = (stream or torch.cuda.current_stream(q.device)).cuda_stream
        rc = fa_decode_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq,
                           Nk, D, float(scale), mk, wl, wr, _DTYPE_CODE[q.dtype], _LAYOUT_CODE[layout], ns,
                           workspace.data_ptr() if workspace is not None else None,
                           workspace.numel() if workspace is not None else 0, s)
    _check(rc, "fa_decode_gqa")
    return out, lse


def attention_bwd(q, k, v, o, lse, d_o, scale=None, causal=False, window=None, layout="bhnd", dq=None, dk=None,
                  dv=None, workspace=None, stream=None):
    """dQ, dK, dV of attention_fwd for an upstream gradient ``d_o``.

    q, k, v, o, lse are the forward's inputs and outputs (O in the inputs'
    16-bit type), d_o has O's shape; the mask and scale must be the forward's.
    The gradients are allocated with torch unless given; the workspace too
    (a CUDA uint8 tensor of at least ``fa_bwd_workspace_bytes`` bytes).
    Returns (dq, dk, dv)."""
    if layout not in _LAYOUT_CODE:
        raise ValueError(f"layout must be one of {sorted(_LAYOUT_CODE)}")
    for t in (q, k, v, o, d_o):
        if t.dim() != 4 or not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, d_o must be contiguous 4-D CUDA tensors of one dtype")
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("the backward pass takes float16 or bfloat16")
    if o.shape != q.shape or d_o.shape != q.shape or v.shape != k.shape:
        raise ValueError("o and d_o must have q's shape, v k's")
    if layout == "bhnd":
        B, H, N, D = q.shape
        Hkv = k.shape[1]
    else:
        B, N, H, D = q.shape
        Hkv = k.shape[2]
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be the forward's contiguous fp32 [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    mk, wl, wr = mask_args(causal, window)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    with torch.cuda.device(q.device):
        wb = fa_bwd_workspace_bytes(B, H, N)
        if workspace is None:
            workspace = torch.empty(wb, dtype=torch.uint8, device=q.device)
        s = (stream or torch.cuda.current_stream(q.device)).cuda_stream
        rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(), lse.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, N, D, float(scale), mk, wl, wr,
                    _DTYPE_CODE[q.dtype], _LAYOUT_CODE[layout], workspace.data_ptr(), workspace.numel(), s)
    _check(rc, "fa_bwd")
    return dq, dk, dv


def rope_tables(n_pos, D, base=10000.0, device="cuda", stream=None):
    """cos, sin fp32 [n_pos, D/2] CUDA tensors for positions 0 .. n_pos-1,
    filled by ``fa_rope_tables`` (angle p * base^(-2i/D))."""
    dev = torch.device(device)
    cos = torch.empty((n_pos, D // 2), dtype=torch.float32, device=dev)
    sin = torch.empty_like(cos)
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        rc = fa_rope_tables(cos.data_ptr(), sin.data_ptr(), n_pos, D, float(base), s)
    _check(rc, "fa_rope_tables")
    return cos, sin


def apply_rope(q=None, k=None, cos=None, sin=None, style="half", q_pos0=0, k_pos0=0, layout="bhnd",
               q_out=None, k_out=None, inplace=False, stream=None):
    """Rotary position embedding of q and/or k with ``fa_rope``.

    q is [B, H, Nq, D] (``layout="bhnd"``) or [B, Nq, H, D] (``"bnhd"``), k
    likewise with H_kv heads; row n of q sits at position q_pos0 + n, of k at
    k_pos0 + n.  ``cos``/``sin`` are fp32 [n_pos, D/2] CUDA tensors
    (``rope_tables``).  ``style``: "half" pairs (i, i + D/2), "interleaved"
    pairs (2i, 2i + 1).  Returns (q_rot, k_rot), None for a tensor not given;
    ``inplace=True`` rotates the given tensors themselves.
    """
    if style not in _ROPE_STYLE:
        raise ValueError(f"style must be one of {sorted(_ROPE_STYLE)}")
    if layout not in _LAYOUT_CODE:
        raise ValueError(f"layout must be one of {sorted(_LAYOUT_CODE)}")
    if q is None and k is None:
        raise ValueError("give q, k or both")
    ref = q if q is not None else k
    if cos is None or sin is None or cos.dtype != torch.float32 or sin.shape != cos.shape or cos.dim() != 2:
        raise ValueError("cos and sin must be fp32 [n_pos, D/2] tensors of one shape")
    for t in (q, k):
        if t is not None and (t.dim() != 4 or not t.is_cuda or not t.is_contiguous() or t.dtype != ref.dtype
                              or t.dtype not in _DTYPE_CODE):
            raise ValueError("q and k must be contiguous 4-D CUDA tensors of one dtype")
    if not (cos.is_cuda and sin.is_cuda and cos.is_contiguous() and sin.is_contiguous()):
        raise ValueError("cos and sin must be contiguous CUDA tensors")
    seq, head = (2, 1) if layout == "bhnd" else (1, 2)
    B, D = ref.shape[0], ref.shape[3]
    if q is not None and k is not None and (k.shape[0] != B or k.shape[3] != D):
        raise ValueError("q and k disagree on B or D")
    if cos.shape[1] != D // 2:
        raise ValueError(f"table has {cos.shape[1]} columns, D/2 = {D // 2}")
    H, Nq = (q.shape[head], q.shape[seq]) if q is not None else (1, 1)
    Hkv, Nk = (k.shape[head], k.shape[seq]) if k is not None else (1, 1)
    if q is not None and q_out is None:
        q_out = q if inplace else torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = k if inplace else torch.empty_like(k)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    with torch.cuda.device(ref.device):
        s = (stream or torch.cuda.current_stream(ref.device)).cuda_stream
        rc = fa_rope(ptr(q), ptr(k), ptr(q_out), ptr(k_out), cos.data_ptr(), sin.data_ptr(), B, H, Hkv, Nq, Nk, D,
                     int(q_pos0), int(k_pos0), cos.shape[0], _ROPE_STYLE[style], _DTYPE_CODE[ref.dtype],
                     _LAYOUT_CODE[layout], s)
    _check(rc, "fa_rope")
    return q_out, k_out


def attention_fwd_rope(q, k, v, cos, sin, style="half", pos0=0, layout="bhnd", fused=True, **kw):
    """attention_fwd on rotary-embedded q and k (rows at positions pos0,
    pos0 + 1, ...).  For fp16 / bf16 with ``fused=True`` only K goes through
    the ``fa_rope`` pass and Q is rotated inside the attention kernel
    (``fa_fwd_rope``); otherwise ``fa_rope`` writes rotated copies of both
    and the plain forward runs on them.  Returns (O, LSE)."""
    if fused and q.dtype in (torch.float16, torch.bfloat16):
        _, kr = apply_rope(None, k, cos, sin, style=style, k_pos0=pos0, layout=layout, stream=kw.get("stream"))
        return attention_fwd(q, kr, v, layout=layout, rope=(cos, sin), rope_style=style, rope_pos0=pos0, **kw)
    qr, kr = apply_rope(q, k, cos, sin, style=style, q_pos0=pos0, k_pos0=pos0, layout=layout,
                        stream=kw.get("stream"))
    return attention_fwd(qr, kr, v, layout=layout, **kw)


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_lens, max_seq_len=None, scale=None, causal=False,
                           window=None, n_splits=0, out=None, lse=None, workspace=None, stream=None, layout="bhnd"):
    """Decode against a paged cache: k_cache, v_cache [num_pages, page_size,
    H_kv, D]; block_table int32 [B, max_pages]; seq_lens int32 [B] (all CUDA).
    Query i of sequence b sits at position seq_lens[b] - Nq + i.  q is
    [B, H, Nq, D] (``layout="bhnd"``) or [B, Nq, H, D].  ``max_seq_len`` (the
    split plan's length, at least every seq_lens[b]) defaults to
    max_pages * page_size.  Returns (O, LSE), LSE [B, H, Nq]."""
    if layout not in _LAYOUT_CODE:
        raise ValueError(f"layout must be one of {sorted(_LAYOUT_CODE)}")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must be [num_pages, page_size, H_kv, D] alike")
    num_pages, page_size, Hkv, D = k_cache.shape
    if layout == "bhnd":
        B, H, Nq, Dq = q.shape
    else:
        B, Nq, H, Dq = q.shape
    if Dq != D or H % Hkv:
        raise ValueError("q does not match the cache's head size or K/V head count")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise ValueError("seq_lens must be int32 [B]")
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all inputs must be contiguous CUDA tensors")
    if not (q.dtype == k_cache.dtype == v_cache.dtype) or q.dtype not in _DTYPE_CODE:
        raise ValueError("q and the caches must share one dtype among float16, bfloat16, float32")
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * page_size
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    mk, wl, wr = mask_args(causal, window)
    with torch.cuda.device(q.device):
        ns, wb = fa_decode_plan_gqa(B, H, Hkv, Nq, max_seq_len, D, n_splits)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        if workspace is None and wb > 0:
            workspace = torch.empty(wb, dtype=torch.uint8, device=q.device)
        s = (stream or torch.cuda.current_stream(q.device)).cuda_stream
        rc = fa_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                             seq_lens.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq, max_seq_len,
                             page_size, max_pages, num_pages, D, float(scale), mk, wl, wr, _DTYPE_CODE[q.dtype],
                             _LAYOUT_CODE[layout], ns, workspace.data_ptr() if workspace is not None else None,
                             workspace.numel() if workspace is not None else 0, s)
    _check(rc, "fa_decode_paged")
    return out, lse


def attention_fwd_host(q, k, v, device="cuda", **kw):
    """The same call for host tensors: copies Q, K, V to the device, runs the
    fused forward, and copies O and LSE back (pinned host buffers make both
    copies asynchronous)."""
    dq, dk, dv = (t.to(device, non_blocking=True) for t in (q, k, v))
    o, lse = attention_fwd(dq, dk, dv, **kw)
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    ho.copy_(o, non_blocking=True)
    hl.copy_(lse, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return ho, hl
