"""GB300-native (sm_103a) fused attention.

``attention_fwd(q, k, v, scale=None, causal=False, window=None)`` returns
(O, LSE) for contiguous [B, H, N, D] (or [B, N, H, D]) CUDA tensors, computed
by libfa's hand-written tcgen05/TMA kernels (fp16 / bf16) or its fp32 FFMA
kernel.  Around it: ``attention_decode`` / ``attention_decode_paged`` (split-K
decode against a contiguous or paged K/V cache), ``attention_bwd`` (dQ, dK,
dV), ``apply_rope`` / ``rope_tables`` / ``attention_fwd_rope`` (rotary
embedding of Q and K).  The C ABI is declared in ``include/fa.h``;
``binding`` mirrors it, and a missing library raises.
"""

from .binding import (  # noqa: F401
    FA_BF16, FA_F16, FA_F32, FA_MASK_CAUSAL, FA_MASK_NONE, FA_MASK_WINDOW, FaError, attention_decode, attention_fwd,
    apply_rope, attention_bwd, attention_decode_paged, fa_decode_paged, fa_bwd, fa_bwd_workspace_bytes, attention_fwd_host, attention_fwd_rope, fa_rope, fa_rope_tables, fa_fwd_rope, rope_tables, fa_fwd_gqa, fa_decode, fa_decode_gqa, fa_decode_plan, fa_decode_plan_gqa, fa_device_status, fa_fwd, fa_fwd_bf16, fa_fwd_ex, fa_fwd_f16, fa_fwd_f32,
    fa_plan_units, fa_selftest_wait_timeout, fa_set_wait_limit_ns, fa_tile_needs_mask, fa_geom_needs_masks, load,
    mask_args)
