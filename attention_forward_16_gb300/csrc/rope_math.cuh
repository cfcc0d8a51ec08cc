// The rotation of one (x_a, x_b) pair by one cos/sin table entry, shared by
// the streaming rotation pass (fa_rope.cu) and the forward kernel's in-place
// rotation of its Q tiles (fa_tc.cu), so the two give the same bits:
//     x_a' = x_a cos - x_b sin,   x_b' = x_b cos + x_a sin
// ("Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention", section 9: rotate Q/K from a cos/sin table),
// each cross product rounded once and the other product fused into the sum.
#pragma once

namespace fa {

__device__ __forceinline__ void rope_rotate(float xa, float xb, float c, float s, float& ya, float& yb) {
    ya = __fmaf_rn(xa, c, -__fmul_rn(xb, s));
    yb = __fmaf_rn(xb, c, __fmul_rn(xa, s));
}

}  // namespace fa
