// The softmax step of the one-CTA forward kernel (fa_tc.cu) and the in-place
// rotation of a Q tile shared by both fused forward kernels (fa_tc.cu and the
// CTA-pair fa_tc2.cu).
//
// One thread owns one query row of a 128-row tile whose scores S (fp32) sit
// in tensor memory, 64 keys at a time.  The step follows the online softmax of
// "Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention" (section 1.2) and the ops-transformer
// walk-through ("online softmax: incremental update"): mask, running row
// max, exponentials relative to it, probabilities P written back over S as
// 16-bit values for the P.V product, and the row sum.  The running max is
// moved lazily: only when a tile's max exceeds it by more than kTau (log2
// units), in which case O and the row sum are rescaled (softmax is unchanged
// by a common shift of a row, so any reference max at or above the true one
// minus kTau gives the same result up to rounding and keeps every p <= 2^kTau).
#pragma once
#include <cmath>

#include "fa_geom.h"
#include "ptx.cuh"
#include "rope_math.cuh"
#include "tc_common.cuh"

namespace fa {

constexpr float kTau = 8.0f;                      // lazy rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;

// Bit i (0 <= i < 32) set iff lo <= i <= hi: the visible columns of one
// 32-column chunk, from the row's visible interval taken relative to the
// chunk's first column.
__device__ __forceinline__ uint32_t span_bits(int lo, int hi) {
    const uint32_t upto = hi >= 31 ? 0xffffffffu : hi < 0 ? 0u : (2u << hi) - 1u;
    const uint32_t from = lo <= 0 ? 0xffffffffu : lo > 31 ? 0u : 0xffffffffu << lo;
    return upto & from;
}

// One half (64 keys) of key tile j for one row (query qi, tile start r0):
// an online-softmax step of its own.  tS / tO: this warp's lane base plus the
// half's 64 S columns / the tile's O columns.  c2 = scale * log2(e).  On
// return P is in tensor memory over the half's first 32 columns (16-bit
// pairs; with `split` the bf16 low parts in the next 32), every tensor-memory
// store has completed and been fenced for a following thread
// synchronisation, m_ref / l are updated (l rescaled, not yet increased) and
// `lsum` holds this half's row sum.  When the running max moves by more than
// kTau, O is rescaled in place after `wait_pv()` has confirmed that the
// product still adding into O (the previous half's P.V) has completed; false
// if that wait gave up.  kMask = false builds the step without the element
// mask, for problems where no tile needs one (geom_needs_masks).
template <int D, bool kBf16, bool kPosScale, bool kMask, class WaitPv>
__device__ __forceinline__ bool softmax_half(const Geom& g, uint32_t tS, uint32_t tO, float c2, int r0, int qi, int j,
                                             int h, bool first, bool split, float& m_ref, float& l, float& lsum,
                                             const WaitPv& wait_pv) {
    using namespace ptx;
    uint32_t s[2][32];
    tmem_ld32(tS, s[0]);
    tmem_ld32(tS + 32, s[1]);
    tmem_wait_ld();

    if (!kPosScale) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float a, b;
                fmul2(a, b, u2f(s[c][i]), u2f(s[c][i + 1]), c2, c2);
                s[c][i] = f2u(a);
                s[c][i + 1] = f2u(b);
            }
    }
    if (kMask && tile_needs_mask(g, r0, j)) {  // the same for the whole tile
        // The row's visible interval as a bit set per 32-column chunk; a chunk
        // the whole warp sees in full is skipped.
        int c_lo, c_hi;
        row_visible_cols(g, qi, j, c_lo, c_hi);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int c0 = 32 * (2 * h + c);
            const uint32_t vis = span_bits(c_lo - c0, c_hi - c0);
            if (__all_sync(0xffffffffu, vis == 0xffffffffu)) continue;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (!((vis >> i) & 1u)) s[c][i] = f2u(-INFINITY);
        }
    }
    // Row max: 32 three-input maxes spread over 8 independent chains.
    float mxk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mxk[k] = fmaxf(u2f(s[0][2 * k]), u2f(s[0][2 * k + 1]));
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = (c == 0 ? 16 : 0); i < 32; i += 2) {
            const int k = (i >> 1) & 7;
            mxk[k] = max3(mxk[k], u2f(s[c][i]), u2f(s[c][i + 1]));
        }
    const float mx = fmaxf(max3(mxk[0], mxk[1], mxk[2]), max3(max3(mxk[3], mxk[4], mxk[5]), mxk[6], mxk[7]));
    const float m_new = kPosScale ? mx * c2 : mx;

    float alpha = 1.f;
    bool resc = false;
    if (first) {
        m_ref = m_new;
    } else if (m_new > m_ref + kTau) {
        alpha = ex2(m_ref - m_new);
        m_ref = m_new;
        resc = true;
    }
    l *= alpha;
    const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
    float l0 = 0.f, l1 = 0.f;
    if (!split) {
        // p = 2^(s*c - m) two at a time (packed FFMA, two ex2), packed into
        // 16-bit pairs; the row sum runs over four packed accumulators.
        float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float a, b;
                if (kPosScale)
                    ffma2(a, b, u2f(s[c][i]), u2f(s[c][i + 1]), c2, c2, neg_m, neg_m);
                else
                    fadd2(a, b, u2f(s[c][i]), u2f(s[c][i + 1]), neg_m, neg_m);
                a = ex2(a);
                b = ex2(b);
                pk[i >> 1] = pack2<kBf16>(a, b);
                const int k = (i >> 1) & 3;
                fadd2(acc[k][0], acc[k][1], acc[k][0], acc[k][1], a, b);
            }
            tmem_st16(tS + 16 * c, pk);
        }
        l0 = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
        l1 = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
    } else {
        // p = hi + lo, both bf16: hi in columns [0, 32), lo in [32, 64).
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float a = kPosScale ? ex2(fmaf(u2f(s[c][i]), c2, neg_m)) : ex2(u2f(s[c][i]) + neg_m);
                const float b =
                    kPosScale ? ex2(fmaf(u2f(s[c][i + 1]), c2, neg_m)) : ex2(u2f(s[c][i + 1]) + neg_m);
                const uint32_t w = pack2<kBf16>(a, b);
                hw[i >> 1] = w;
                lw[i >> 1] = pack2<kBf16>(a - lo_half<kBf16>(w), b - hi_half<kBf16>(w));
                l0 += a;
                l1 += b;
            }
            tmem_st16(tS + 16 * c, hw);
            tmem_st16(tS + 32 + 16 * c, lw);
        }
    }
    bool ok = true;
    if (!first && __any_sync(0xffffffffu, resc)) {
        // Rare: the running max moved by more than kTau; rescale this row of O
        // once the P.V still in flight has landed (the next one waits for this
        // warpgroup's arrival).
        ok = wait_pv();
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                tmem_st32(tO + c * 32, o);
            }
        }
    }
    tmem_wait_st();
    tc_fence_before();
    lsum = l0 + l1;
    return ok;
}

// ------------------------------------------- rotary embedding of a Q tile
// One query row of a Q tile in shared memory, rotated in place by the table
// entries of its position (the rotation of "Ascend C advanced practice:
// high-performance FlashAttention-2-style tile-level fused attention",
// section 9, applied to Q as it is loaded; K arrives already rotated).  The
// tile holds D/64 column chunks of 128 rows x 128 bytes, 128-byte swizzled:
// 16-byte unit U of row r sits at chunk U/8, slot (U%8) ^ (r%8).  Groups of
// eight pairs: half-split pairs units g and D/16 + g element by element,
// interleaved pairs neighbours inside units 2g and 2g + 1.
template <int D, bool kBf16, int kBox>
__device__ __forceinline__ void rope_q_row(uint8_t* tile, int row, const float* cos_row, const float* sin_row,
                                           int style) {
    uint8_t* rb = tile + row * 128;
    const int sw = row & 7;
#pragma unroll
    for (int g = 0; g < D / 16; ++g) {
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(cos_row + 8 * g));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(cos_row + 8 * g + 4));
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(sin_row + 8 * g));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(sin_row + 8 * g + 4));
        const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const int ua = style == ROPE_HALF ? g : 2 * g;
        const int ub = style == ROPE_HALF ? D / 16 + g : 2 * g + 1;
        uint4* pa = reinterpret_cast<uint4*>(rb + (ua >> 3) * kBox + (((ua & 7) ^ sw) << 4));
        uint4* pb = reinterpret_cast<uint4*>(rb + (ub >> 3) * kBox + (((ub & 7) ^ sw) << 4));
        const uint4 wa = *pa, wb = *pb;
        const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t xb[4] = {wb.x, wb.y, wb.z, wb.w};
        float u[8], v[8], yu[8], yv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            u[2 * i] = lo_half<kBf16>(xa[i]);
            u[2 * i + 1] = hi_half<kBf16>(xa[i]);
            v[2 * i] = lo_half<kBf16>(xb[i]);
            v[2 * i + 1] = hi_half<kBf16>(xb[i]);
        }
        if (style == ROPE_HALF) {
#pragma unroll
            for (int m = 0; m < 8; ++m) rope_rotate(u[m], v[m], c[m], sn[m], yu[m], yv[m]);
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                rope_rotate(u[2 * m], u[2 * m + 1], c[m], sn[m], yu[2 * m], yu[2 * m + 1]);
                rope_rotate(v[2 * m], v[2 * m + 1], c[4 + m], sn[4 + m], yv[2 * m], yv[2 * m + 1]);
            }
        }
        *pa = make_uint4(pack2<kBf16>(yu[0], yu[1]), pack2<kBf16>(yu[2], yu[3]), pack2<kBf16>(yu[4], yu[5]),
                         pack2<kBf16>(yu[6], yu[7]));
        *pb = make_uint4(pack2<kBf16>(yv[0], yv[1]), pack2<kBf16>(yv[2], yv[3]), pack2<kBf16>(yv[4], yv[5]),
                         pack2<kBf16>(yv[6], yv[7]));
    }
}

}  // namespace fa
