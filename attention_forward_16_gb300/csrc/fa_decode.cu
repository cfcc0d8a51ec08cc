// Split-K attention decode: a few new queries against a long K/V cache.
//
// "FlashAttention extreme optimisation on Ascend NPUs", optimisation four
// (KV-cache incremental decode) computes one new token's attention over the
// cached keys, but merges block results with a running average that is not
// softmax-correct.  Here each CTA takes one split of the cache and produces a
// normalised partial O_s with its log-sum-exp LSE_s; a combine pass then
// forms the exact result
//
//     LSE = ln sum_s e^{LSE_s},    O = sum_s e^{LSE_s - LSE} O_s
//
// (the same identity as the online softmax of "Ascend C advanced practice:
// high-performance FlashAttention-2-style tile-level fused attention",
// section 1.2, applied to whole blocks of keys).
//
// Decode reads every cached key and value once and does about one FLOP per
// byte, so it is bound by HBM bandwidth, not by the tensor cores: the kernel
// streams K and V with coalesced 8- or 16-byte loads (each lane owns D/32
// consecutive elements of a row; a warp reads whole rows), keeps four keys in
// flight per warp, and runs the online softmax in fp32 registers.  Query i
// sits at key position Nk - Nq + i (the new tokens are the last Nq entries of
// the cache), which sets the causal and window masks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kKeysPerIter = 4;
constexpr float kDecLn2 = 0.69314718055994530942f;

template <typename T, int DV>
struct Vec;
template <>
struct Vec<__half, 2> {
    using raw = uint32_t;
    static __device__ __forceinline__ void cvt(raw r, float* f) {
        const float2 a = __half22float2(*reinterpret_cast<__half2*>(&r));
        f[0] = a.x; f[1] = a.y;
    }
};
template <>
struct Vec<__half, 4> {
    using raw = uint2;
    static __device__ __forceinline__ void cvt(raw r, float* f) {
        const float2 a = __half22float2(*reinterpret_cast<__half2*>(&r.x));
        const float2 b = __half22float2(*reinterpret_cast<__half2*>(&r.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
};
template <>
struct Vec<__nv_bfloat16, 2> {
    using raw = uint32_t;
    static __device__ __forceinline__ void cvt(raw r, float* f) {
        f[0] = __uint_as_float(r << 16); f[1] = __uint_as_float(r & 0xFFFF0000u);
    }
};
template <>
struct Vec<__nv_bfloat16, 4> {
    using raw = uint2;
    static __device__ __forceinline__ void cvt(raw r, float* f) {
        f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xFFFF0000u);
        f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xFFFF0000u);
    }
};
template <>
struct Vec<float, 2> {
    using raw = float2;
    static __device__ __forceinline__ void cvt(raw r, float* f) { f[0] = r.x; f[1] = r.y; }
};
template <>
struct Vec<float, 4> {
    using raw = float4;
    static __device__ __forceinline__ void cvt(raw r, float* f) { f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w; }
};

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }

// Element offsets of query row r (= g * Nq + i: query head g of the group,
// query i) and of key/value row j, for the (batch, K/V head) group bhk.
__device__ __forceinline__ size_t dec_qrow(const DecodeParams& p, long long bhk, int r, int D) {
    const int g = r / p.Nq, i = r % p.Nq;
    if (p.layout == LAYOUT_BHND) return ((size_t)(bhk * p.G + g) * p.Nq + i) * D;
    const long long b = bhk / p.Hkv, h = (bhk % p.Hkv) * p.G + g;
    return (((size_t)b * p.Nq + i) * ((size_t)p.Hkv * p.G) + h) * D;
}
__device__ __forceinline__ size_t dec_krow(const DecodeParams& p, long long bhk, int j, int D) {
    if (p.block_table) {
        // paged: [num_pages, page_size, Hkv, D]; a bad page index is clamped, never followed
        const long long b = bhk / p.Hkv, hk = bhk % p.Hkv;
        int page = p.block_table[(size_t)b * p.max_pages + (j >> p.page_shift)];
        page = page < 0 ? 0 : (page >= p.num_pages ? p.num_pages - 1 : page);
        const int r = j & ((1 << p.page_shift) - 1);
        return ((((size_t)page << p.page_shift) + r) * p.Hkv + hk) * D;
    }
    if (p.layout == LAYOUT_BHND) return ((size_t)bhk * p.Nk + j) * D;
    const long long b = bhk / p.Hkv, hk = bhk % p.Hkv;
    return (((size_t)b * p.Nk + j) * p.Hkv + hk) * D;
}

// Cached positions of the sequence of (batch, K/V head) group bhk.
__device__ __forceinline__ int dec_len(const DecodeParams& p, long long bhk) {
    if (!p.seq_lens) return p.Nk;
    const int n = p.seq_lens[bhk / p.Hkv];
    return n < 0 ? 0 : (n > p.Nk ? p.Nk : n);
}

// Query i of a sequence of `len` cached positions sits at len - Nq + i.
__device__ __forceinline__ bool dec_visible(const DecodeParams& p, int i, int j, int len) {
    const long long pos = (long long)len - p.Nq + i;
    if (p.win_l >= 0 && j < pos - p.win_l) return false;
    if (p.win_r >= 0 && j > pos + p.win_r) return false;
    return true;
}

// One CTA = one (b, h, split).  Warps take keys round-robin in groups of four.
template <typename T, int DV, int NQ>
__global__ void __launch_bounds__(kDecThreads) fa_decode_split_kernel(const DecodeParams p) {
    using V = Vec<T, DV>;
    constexpr int D = 32 * DV;
    extern __shared__ float dsm[];  // [warps][NQ][D + 2]: m, l, acc
    ptx::griddep_launch_dependents();    // the combine pass may start launching
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.n_splits;
    const long long bh = blockIdx.x / p.n_splits;
    const int len = dec_len(p, bh);
    const int k0 = split * p.chunk;
    const int k1 = min(len, k0 + p.chunk);
    const int rows = p.G * p.Nq;
    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k);
    const T* vg = static_cast<const T*>(p.v);

    float q[NQ][DV], acc[NQ][DV], m[NQ], l[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < DV; ++e) acc[i][e] = 0.f;
        if (i < rows) {
            V::cvt(*reinterpret_cast<const typename V::raw*>(qg + dec_qrow(p, bh, i, D) + lane * DV), q[i]);
#pragma unroll
            for (int e = 0; e < DV; ++e) q[i][e] *= p.scale_log2;  // scores in log2 units
        } else {
#pragma unroll
            for (int e = 0; e < DV; ++e) q[i][e] = 0.f;
        }
    }

    // Double-buffered in registers: the next group's loads are issued before
    // this group's arithmetic, so each warp keeps eight rows of K and V in flight.
    constexpr int kStride = kDecWarps * kKeysPerIter;
    typename V::raw kn[kKeysPerIter], vn[kKeysPerIter];
    auto load_group = [&](int base) {
#pragma unroll
        for (int u = 0; u < kKeysPerIter; ++u) {
            const int j = base + u < k1 ? base + u : k1 - 1;  // clamp: tail keys are masked below
            const size_t kr_off = dec_krow(p, bh, j, D) + lane * DV;
            kn[u] = *reinterpret_cast<const typename V::raw*>(kg + kr_off);
            vn[u] = *reinterpret_cast<const typename V::raw*>(vg + kr_off);
        }
    };
    if (k0 + warp * kKeysPerIter < k1) load_group(k0 + warp * kKeysPerIter);
    for (int base = k0 + warp * kKeysPerIter; base < k1; base += kStride) {
        typename V::raw kr[kKeysPerIter], vr[kKeysPerIter];
#pragma unroll
        for (int u = 0; u < kKeysPerIter; ++u) {
            kr[u] = kn[u];
            vr[u] = vn[u];
        }
        if (base + kStride < k1) load_group(base + kStride);
        float kf[kKeysPerIter][DV], vf[kKeysPerIter][DV];
#pragma unroll
        for (int u = 0; u < kKeysPerIter; ++u) {
            V::cvt(kr[u], kf[u]);
            V::cvt(vr[u], vf[u]);
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= rows) break;
            float s[kKeysPerIter];
#pragma unroll
            for (int u = 0; u < kKeysPerIter; ++u) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < DV; ++e) d = fmaf(q[i][e], kf[u][e], d);
                s[u] = d;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int u = 0; u < kKeysPerIter; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < kKeysPerIter; ++u) {
                if (base + u >= k1 || !dec_visible(p, i % p.Nq, base + u, len)) s[u] = -INFINITY;
                mx = fmaxf(mx, s[u]);
            }
            if (mx == -INFINITY) continue;  // warp-uniform: no visible key in this group
            if (mx > m[i]) {
                const float a = m[i] == -INFINITY ? 0.f : ptx::ex2(m[i] - mx);
                l[i] *= a;
#pragma unroll
                for (int e = 0; e < DV; ++e) acc[i][e] *= a;
                m[i] = mx;
            }
#pragma unroll
            for (int u = 0; u < kKeysPerIter; ++u) {
                const float pu = ptx::ex2(s[u] - m[i]);
                l[i] += pu;
#pragma unroll
                for (int e = 0; e < DV; ++e) acc[i][e] = fmaf(pu, vf[u][e], acc[i][e]);
            }
        }
    }

    // Merge the four warps' states through shared memory.
    float* mine = dsm + (size_t)warp * NQ * (D + 2);
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (i >= rows) break;
        if (lane == 0) {
            mine[i * (D + 2) + D] = m[i];
            mine[i * (D + 2) + D + 1] = l[i];
        }
#pragma unroll
        for (int e = 0; e < DV; ++e) mine[i * (D + 2) + lane * DV + e] = acc[i][e];
    }
    __syncthreads();
    for (int i = warp; i < rows; i += kDecWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, dsm[((size_t)w * NQ + i) * (D + 2) + D]);
        float L = 0.f, o[DV];
#pragma unroll
        for (int e = 0; e < DV; ++e) o[e] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kDecWarps; ++w) {
                const float* st = dsm + ((size_t)w * NQ + i) * (D + 2);
                const float a = st[D] == -INFINITY ? 0.f : ptx::ex2(st[D] - M);
                L += a * st[D + 1];
#pragma unroll
                for (int e = 0; e < DV; ++e) o[e] = fmaf(a, st[lane * DV + e], o[e]);
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse = L > 0.f ? (M + log2f(L)) * kDecLn2 : -INFINITY;
        if (p.n_splits == 1) {
            T* ob = static_cast<T*>(p.o) + dec_qrow(p, bh, i, D) + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) ob[e] = from_float<T>(o[e] * inv);
            if (p.lse && lane == 0) p.lse[(size_t)bh * rows + i] = lse;   // [B, H, Nq] row of query head g, query i
        } else {
            const size_t prow = ((size_t)bh * p.n_splits + split) * rows + i;
            float* po = p.part_o + prow * D + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) po[e] = o[e] * inv;
            if (lane == 0) p.part_lse[prow] = lse;
        }
    }
}

// Eight consecutive elements of a row as fp32.
template <typename T>
struct Row8 {
    using raw = uint4;  // 8 x 16-bit
    static __device__ __forceinline__ raw load(const T* p) { return *reinterpret_cast<const uint4*>(p); }
    static __device__ __forceinline__ void cvt(const raw& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
                f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
            }
        }
    }
};
template <>
struct Row8<float> {
    struct raw {
        float4 a, b;
    };
    static __device__ __forceinline__ raw load(const float* p) {
        return raw{reinterpret_cast<const float4*>(p)[0], reinterpret_cast<const float4*>(p)[1]};
    }
    static __device__ __forceinline__ void cvt(const raw& r, float* f) {
        f[0] = r.a.x, f[1] = r.a.y, f[2] = r.a.z, f[3] = r.a.w, f[4] = r.b.x, f[5] = r.b.y, f[6] = r.b.z, f[7] = r.b.w;
    }
};

// Sum of four rows' partial dot products over the L lanes of a lane group,
// transposed: the first two steps exchange half of the remaining rows
// instead of all of them, so 4 rows cost L/8 + 4 shuffles rather than
// 4 log2(L).  Afterwards lane t holds the full sum of row
// 2 * ((t / (L/2)) & 1) + ((t / (L/4)) & 1); lane r * (L/4) holds row r.
template <int L>
__device__ __forceinline__ float reduce_rows4(const float (&d)[4], int t) {
    constexpr int B1 = L / 2, B2 = L / 4;
    const bool h1 = t & B1;
    float k0 = h1 ? d[2] : d[0], k1 = h1 ? d[3] : d[1];
    k0 += __shfl_xor_sync(0xffffffffu, h1 ? d[0] : d[2], B1);
    k1 += __shfl_xor_sync(0xffffffffu, h1 ? d[1] : d[3], B1);
    const bool h2 = t & B2;
    float v = h2 ? k1 : k0;
    v += __shfl_xor_sync(0xffffffffu, h2 ? k0 : k1, B2);
#pragma unroll
    for (int off = B2 / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Two to four query rows per (batch, K/V head) -- grouped heads, or a few
// new tokens.  A key row is split over L = D/8 lanes (16 bytes each for
// 16-bit types), so a warp takes 32/L keys side by side; each lane group
// keeps its own online-softmax state for the keys it sees, and all groups of
// the CTA merge at the end.  Against one key per warp with a five-step
// butterfly per row, this cuts the shuffles per key and row from 5 to about 1.
template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) fa_decode_rows_kernel(const DecodeParams p) {
    using R8 = Row8<T>;
    constexpr int L = D / 8;                        // lanes per key
    constexpr int KPW = 32 / L;                     // keys side by side in a warp
    constexpr int U = sizeof(T) == 4 ? 2 : 4;       // keys per lane group per iteration
    constexpr int kBlock = KPW * U;                 // keys per warp per iteration
    constexpr int kStates = kDecWarps * KPW;
    constexpr int DV = D / 32;
    extern __shared__ float dsm[];                  // [kStates][4][D + 2]: m, l, acc
    ptx::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane / L;
    const int t = lane % L;
    const int split = blockIdx.x % p.n_splits;
    const long long bh = blockIdx.x / p.n_splits;
    const int len = dec_len(p, bh);
    const int k0 = split * p.chunk;
    const int k1 = min(len, k0 + p.chunk);
    const int rows = p.G * p.Nq;
    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k);
    const T* vg = static_cast<const T*>(p.v);

    float q[4][8], acc[4][8], m[4], l[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;
        if (r < rows) {
            R8::cvt(R8::load(qg + dec_qrow(p, bh, r, D) + t * 8), q[r]);
#pragma unroll
            for (int e = 0; e < 8; ++e) q[r][e] *= p.scale_log2;  // scores in log2 units
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q[r][e] = 0.f;
        }
    }

    // Keys every query sees: [vis_lo, vis_hi], the intersection of the
    // queries' bands (query i sits at len - Nq + i).  A block inside it skips
    // the per-key test, so only blocks at a band's edge pay for the mask.
    const long long vis_lo = p.win_l >= 0 ? (long long)len - 1 - p.win_l : LLONG_MIN;
    const long long vis_hi = p.win_r >= 0 ? (long long)len - p.Nq + p.win_r : LLONG_MAX;

    // key u of a block for this lane group: base + u * KPW + grp, so one load
    // instruction of the warp reads KPW consecutive rows
    typename R8::raw kn[U], vn[U];
    auto load_block = [&](int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int j = base + u * KPW + grp;
            if (j >= k1) j = k1 - 1;  // clamp: tail keys are masked below
            const size_t off = dec_krow(p, bh, j, D) + t * 8;
            kn[u] = R8::load(kg + off);
            vn[u] = R8::load(vg + off);
        }
    };
    constexpr int kStride = kDecWarps * kBlock;
    if (k0 + warp * kBlock < k1) load_block(k0 + warp * kBlock);
    for (int base = k0 + warp * kBlock; base < k1; base += kStride) {
        typename R8::raw vr[U];
        float sc[U][4];
        // scores of the group's U keys for all four rows: U independent dot
        // products and shuffle chains
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float kf[8];
            R8::cvt(kn[u], kf);
            vr[u] = vn[u];
            float d[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(q[r][e], kf[e], a);
                d[r] = a;
            }
            const float own = reduce_rows4<L>(d, t);
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[u][r] = __shfl_sync(0xffffffffu, own, grp * L + r * (L / 4));
        }
        if (base + kStride < k1) load_block(base + kStride);
        const bool full_block = base >= vis_lo && (long long)base + kBlock - 1 <= vis_hi && base + kBlock <= k1;
        if (!full_block) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = base + u * KPW + grp;
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (j >= k1 || !dec_visible(p, r % p.Nq, j, len)) sc[u][r] = -INFINITY;
            }
        }
        float vf[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) R8::cvt(vr[u], vf[u]);
        // online softmax, one max and one rescale check per row per U keys
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r >= rows) break;
            float mx = sc[0][r];
#pragma unroll
            for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u][r]);
            if (mx == -INFINITY) continue;
            if (mx > m[r]) {
                const float a = m[r] == -INFINITY ? 0.f : ptx::ex2(m[r] - mx);
                l[r] *= a;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][e] *= a;
                m[r] = mx;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float pr = ptx::ex2(sc[u][r] - m[r]);
                l[r] += pr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr, vf[u][e], acc[r][e]);
            }
        }
    }

    // Merge the kStates lane-group states through shared memory.
    float* mine = dsm + (size_t)(warp * KPW + grp) * 4 * (D + 2);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (r >= rows) break;
        if (t == 0) {
            mine[r * (D + 2) + D] = m[r];
            mine[r * (D + 2) + D + 1] = l[r];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) mine[r * (D + 2) + t * 8 + e] = acc[r][e];
    }
    __syncthreads();
    for (int i = warp; i < rows; i += kDecWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kStates; ++w) M = fmaxf(M, dsm[((size_t)w * 4 + i) * (D + 2) + D]);
        float Lsum = 0.f, o[DV];
#pragma unroll
        for (int e = 0; e < DV; ++e) o[e] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kStates; ++w) {
                const float* st = dsm + ((size_t)w * 4 + i) * (D + 2);
                const float a = st[D] == -INFINITY ? 0.f : ptx::ex2(st[D] - M);
                Lsum += a * st[D + 1];
#pragma unroll
                for (int e = 0; e < DV; ++e) o[e] = fmaf(a, st[lane * DV + e], o[e]);
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * kDecLn2 : -INFINITY;
        if (p.n_splits == 1) {
            T* ob = static_cast<T*>(p.o) + dec_qrow(p, bh, i, D) + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) ob[e] = from_float<T>(o[e] * inv);
            if (p.lse && lane == 0) p.lse[(size_t)bh * rows + i] = lse;
        } else {
            const size_t prow = ((size_t)bh * p.n_splits + split) * rows + i;
            float* po = p.part_o + prow * D + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) po[e] = o[e] * inv;
            if (lane == 0) p.part_lse[prow] = lse;
        }
    }
}

// ------------------------------------------------- tensor-core decode rows
// Two to sixteen query rows per (batch, K/V head), 16-bit inputs: the scores
// and P.V of a block of 16 keys are warp-level m16n8k16 MMAs (rows padded to
// 16), so the per-key work no longer costs an FMA and a shuffle per element
// on the CUDA cores, and the kernel is left with the streaming of K and V.
// The scores' accumulator fragments are, element for element, the A operand
// fragments of the P.V product, so P never leaves registers; it enters that
// product as hi + lo, two 16-bit parts, which keeps the result as close to
// the fp32 arithmetic of the other decode kernels as their own rounding (the
// tensor cores have room to spare: the kernel is bound by HBM).
//
// Each warp streams its own 16-key blocks (round robin over the split)
// through a two-stage shared-memory ring filled by 16-byte asynchronous
// copies: the next block lands while this one is computed.  At 64 KB a CTA,
// three CTAs (twelve warps) share an SM, which hides the MMA and shuffle
// latencies that a deeper ring with four or eight warps an SM left exposed.
// Rows are 16-byte-chunk swizzled (chunk c of row r at c ^ (r % 8)), so the
// ldmatrix reads are free of bank conflicts.
namespace mmadec {

constexpr int kKeys = 16;   // keys per block
constexpr int kStages = 2;  // ring depth per warp (three CTAs per SM fit)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// c[16 x 8] += a[16 x 16] b[16 x 8], fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <typename T>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return ptx::pack_bf16x2(lo, hi);
    else return ptx::pack_f16x2(lo, hi);
}
// The two 16-bit values of a packed word, as fp32.
template <typename T>
__device__ __forceinline__ float2 unpack16(uint32_t w) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
// p as an unevaluated sum hi + lo of two 16-bit values (lo = the rounding
// error of hi), so that P.V keeps about twice the 16-bit precision of p.
template <typename T>
__device__ __forceinline__ void split16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
    hi = pack16<T>(p0, p1);
    const float2 h = unpack16<T>(hi);
    lo = pack16<T>(p0 - h.x, p1 - h.y);
}

template <int D>
struct Cfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kChunks = kRowBytes / 16;         // 16-byte chunks per row
    static constexpr int kBlockBytes = kKeys * kRowBytes;  // one block of K (or V)
    static constexpr int kStageBytes = 2 * kBlockBytes;    // K | V
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kRingBytes = kDecWarps * kWarpBytes;
    static constexpr int kMergeBytes = kDecWarps * kDecodeMaxQ * (D + 2) * 4;
    static constexpr int kSmem = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static __device__ __forceinline__ uint32_t swz(int row, int chunk) {
        return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
    }
};

}  // namespace mmadec

// One CTA = one (b, K/V head, split); 16-bit K/V, 2 <= G * Nq <= 16.
template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) fa_decode_mma_kernel(const DecodeParams p) {
    using namespace mmadec;
    using C = Cfg<D>;
    constexpr float kTauDec = 8.0f;  // lazy rescale threshold (log2 units), as in the forward
    extern __shared__ __align__(128) uint8_t dec_smem[];
    ptx::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;  // fragment row (and row + 8)
    const int q4 = lane & 3;  // fragment column pair
    const int split = blockIdx.x % p.n_splits;
    const long long bh = blockIdx.x / p.n_splits;
    const int len = dec_len(p, bh);
    const int k0 = split * p.chunk;
    const int k1 = min(len, k0 + p.chunk);
    const int rows = p.G * p.Nq;
    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k);
    const T* vg = static_cast<const T*>(p.v);
    const uint32_t ring = ptx::smem_u32(dec_smem) + warp * C::kWarpBytes;

    // Q as the A operand of every score product: rows g and g + 8 (zero past
    // `rows`), columns 16 ks + 2 q4 (+1) and 16 ks + 8 + 2 q4 (+1).
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = g + 8 * hr;
        const uint32_t* qrow = r < rows ? reinterpret_cast<const uint32_t*>(qg + dec_qrow(p, bh, r, D)) : nullptr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][hr] = qrow ? qrow[(16 * ks + 2 * q4) / 2] : 0u;
            qa[ks][2 + hr] = qrow ? qrow[(16 * ks + 8 + 2 * q4) / 2] : 0u;
        }
    }

    // Blocks of this split for this warp: b = warp, warp + 4, ...
    const int nb = k1 > k0 ? (k1 - k0 + kKeys - 1) / kKeys : 0;
    auto load_block = [&](int b, int st) {
        const uint32_t sK = ring + st * C::kStageBytes, sV = sK + C::kBlockBytes;
        const int base = k0 + b * kKeys;
        // lane covers chunk (lane % kChunks) of rows lane / kChunks + (32 / kChunks) i
        constexpr int kRowsPerPass = 32 / C::kChunks;
        const int ch = lane % C::kChunks;
        // A whole block inside one page (or an unpaged cache) is 16 rows at a
        // fixed stride: one address computation (one page lookup) per block.
        const bool even = base + kKeys <= k1 &&
                          (!p.block_table || (base >> p.page_shift) == ((base + kKeys - 1) >> p.page_shift));
        const size_t row0 = even ? dec_krow(p, bh, base, D) : 0;
        const size_t stride = (p.block_table || p.layout != LAYOUT_BHND) ? (size_t)p.Hkv * D : (size_t)D;
#pragma unroll
        for (int i = 0; i < kKeys / kRowsPerPass; ++i) {
            const int row = lane / C::kChunks + kRowsPerPass * i;
            int j = base + row;
            if (j >= k1) j = k1 - 1;  // clamp: tail keys are masked below
            const size_t off = (even ? row0 + (size_t)row * stride : dec_krow(p, bh, j, D)) + ch * 8;
            cp_async16(sK + C::swz(row, ch), kg + off);
            cp_async16(sV + C::swz(row, ch), vg + off);
        }
    };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (warp + kDecWarps * s < nb) load_block(warp + kDecWarps * s, s);
        cp_async_commit();
    }

    // Keys every query sees (see the lane-group kernel above).
    const long long vis_lo = p.win_l >= 0 ? (long long)len - 1 - p.win_l : LLONG_MIN;
    const long long vis_hi = p.win_r >= 0 ? (long long)len - p.Nq + p.win_r : LLONG_MAX;

    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    // ldmatrix row addresses: key rows (lane & 7) + 8 (lane >> 4) at chunk
    // offset (lane >> 3) & 1 for K; key rows (lane & 7) + 8 ((lane >> 3) & 1)
    // at chunk offset lane >> 4 for V (transposed).
    const int krow = (lane & 7) + ((lane >> 4) << 3), kch = (lane >> 3) & 1;
    const int vrow = (lane & 7) + (((lane >> 3) & 1) << 3), vch = lane >> 4;

    for (int it = 0;; ++it) {
        const int b = warp + kDecWarps * it;
        if (b >= nb) break;
        const int nxt = b + kDecWarps * (kStages - 1);
        if (nxt < nb) load_block(nxt, (it + kStages - 1) % kStages);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint32_t sK = ring + (it % kStages) * C::kStageBytes, sV = sK + C::kBlockBytes;
        const int base = k0 + b * kKeys;

        // S = Q K^T for 16 rows x 16 keys (two 8-key halves), in log2 units.
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t kb[4];
            ldsm_x4(kb, sK + C::swz(krow, 2 * ks + kch));
            mma16816<T>(s[0], qa[ks], kb[0], kb[1]);
            mma16816<T>(s[1], qa[ks], kb[2], kb[3]);
        }
        const bool full_block = base >= vis_lo && (long long)base + kKeys - 1 <= vis_hi && base + kKeys <= k1;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[h][e] *= p.scale_log2;
                if (!full_block) {
                    const int j = base + 8 * h + 2 * q4 + (e & 1);
                    const int r = g + 8 * (e >> 1);
                    if (j >= k1 || !dec_visible(p, r % p.Nq, j, len)) s[h][e] = -INFINITY;
                }
            }

        // Online softmax per row (g: elements 0, 1; g + 8: elements 2, 3); the
        // four lanes of a quad hold one row's 16 scores.  The reference max
        // moves lazily, only when the block's max passes it by kTauDec.
        uint32_t pa[4], pl[4];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float mx = fmaxf(fmaxf(s[0][2 * hr], s[0][2 * hr + 1]), fmaxf(s[1][2 * hr], s[1][2 * hr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            if (mx > m[hr] + kTauDec) {  // also the first finite max (m = -inf)
                const float a = m[hr] == -INFINITY ? 0.f : ptx::ex2(m[hr] - mx);
                l[hr] *= a;
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][2 * hr] *= a;
                    o[nd][2 * hr + 1] *= a;
                }
                m[hr] = mx;
            }
            const float neg = m[hr] == -INFINITY ? 0.f : -m[hr];
            const float p0 = ptx::ex2(s[0][2 * hr] + neg), p1 = ptx::ex2(s[0][2 * hr + 1] + neg);
            const float p2 = ptx::ex2(s[1][2 * hr] + neg), p3 = ptx::ex2(s[1][2 * hr + 1] + neg);
            l[hr] += (p0 + p1) + (p2 + p3);
            split16<T>(p0, p1, pa[hr], pl[hr]);          // keys 2 q4, +1 of the first 8
            split16<T>(p2, p3, pa[2 + hr], pl[2 + hr]);  // the same of the second 8
        }

        // O += P V: V rows are the K dimension (transposed ldmatrix), two
        // 8-column tiles of O per load.
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
            uint32_t vb[4];
            ldsm_x4_t(vb, sV + C::swz(vrow, nd + vch));
            mma16816<T>(o[nd], pa, vb[0], vb[1]);
            mma16816<T>(o[nd + 1], pa, vb[2], vb[3]);
            mma16816<T>(o[nd], pl, vb[0], vb[1]);
            mma16816<T>(o[nd + 1], pl, vb[2], vb[3]);
        }
        __syncwarp();  // this stage is refilled by a later iteration's copies
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring; it becomes the merge area

    // Per-warp state: the quad sums l; rows g and g + 8 of O.
    float* st = reinterpret_cast<float*>(dec_smem) + (size_t)warp * kDecodeMaxQ * (D + 2);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        float lv = l[hr];
        lv += __shfl_xor_sync(0xffffffffu, lv, 1);
        lv += __shfl_xor_sync(0xffffffffu, lv, 2);
        const int r = g + 8 * hr;
        if (r < rows) {
            float* row = st + r * (D + 2);
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                row[8 * nd + 2 * q4] = o[nd][2 * hr];
                row[8 * nd + 2 * q4 + 1] = o[nd][2 * hr + 1];
            }
            if (q4 == 0) {
                row[D] = m[hr];
                row[D + 1] = lv;
            }
        }
    }
    __syncthreads();
    constexpr int DV = D / 32;
    const float* dsm = reinterpret_cast<const float*>(dec_smem);
    for (int i = warp; i < rows; i += kDecWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, dsm[((size_t)w * kDecodeMaxQ + i) * (D + 2) + D]);
        float Lsum = 0.f, ov[DV];
#pragma unroll
        for (int e = 0; e < DV; ++e) ov[e] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kDecWarps; ++w) {
                const float* sw = dsm + ((size_t)w * kDecodeMaxQ + i) * (D + 2);
                const float a = sw[D] == -INFINITY ? 0.f : ptx::ex2(sw[D] - M);
                Lsum += a * sw[D + 1];
#pragma unroll
                for (int e = 0; e < DV; ++e) ov[e] = fmaf(a, sw[lane * DV + e], ov[e]);
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * kDecLn2 : -INFINITY;
        if (p.n_splits == 1) {
            T* ob = static_cast<T*>(p.o) + dec_qrow(p, bh, i, D) + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) ob[e] = from_float<T>(ov[e] * inv);
            if (p.lse && lane == 0) p.lse[(size_t)bh * rows + i] = lse;
        } else {
            const size_t prow = ((size_t)bh * p.n_splits + split) * rows + i;
            float* po = p.part_o + prow * D + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) po[e] = ov[e] * inv;
            if (lane == 0) p.part_lse[prow] = lse;
        }
    }
}


// One warp per output row: O = sum_s e^{LSE_s - LSE} O_s.  It is launched as a
// programmatic dependent of the split pass, so its CTAs can be resident before
// that pass ends; griddep_wait holds them until the partials are written.
template <typename T, int DV>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const DecodeParams p) {
    constexpr int D = 32 * DV;
    ptx::griddep_wait();
    const int lane = threadIdx.x & 31;
    const int rows = p.G * p.Nq;
    const long long rowid = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (rowid >= (long long)p.BH * rows) return;
    const long long bh = rowid / rows;
    const int i = (int)(rowid % rows);
    float M = -INFINITY;
    for (int s = lane; s < p.n_splits; s += 32) M = fmaxf(M, p.part_lse[((size_t)bh * p.n_splits + s) * rows + i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float o[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) o[e] = 0.f;
    float L = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < p.n_splits; ++s) {
            const size_t prow = ((size_t)bh * p.n_splits + s) * rows + i;
            const float ls = p.part_lse[prow];
            if (ls == -INFINITY) continue;
            const float w = expf(ls - M);
            L += w;
            const float* po = p.part_o + prow * D + lane * DV;
#pragma unroll
            for (int e = 0; e < DV; ++e) o[e] = fmaf(w, po[e], o[e]);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    T* ob = static_cast<T*>(p.o) + dec_qrow(p, bh, i, D) + lane * DV;
#pragma unroll
    for (int e = 0; e < DV; ++e) ob[e] = from_float<T>(o[e] * inv);
    if (p.lse && lane == 0) p.lse[rowid] = L > 0.f ? M + logf(L) : -INFINITY;
}

template <typename T, int DV, int NQ>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t s) {
    constexpr int D = 32 * DV;
    const long long blocks = (long long)p.BH * p.n_splits;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * kDecWarps * NQ * (D + 2);
    auto kern = fa_decode_split_kernel<T, DV, NQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kDecThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_rows(const DecodeParams& p, cudaStream_t s) {
    const long long blocks = (long long)p.BH * p.n_splits;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * kDecWarps * (32 / (D / 8)) * 4 * (D + 2);
    auto kern = fa_decode_rows_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kDecThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_mma(const DecodeParams& p, cudaStream_t s) {
    const long long blocks = (long long)p.BH * p.n_splits;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    constexpr int smem = mmadec::Cfg<D>::kSmem;
    auto kern = fa_decode_mma_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kDecThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// One query row: the one-key-per-warp kernel.  Two or more rows: with 16-bit
// inputs the tensor-core kernel; fp32 keeps the CUDA-core kernels (the lane-
// group one for up to four rows), whose per-row register arrays are sized by
// these buckets.
template <typename T, int DV>
cudaError_t launch_typed(const DecodeParams& p, cudaStream_t s) {
    const int rows = p.G * p.Nq;
    constexpr bool k16 = !std::is_same<T, float>::value;
    cudaError_t e = rows == 1         ? launch_split<T, DV, 1>(p, s)
                    : k16             ? launch_mma<T, 32 * DV>(p, s)
                    : rows <= 4       ? launch_rows<T, 32 * DV>(p, s)
                                      : launch_split<T, DV, kDecodeMaxQ>(p, s);
    if (e != cudaSuccess || p.n_splits == 1) return e;
    const long long all_rows = (long long)p.BH * rows;
    if ((all_rows + 3) / 4 > 0x7fffffffLL) return cudaErrorInvalidValue;
    // Programmatic stream serialization: the combine grid launches while the
    // split pass drains instead of after it, hiding its launch latency.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((all_rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<T, DV>, p);
}

template <typename Kern>
int resident_ctas(Kern kern, size_t smem) {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecThreads, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace

int decode_ctas_per_sm(int rows, int D) {
    // The 16-bit instantiations stand for every dtype: the split plan (and so
    // the workspace size) must not depend on the element type.
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev][3][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    const int cls = rows == 1 ? 0 : 1;
    const int di = D == 128 ? 1 : 0;
    int n = cache[dev][cls][di].load(std::memory_order_relaxed);
    if (n > 0) return n;
    using T = __nv_bfloat16;
    if (cls == 0)
        n = di ? resident_ctas(fa_decode_split_kernel<T, 4, 1>, sizeof(float) * kDecWarps * 1 * (128 + 2))
               : resident_ctas(fa_decode_split_kernel<T, 2, 1>, sizeof(float) * kDecWarps * 1 * (64 + 2));
    else
        n = di ? resident_ctas(fa_decode_mma_kernel<T, 128>, mmadec::Cfg<128>::kSmem)
               : resident_ctas(fa_decode_mma_kernel<T, 64>, mmadec::Cfg<64>::kSmem);
    if (n > 0) cache[dev][cls][di].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype_code, cudaStream_t s) {
    const int dv = p.D / 32;
    switch (dtype_code) {
        case 0: return dv == 4 ? launch_typed<__half, 4>(p, s) : launch_typed<__half, 2>(p, s);
        case 1: return dv == 4 ? launch_typed<__nv_bfloat16, 4>(p, s) : launch_typed<__nv_bfloat16, 2>(p, s);
        default: return dv == 4 ? launch_typed<float, 4>(p, s) : launch_typed<float, 2>(p, s);
    }
}


// ---------------------------------------------------------------------------
// Decode without any allocation.
//
// Some callers cannot allocate device memory at the moment they need attention:
// code running inside an allocator or memory-pool callback, a runtime that has
// handed all device memory to its own pool and forbids cudaMalloc/cudaFree on
// the hot path (a cudaMalloc there can block on the device or fail), or a
// plugin host that gives the library nothing but its input and output buffers.
// fa_decode_noalloc serves them: the split-K partial results live in a fixed
// array compiled into this library instead of a caller workspace.
namespace {

// Room for the fp32 partials (O rows plus their log-sum-exps) of one call.
constexpr unsigned long long kNoAllocScratchBytes = 16ull << 20;  // 16 MiB on every device that loads the library
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
    std::once_flag once;
    void* scratch = nullptr;  // device address of g_decode_scratch on this device
    int sms = 0;
    cudaError_t err = cudaSuccess;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

bool na_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int fa_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int Nq, int Nk, int D, float scale, int mask_kind, int win_l, int win_r, int dtype,
                                 int n_splits, void* stream) {
    if (!q || !k || !v || !o) return FA_ERR_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || D <= 0 || Nq > Nk) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    int wl, wr;
    switch (mask_kind) {
        case FA_MASK_NONE: wl = -1; wr = -1; break;
        case FA_MASK_CAUSAL: wl = -1; wr = 0; break;
        case FA_MASK_WINDOW:
            if (win_l < -1 || win_r < -1) return FA_ERR_ARG;
            wl = win_l;
            wr = win_r;
            break;
        default: return FA_ERR_ARG;
    }
    if ((long long)B * H > 0x7fffffffLL) return FA_ERR_ARG;
    if (dtype < FA_F16 || dtype > FA_F32 || (D != 64 && D != 128) || Nq > kDecodeMaxQ) return FA_ERR_UNSUPPORTED;
    if (!na_aligned(q, 16) || !na_aligned(k, 16) || !na_aligned(v, 16) || !na_aligned(o, 16)) return FA_ERR_ALIGN;
    if (lse && !na_aligned(lse, 4)) return FA_ERR_ALIGN;

    // Set-up, once per device, with that device current: the host-side name of
    // the array is not a device address, so ask the runtime for the real one.
    int dev = 0;
    const cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return record_cuda_error(de);
    if (dev < 0 || dev >= kNoAllocMaxDevices) return record_cuda_error(cudaErrorInvalidDevice);
    NoAllocDevice& nd = g_noalloc_dev[dev];
    std::call_once(nd.once, [&] {
        nd.err = cudaGetSymbolAddress(&nd.scratch, g_decode_scratch);
        if (nd.err == cudaSuccess) nd.err = cudaDeviceGetAttribute(&nd.sms, cudaDevAttrMultiProcessorCount, dev);
        if (nd.err == cudaSuccess && !nd.scratch) nd.err = cudaErrorInvalidSymbol;
    });
    // A failed set-up is cached; every later call reports its error again.
    if (nd.err != cudaSuccess) return record_cuda_error(nd.err);

    DecodeParams p;
    p.BH = (long long)B * H;
    decode_plan(p.BH, Nk, nd.sms, n_splits, &p.n_splits, &p.chunk);
    const unsigned long long need = decode_workspace_bytes(p.BH, Nq, D, p.n_splits);
    if (need > kNoAllocScratchBytes) return FA_ERR_SCRATCH;
    p.part_o = nullptr;
    p.part_lse = nullptr;
    if (need > 0) {
        // Every partial row is written before it is read, so nothing in the
        // array needs clearing between calls.
        p.part_o = static_cast<float*>(nd.scratch);
        p.part_lse = reinterpret_cast<float*>(static_cast<char*>(nd.scratch) +
                                              ((unsigned long long)p.BH * p.n_splits * Nq * D * 4 + 255) / 256 * 256);
    }
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.Nq = Nq;
    p.Nk = Nk;
    p.D = D;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.win_l = wl;
    p.win_r = wr;
    const cudaError_t e = launch_decode(p, dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : record_cuda_error(e);
}

extern "C" unsigned long long fa_decode_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

}  // namespace fa
