// Rotary position embedding of Q and K: one streaming pass in HBM.
//
// "Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention", section 9 ("Extensions: integration with RoPE
// and a paged KV cache"), applies the rotation to Q and K from a cos/sin
// table.  Row n of a tensor sits at position pos0 + n; its pair i, (x_a, x_b),
// turns by the table entry (p, i):
//     x_a' = x_a cos - x_b sin,   x_b' = x_b cos + x_a sin
// with pairs (i, i + D/2) (half-split) or (2i, 2i + 1) (interleaved).
//
// One thread takes one (tensor, batch, chunk of four heads, position, group
// of 8 pairs): it loads the group's 8 cos and 8 sin once and rotates that
// position's rows of the four heads, so the table is read once per four rows.
// Consecutive threads take consecutive groups of one row and then the next
// position, so each warp reads and writes whole rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "rope_math.cuh"

namespace fa {
namespace {

// Eight consecutive elements as fp32, and back.
template <typename T>
struct Vec8;

template <>
struct Vec8<float> {
    static __device__ __forceinline__ void load(const float* p, float* f) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* f) {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};

template <>
struct Vec8<__half> {
    static __device__ __forceinline__ void load(const __half* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
            f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
        }
    }
    static __device__ __forceinline__ void store(__half* p, const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)__half_as_ushort(__float2half_rn(f[2 * i])) |
                   ((uint32_t)__half_as_ushort(__float2half_rn(f[2 * i + 1])) << 16);
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i])) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i + 1])) << 16);
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

constexpr int kHeadsPerItem = 4;

template <typename T, int kStyle>
__global__ void __launch_bounds__(256) fa_rope_kernel(const RopeParams p) {
    const int G = p.D / 16;  // groups of 8 pairs per row
    const int half = p.D / 2;
    const int hc0 = (p.heads[0] + kHeadsPerItem - 1) / kHeadsPerItem;
    const int hc1 = (p.heads[1] + kHeadsPerItem - 1) / kHeadsPerItem;
    const long long items0 = p.x[0] ? (long long)p.B * hc0 * p.n[0] * G : 0;
    const long long items1 = p.x[1] ? (long long)p.B * hc1 * p.n[1] * G : 0;
    const long long total = items0 + items1;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < total;
         w += (long long)gridDim.x * blockDim.x) {
        // item = (tensor, b, chunk of kHeadsPerItem heads, position i, group g),
        // g fastest, then i: a warp covers whole consecutive rows of one head
        const int t = w < items0 ? 0 : 1;
        const long long lw = t ? w - items0 : w;
        const int g = (int)(lw % G);
        long long rest = lw / G;
        // selects, not indexing: a run-time index into the parameter arrays
        // would copy them to local memory
        const int N = t ? p.n[1] : p.n[0];
        const int i = (int)(rest % N);
        rest /= N;
        const int hcn = t ? hc1 : hc0;
        const int hc = (int)(rest % hcn);
        const int b = (int)(rest / hcn);
        const int heads = t ? p.heads[1] : p.heads[0];
        const long long pos = (long long)(t ? p.pos0[1] : p.pos0[0]) + i;

        float c[8], s[8];
        Vec8<float>::load(p.cos + pos * half + 8 * g, c);
        Vec8<float>::load(p.sin + pos * half + 8 * g, s);
        // element offsets of the two 8-element vectors this group rotates
        const int oa = kStyle == ROPE_HALF ? 8 * g : 16 * g;
        const int ob = kStyle == ROPE_HALF ? half + 8 * g : 16 * g + 8;
        const T* x = static_cast<const T*>(t ? p.x[1] : p.x[0]);
        T* y = static_cast<T*>(t ? p.y[1] : p.y[0]);
#pragma unroll
        for (int hh = 0; hh < kHeadsPerItem; ++hh) {
            const int h = hc * kHeadsPerItem + hh;
            if (h >= heads) break;
            const long long r = row_index(p.layout, b, h, i, heads, N) * p.D;
            float u[8], v[8];
            Vec8<T>::load(x + r + oa, u);
            Vec8<T>::load(x + r + ob, v);
            float yu[8], yv[8];
            if (kStyle == ROPE_HALF) {
                // pair m: (u[m], v[m]) with table column 8g + m
#pragma unroll
                for (int m = 0; m < 8; ++m) rope_rotate(u[m], v[m], c[m], s[m], yu[m], yv[m]);
            } else {
                // pairs (u[2m], u[2m+1]) with column 8g + m, (v[2m], v[2m+1]) with 8g + 4 + m
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    rope_rotate(u[2 * m], u[2 * m + 1], c[m], s[m], yu[2 * m], yu[2 * m + 1]);
                    rope_rotate(v[2 * m], v[2 * m + 1], c[4 + m], s[4 + m], yv[2 * m], yv[2 * m + 1]);
                }
            }
            Vec8<T>::store(y + r + oa, yu);
            Vec8<T>::store(y + r + ob, yv);
        }
    }
}

// cos/sin (p * base^(-2i/D)) in double precision, rounded once to fp32.
__global__ void __launch_bounds__(256) fa_rope_tables_kernel(float* cos_tab, float* sin_tab, int n_pos, int D,
                                                            double base) {
    const int half = D / 2;
    const long long total = (long long)n_pos * half;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(e % half);
        const long long pos = e / half;
        const double theta = pow(base, -2.0 * i / D);
        double sv, cv;
        sincos((double)pos * theta, &sv, &cv);
        cos_tab[e] = (float)cv;
        sin_tab[e] = (float)sv;
    }
}

template <typename T, int kStyle>
cudaError_t launch_styled(const RopeParams& p, long long items, int sms, cudaStream_t s) {
    // every CTA resident at once, each thread striding over many small items,
    // so no partial last wave leaves SMs idle
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fa_rope_kernel<T, kStyle>, 256, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    long long grid = (items + 255) / 256;
    if (grid > (long long)per_sm * sms) grid = (long long)per_sm * sms;
    fa_rope_kernel<T, kStyle><<<(int)grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const RopeParams& p, long long items, int sms, cudaStream_t s) {
    return p.style == ROPE_HALF ? launch_styled<T, ROPE_HALF>(p, items, sms, s)
                                : launch_styled<T, ROPE_INTERLEAVED>(p, items, sms, s);
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int dtype_code, int sms, cudaStream_t s) {
    const int G = p.D / 16;
    auto items_of = [&](int t) {
        return p.x[t] ? (long long)p.B * ((p.heads[t] + kHeadsPerItem - 1) / kHeadsPerItem) * p.n[t] * G : 0LL;
    };
    const long long items = items_of(0) + items_of(1);
    if (items == 0) return cudaSuccess;
    switch (dtype_code) {
        case 0: return launch_typed<__half>(p, items, sms, s);
        case 1: return launch_typed<__nv_bfloat16>(p, items, sms, s);
        default: return launch_typed<float>(p, items, sms, s);
    }
}

cudaError_t launch_rope_tables(float* cos_tab, float* sin_tab, int n_pos, int D, double base, int sms,
                               cudaStream_t s) {
    const long long total = (long long)n_pos * (D / 2);
    long long grid = (total + 255) / 256;
    if (grid > 8LL * sms) grid = 8LL * sms;
    fa_rope_tables_kernel<<<(int)grid, 256, 0, s>>>(cos_tab, sin_tab, n_pos, D, base);
    return cudaGetLastError();
}

}  // namespace fa
