// fp32 fused attention forward on the FFMA pipe (no tensor cores: TF32 would
// not hold a 1e-5 error bound).
//
// Same method as the tensor-core kernel -- key tiles streamed through shared
// memory, a running row max and row sum, one division at the end -- as in
// "Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention", section 4.2 (fp32 kernel: Q block in shared
// memory, K/V blocks loaded per step, masked scores, online update), with
// the update written in its consistent form (section 1.2 identity).
//
// Block: 128 threads = 4 warps, 32 query rows of one (b, h); each warp owns
// 8 rows.  A key tile holds 32 keys: lane l scores key l, then the warp
// updates the row's running max / sum and its D-wide accumulator, each lane
// owning output columns lane, lane + 32, ...
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRows = 32;     // query rows per block
constexpr int kKeys = 32;     // keys per tile
constexpr int kMaxD = 128;
constexpr int kRowsPerWarp = 8;

__device__ __forceinline__ bool visible(const Geom& g, int i, int j) {
    if (j >= g.N) return false;
    if (g.win_l >= 0 && j < i - g.win_l) return false;
    if (g.win_r >= 0 && j > i + g.win_r) return false;
    return true;
}

__global__ void __launch_bounds__(128) fa_fwd_simt_f32_kernel(const SimtParams p) {
    extern __shared__ float sm[];
    const int D = p.D;
    const int ld = D + 1;                     // padded row stride: conflict-free column walks
    float* sq = sm;                           // [kRows][ld]
    float* sk = sq + kRows * ld;              // [kKeys][ld]
    float* sv = sk + kKeys * ld;              // [kKeys][D]

    const int N = p.g.N;
    const int n_rb = (N + kRows - 1) / kRows;
    const int bh = blockIdx.x / n_rb;
    const int r0 = (blockIdx.x % n_rb) * kRows;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = bh / p.H, h = bh % p.H, hk = h / p.G, Hkv = p.H / p.G;
    auto qrow = [&](int i) { return (size_t)row_index(p.layout, b, h, i, p.H, N) * D; };
    auto krow = [&](int j) { return (size_t)row_index(p.layout, b, hk, j, Hkv, N) * D; };

    for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        sq[r * ld + d] = (r0 + r < N) ? p.q[qrow(r0 + r) + d] : 0.f;
    }

    // Key range of this row block.
    const int r1 = min(N, r0 + kRows);
    int kmin = p.g.win_l < 0 ? 0 : max(0, r0 - p.g.win_l);
    long long kmax = p.g.win_r < 0 ? (long long)N - 1 : min((long long)N - 1, (long long)(r1 - 1) + p.g.win_r);
    const int t_lo = kmin / kKeys;
    const int t_hi = (int)(kmax / kKeys) + 1;

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxD / 32];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) acc[rr][c] = 0.f;
    }

    for (int t = t_lo; t < t_hi; ++t) {
        const int k0 = t * kKeys;
        __syncthreads();
        for (int idx = threadIdx.x; idx < kKeys * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            const bool in = k0 + r < N;
            sk[r * ld + d] = in ? p.k[krow(k0 + r) + d] : 0.f;
            sv[r * D + d] = in ? p.v[krow(k0 + r) + d] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const int i = r0 + r;
            if (i >= N) continue;                      // warp-uniform
            const int j = k0 + lane;
            float s = -INFINITY;
            if (visible(p.g, i, j)) {
                float dot = 0.f;
                for (int d = 0; d < D; ++d) dot = fmaf(sq[r * ld + d], sk[lane * ld + d], dot);
                s = dot * p.scale;
            }
            float mx = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_new = fmaxf(m[rr], mx);
            if (m_new == -INFINITY) continue;          // nothing visible yet (warp-uniform)
            const float alpha = m[rr] == -INFINITY ? 0.f : expf(m[rr] - m_new);
            const float pj = s == -INFINITY ? 0.f : expf(s - m_new);
            float ps = pj;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l[rr] = l[rr] * alpha + ps;
            m[rr] = m_new;
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) acc[rr][c] *= alpha;
            for (int jj = 0; jj < kKeys; ++jj) {
                const float w = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
                for (int c = 0; c < kMaxD / 32; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) acc[rr][c] = fmaf(w, sv[jj * D + d], acc[rr][c]);
                }
            }
        }
    }

#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int i = r0 + warp * kRowsPerWarp + rr;
        if (i >= N) continue;
        const bool live = l[rr] > 0.f;
        const float inv = live ? 1.f / l[rr] : 0.f;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) {
            const int d = lane + 32 * c;
            if (d < D) p.o[qrow(i) + d] = acc[rr][c] * inv;
        }
        if (lane == 0 && p.lse) p.lse[(size_t)bh * N + i] = live ? m[rr] + logf(l[rr]) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_simt_f32(const SimtParams& p, cudaStream_t s) {
    const int ld = p.D + 1;
    const size_t smem = sizeof(float) * ((size_t)kRows * ld + (size_t)kKeys * ld + (size_t)kKeys * p.D);
    const long long blocks = (long long)((p.g.N + kRows - 1) / kRows) * p.BH;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_simt_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fa_fwd_simt_f32_kernel<<<(unsigned)blocks, 128, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
