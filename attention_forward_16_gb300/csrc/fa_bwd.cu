// Tensor-core attention backward for sm_103a (fp16 / bf16 in, fp32 accumulate).
//
// The gradient of the attention definition of "Ascend C advanced practice:
// high-performance FlashAttention-2-style tile-level fused attention"
// (section 1.1), for the backward pass the ops-transformer walk-through says
// the operator also has.  With P = exp(scale * S - LSE) recomputed from the
// forward's LSE, and Dsum_i = rowsum(dO_i * O_i) (= rowsum(P * dP)):
//
//     dV = P^T dO      dP = dO V^T      dS = P * (dP - Dsum)
//     dK = scale * dS^T Q                dQ = scale * dS K
//
// Three kernels, no atomics, deterministic:
//   pre   one pass over O and dO: Dsum and LSE * log2(e) per row, padded to
//         whole 128-row tiles (HBM-bound);
//   dkdv  one CTA per (b, K/V head, 128-key tile): K and V stay in shared
//         memory, the query tiles of every query head of the group stream
//         through a TMA ring; TMEM holds S^T | dP^T | dV | dK;
//   dq    one CTA per (b, head, 128-row query tile): K/V tiles stream; the
//         stationary Q and dO rows sit in TMEM beside S | dP | dQ, so S and dP
//         are TS products that read only K and V from shared memory.
// The dq kernel recomputes S and dP rather than adding partial dQ tiles with
// atomics from the dkdv kernel: two more products per tile pair, in exchange
// for a deterministic result and no read-modify-write traffic in L2.
//
// Warp roles in both kernels (384 threads): warp 0 issues TMA loads, warp 1
// allocates TMEM and issues tcgen05.mma (the whole warp on one uniform path,
// one elected lane issuing), warps 4-11 turn
// scores into P and dS and write the result; warps 2-3 only take part in the
// CTA barriers.  Warps w and w + 4 share TMEM lanes 32 (w % 4) .. + 31 (one
// row per thread) and split the 128 columns of a tile: nothing in P or dS
// reduces over a row, so the halves never exchange values, and two warps per
// sub-partition hide the exponential's latency better than one.  Each half
// writes its 16-bit P or dS into the first columns of its own fp32 half, so
// neither overwrites values the other still reads; the products that read
// them from TMEM address the halves separately.  Every mbarrier wait is
// bounded, as in the forward kernel.
#include <atomic>
#include <cmath>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

constexpr int kParts = 2;                     // column parts of a tile row, one warp each
constexpr int kColsPerPart = 128 / kParts;
constexpr int kBwdThreads = 128 + 128 * kParts;
constexpr int kWarpTmaB = 0;
constexpr int kWarpMmaB = 1;
constexpr int kWarpEw0 = 4;  // first of the 4 * kParts elementwise warps
constexpr int kEwThreads = 128 * kParts;
constexpr float kLog2e = 1.4426950408889634074f;

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;                   // 128-byte column chunks per row
    static constexpr int kBoxBytes = kTileM * 64 * 2;        // one TMA box: 128 rows x 64 elements
    static constexpr int kTileBytes = kChunks * kBoxBytes;   // 128 rows x D
    static constexpr int kVecBytes = kTileM * 4;             // 128 fp32 per-row values
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr int kStagesQ = D == 128 ? 3 : 4;       // dq ring: Q and dO live in TMEM
    // dkdv ring stage: Q tile | dO tile | LSE*log2e | Dsum (a multiple of 1024 bytes)
    static constexpr int kStageKV = 2 * kTileBytes + 1024;
    // dq ring stage: K tile | V tile
    static constexpr int kStageQ = 2 * kTileBytes;
    static constexpr int kColS = 0;
    static constexpr int kColDP = 128;
    static constexpr int kColA = 256;       // dV (dkdv) or dQ (dq)
    static constexpr int kColB = 256 + D;   // dK (dkdv)
    static constexpr int kColQ = 256 + D;   // dq: Q, 16-bit pairs (D / 2 columns)
    static constexpr int kColDO = 256 + D + D / 2;  // dq: dO, likewise
    static constexpr int kTmemCols = 512;
};

struct __align__(16) BwdCtl {
    uint64_t fixed_full;
    uint64_t qd_full;  // dq: Q and dO rows stored in TMEM (one arrival per elementwise thread)
    uint64_t ring_full[4], ring_empty[4];
    // Per column part of a tile in the dQ kernel (its 64 keys of S and dP),
    // whose parts run on their own barriers; the dK/dV kernel uses index 0.
    uint64_t s_full[kParts], s_free[kParts], dp_full[kParts], p_full[kParts], ds_full[kParts];
    uint64_t acc_done, drain;
    uint64_t kv_free, acc_free;  // dK/dV: K and V reusable; dV and dK read out of TMEM
    uint32_t tmem_base;
    int abort;
};

template <int D>
constexpr int dkdv_smem_bytes() {
    return 2 * BwdCfg<D>::kTileBytes + BwdCfg<D>::kStages * BwdCfg<D>::kStageKV + (int)sizeof(BwdCtl) + 1024;
}
template <int D>
constexpr int dq_smem_bytes() {
    return BwdCfg<D>::kStagesQ * BwdCfg<D>::kStageQ + (int)sizeof(BwdCtl) + 1024;
}
static_assert(BwdCfg<128>::kStagesQ <= 4 && BwdCfg<64>::kStagesQ <= 4, "ring barriers");
static_assert(BwdCfg<128>::kColDO + 64 <= BwdCfg<128>::kTmemCols && BwdCfg<64>::kColDO + 32 <= 512, "TMEM (dq)");
static_assert(dkdv_smem_bytes<128>() <= 227 * 1024 && dq_smem_bytes<128>() <= 227 * 1024, "smem (D=128)");
static_assert(dkdv_smem_bytes<64>() <= 227 * 1024 && dq_smem_bytes<64>() <= 227 * 1024, "smem (D=64)");

// One 128-row tile (all D columns, as D/64 swizzled 128-byte-wide blocks) in
// one TMA instruction: the 5-D map's coordinates are (column, row, chunk,
// head, batch) in either layout.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int layout, int b,
                                          int head, int row) {
    (void)layout;
    tma_load_5d(dst, tm, bar, 0, row, 0, head, b);
}

// Products shared by both kernels.  A tiles are K-major 128 x D (TMA boxes
// with the 128-byte swizzle); "MN-major" B tiles are the same boxes read as
// [K = 128 rows] x [N = D columns].
template <int D, bool kBf16>
struct Mma {
    static constexpr uint32_t kIdescRows = make_idesc(kBf16, kTileM, kTileN, false);  // 128 x 128, K = D
    static constexpr uint32_t kIdescCols = make_idesc(kBf16, kTileM, D, true);         // 128 x D, K = 128
    static constexpr uint32_t kIdescPart = make_idesc(kBf16, kTileM, kColsPerPart, false);  // 128 x 64, K = D
    // dst[128 x 128] = A[128 x D] B[128 x D]^T, both from shared memory.
    // Called by the whole issuing warp; `leader` (one elected lane) issues.
    // Descriptors advance by encoded offsets (address / 16 in the low field;
    // shared addresses stay below 256 KiB, so the add never leaves the field).
    static __device__ __forceinline__ void rows(uint32_t dst, uint32_t a, uint32_t b, bool leader) {
        const uint64_t ad = make_sdesc(a, 16, 1024), bd = make_sdesc(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * BwdCfg<D>::kBoxBytes + (kk % 4) * 32) >> 4;
            if (leader) mma_ss(dst, ad + off, bd + off, kIdescRows, kk > 0);
        }
    }
    // Part h of dst[128 x 128] = A[128 x D] B[128 x D]^T with A in TMEM as
    // 16-bit pairs (a TS product: only B is read from shared memory): its 64
    // columns dst[:, 64h, 64h + 64) from rows [64h, 64h + 64) of B, which
    // start 8 swizzle atoms into each column chunk.
    static __device__ __forceinline__ void rows_part_t(uint32_t dst, uint32_t ta, uint32_t b, int h, bool leader) {
        const uint64_t bd = make_sdesc(b, 16, 1024) + (uint64_t)((h * kColsPerPart * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * BwdCfg<D>::kBoxBytes + (kk % 4) * 32) >> 4;
            if (leader) mma_ts(dst + h * kColsPerPart, ta + kk * 8, bd + off, kIdescPart, kk > 0);
        }
    }
    // dst[128 x D] (+)= T_h[128 x 64] B_h[64 x D]: part h of cols() below.
    static __device__ __forceinline__ void cols_part(uint32_t dst, uint32_t t, uint32_t b, int h, bool acc,
                                                     bool leader) {
        constexpr int kSteps = kColsPerPart / 16;
        const uint64_t bd = make_sdesc(b, BwdCfg<D>::kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            if (leader)
                mma_ts(dst, t + h * kColsPerPart + kk * 8, bd + (uint64_t)((h * kSteps + kk) * (2048 >> 4)),
                       kIdescCols, (acc || kk > 0) ? 1u : 0u);
        }
    }
    // dst[128 x D] (+)= T[128 x 128] B[128 x D]: T 16-bit in TMEM, its K
    // columns of part c, [c P, c P + P) with P = kColsPerPart, packed at TMEM
    // column t + c P (P / 2 columns).
    static __device__ __forceinline__ void cols(uint32_t dst, uint32_t t, uint32_t b, bool acc, bool leader) {
        constexpr int kSteps = kColsPerPart / 16;  // K-steps of 16 per part
        const uint64_t bd = make_sdesc(b, BwdCfg<D>::kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
            if (leader)
                mma_ts(dst, t + (kk / kSteps) * kColsPerPart + (kk % kSteps) * 8, bd + (uint64_t)(kk * (2048 >> 4)),
                       kIdescCols, (acc || kk > 0) ? 1u : 0u);
        }
    }
};

// `ew_count`: arrivals that complete an elementwise barrier (every
// elementwise thread, or one part's threads where the parts run apart).
__device__ __forceinline__ void init_ctl(BwdCtl* sh, int ring_empty_count, int ew_count) {
    mbar_init(smem_u32(&sh->fixed_full), 1);
    mbar_init(smem_u32(&sh->qd_full), kEwThreads);
    for (int s = 0; s < 4; ++s) {
        mbar_init(smem_u32(&sh->ring_full[s]), 1);
        mbar_init(smem_u32(&sh->ring_empty[s]), ring_empty_count);
    }
    for (int h = 0; h < kParts; ++h) {
        mbar_init(smem_u32(&sh->s_full[h]), 1);
        mbar_init(smem_u32(&sh->s_free[h]), ew_count);
        mbar_init(smem_u32(&sh->dp_full[h]), 1);
        mbar_init(smem_u32(&sh->p_full[h]), ew_count);
        mbar_init(smem_u32(&sh->ds_full[h]), ew_count);
    }
    mbar_init(smem_u32(&sh->acc_done), 1);
    mbar_init(smem_u32(&sh->drain), 1);
    mbar_init(smem_u32(&sh->kv_free), 1);
    mbar_init(smem_u32(&sh->acc_free), kEwThreads);
    sh->abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
}

// Four floats from shared memory at a shared-space address.  The per-query
// values sit behind a pointer the compiler cannot prove to be shared (the
// dynamic shared base is rounded up through an integer), so a plain load
// would be a generic one; naming the space took the dK/dV kernel's P phase
// from about 2,200 to 1,700 cycles per tile.  Volatile, so the loads never
// move above the barrier wait that makes the TMA copy visible.
__device__ __forceinline__ float4 lds_f4(const void* p) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

constexpr int kChunks = kColsPerPart / 32;  // 32-column TMEM loads per part

// A thread's part of a row (kColsPerPart fp32 values) from TMEM into registers.
__device__ __forceinline__ void ld_part(uint32_t t, uint32_t (&r)[kChunks][32]) {
#pragma unroll
    for (int c = 0; c < kChunks; ++c) tmem_ld32(t + 32 * c, r[c]);
    tmem_wait_ld();
}

// Store part `pt`'s 32-column chunks (pt, pt + kParts, ...) of a thread's row
// of a 16-bit gradient (fp32 in TMEM, times `mul`).
template <int D, bool kBf16>
__device__ __forceinline__ void store_row(uint32_t t, void* out, size_t row, int pt, float mul, bool live) {
#pragma unroll 1
    for (int c = pt; c < D / 32; c += kParts) {
        uint32_t v[32];
        tmem_ld32(t + c * 32, v);
        tmem_wait_ld();
        if (live) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row * D + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack2<kBf16>(u2f(v[8 * i]) * mul, u2f(v[8 * i + 1]) * mul),
                                    pack2<kBf16>(u2f(v[8 * i + 2]) * mul, u2f(v[8 * i + 3]) * mul),
                                    pack2<kBf16>(u2f(v[8 * i + 4]) * mul, u2f(v[8 * i + 5]) * mul),
                                    pack2<kBf16>(u2f(v[8 * i + 6]) * mul, u2f(v[8 * i + 7]) * mul));
        }
    }
}

template <int D>
__device__ __forceinline__ void zero_row(void* out, size_t row, int pt) {
    for (int c = pt; c < D / 32; c += kParts) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row * D + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    }
}

// ===================================================================== dK, dV
// A dK/dV CTA takes `per_cta` consecutive key tiles of the (b, K/V head)-
// major order, one after the other.  The CTA's set-up is paid once, and the
// next tile's K/V loads and first S^T / dP^T products run while the
// elementwise warps write out the previous tile's dK and dV.  Under a mask
// the tiles' lengths differ and one tile per CTA balances better; without,
// dkdv_tiles_per_cta picks the count (at most kDkdvMaxTiles).
constexpr int kDkdvMaxTiles = 4;

template <int D, bool kBf16, bool kMask>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p,
                                                                      const int n_work, const int per_cta) {
    using C = BwdCfg<D>;
    using M = Mma<D, kBf16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sK = smem_u32(smem);
    const uint32_t sV = sK + C::kTileBytes;
    const uint32_t sRing = sV + C::kTileBytes;
    BwdCtl* sh = reinterpret_cast<BwdCtl*>(smem + 2 * C::kTileBytes + C::kStages * C::kStageKV);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);  // warp-uniform to the compiler
    const int lane = threadIdx.x & 31;

    // Key tile w -> (b, K/V head, j), its query tiles [ilo, ihi) and its
    // (query head of the group, query tile) items, head-major.  Every role
    // derives the same sequence, and tiles without items are skipped by all
    // but the elementwise warps (which write their zero gradients).
    struct Tile {
        int j, b, hk, ilo, ni, n_items;
    };
    auto tile = [&](int t) {
        Tile tl;
        const int w = per_cta * (int)blockIdx.x + t;
        tl.j = w % p.n_tiles;
        const int bk = w / p.n_tiles;
        tl.b = bk / p.Hkv;
        tl.hk = bk % p.Hkv;
        int ihi;
        q_tile_range(p.g, tl.j, tl.ilo, ihi);
        tl.ni = ihi - tl.ilo;
        tl.n_items = tl.ni * p.G;
        return tl;
    };
    // (the masked build always takes one tile: a compile-time count lets the
    // compiler drop the cross-tile waits)
    const int n_mine = kMask ? 1
                             : (n_work - per_cta * (int)blockIdx.x < per_cta ? n_work - per_cta * (int)blockIdx.x
                                                                             : per_cta);

    if (threadIdx.x == 0) init_ctl(sh, 1, kEwThreads);
    if (warp == kWarpMmaB) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, sh->tmem_base, 0);
    const Waiter W{&sh->abort, p.status, p.wait_limit_ns};

    if (warp == kWarpTmaB && lane == 0) {
        // ------------------------------------------------------------ TMA
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_do);
        const uint32_t fixed = smem_u32(&sh->fixed_full);
        bool ok = true;
        int g = 0;   // ring position across tiles
        int ti = 0;  // tiles with items so far
        for (int t = 0; t < n_mine && ok; ++t) {
            const Tile tl = tile(t);
            if (tl.n_items == 0) continue;
            // K and V of the previous tile are free once its last S^T and dP^T
            // have completed.
            if (ti > 0 && !(ok = W.wait(smem_u32(&sh->kv_free), (ti - 1) & 1))) break;
            mbar_arrive_expect_tx(fixed, 2 * C::kTileBytes);
            load_tile<D>(sK, &p.tm_k, fixed, p.layout, tl.b, tl.hk, tl.j * kTileN);
            load_tile<D>(sV, &p.tm_v, fixed, p.layout, tl.b, tl.hk, tl.j * kTileN);
            ++ti;
            for (int n = 0; n < tl.n_items && ok; ++n, ++g) {
                const int st = g % C::kStages;
                if (g >= C::kStages && !(ok = W.wait(smem_u32(&sh->ring_empty[st]), ((g / C::kStages) - 1) & 1)))
                    break;
                const int h = tl.hk * p.G + n / tl.ni, i = tl.ilo + n % tl.ni;
                const uint32_t full = smem_u32(&sh->ring_full[st]);
                const uint32_t stage = sRing + st * C::kStageKV;
                mbar_arrive_expect_tx(full, 2 * C::kTileBytes + 2 * C::kVecBytes);
                load_tile<D>(stage, &p.tm_q, full, p.layout, tl.b, h, i * kTileM);
                load_tile<D>(stage + C::kTileBytes, &p.tm_do, full, p.layout, tl.b, h, i * kTileM);
                const size_t vrow = ((size_t)tl.b * p.H + h) * p.Npad + (size_t)i * kTileM;
                bulk_load(stage + 2 * C::kTileBytes, p.lse2 + vrow, C::kVecBytes, full);
                bulk_load(stage + 2 * C::kTileBytes + C::kVecBytes, p.dsum + vrow, C::kVecBytes, full);
            }
        }
        // let every issued copy land before the CTA releases shared memory
        if (ti > 0) W.drain(fixed, (ti - 1) & 1);
        for (int m = g - C::kStages < 0 ? 0 : g - C::kStages; m < g; ++m)
            W.drain(smem_u32(&sh->ring_full[m % C::kStages]), (m / C::kStages) & 1);
    } else if (warp == kWarpMmaB) {
        // ------------------------------------------------------------ MMA
        // The whole warp follows one path; the elected lane issues.
        const bool leader = elect_one();
        const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP;
        const uint32_t tDV = tmem + C::kColA, tDK = tmem + C::kColB;
        auto stage = [&](int g) { return sRing + (g % C::kStages) * C::kStageKV; };
        auto ring_full = [&](int g) {
            return W.wait_warp(smem_u32(&sh->ring_full[g % C::kStages]), (g / C::kStages) & 1);
        };
        bool ok = true;
        int g = 0;   // ring position (and item count) across tiles
        int ti = 0;
        for (int t = 0; t < n_mine && ok; ++t) {
            const Tile tl = tile(t);
            if (tl.n_items == 0) continue;
            if (!(ok = W.wait_warp(smem_u32(&sh->fixed_full), ti & 1) && ring_full(g))) break;
            tc_fence_after();
            M::rows(tS, sK, stage(g), leader);                       // S^T = K Q^T
            if (leader) mma_commit(smem_u32(&sh->s_full[0]));
            M::rows(tDP, sV, stage(g) + C::kTileBytes, leader);      // dP^T = V dO^T
            if (leader) mma_commit(smem_u32(&sh->dp_full[0]));
            for (int n = 0; n < tl.n_items && ok; ++n, ++g) {
                if (!(ok = W.wait_warp(smem_u32(&sh->p_full[0]), g & 1))) break;
                // dV and dK of the previous tile have been read out of TMEM
                if (n == 0 && ti > 0 && !(ok = W.wait_warp(smem_u32(&sh->acc_free), (ti - 1) & 1))) break;
                tc_fence_after();
                M::cols(tDV, tS, stage(g) + C::kTileBytes, n > 0, leader);   // dV += P^T dO
                if (n + 1 < tl.n_items) {
                    if (!(ok = ring_full(g + 1))) break;
                    tc_fence_after();
                    M::rows(tS, sK, stage(g + 1), leader);
                    if (leader) mma_commit(smem_u32(&sh->s_full[0]));
                }
                if (!(ok = W.wait_warp(smem_u32(&sh->ds_full[0]), g & 1))) break;
                tc_fence_after();
                M::cols(tDK, tDP, stage(g), n > 0, leader);                  // dK += dS^T Q
                if (leader) mma_commit(smem_u32(&sh->ring_empty[g % C::kStages]));
                if (n + 1 < tl.n_items) {
                    M::rows(tDP, sV, stage(g + 1) + C::kTileBytes, leader);
                    if (leader) mma_commit(smem_u32(&sh->dp_full[0]));
                }
            }
            if (!ok) break;
            // every product of the tile is issued: K and V go back to the
            // loader, dV and dK to the epilogue, once they complete
            if (leader) mma_commit(smem_u32(&sh->kv_free));
            if (leader) mma_commit(smem_u32(&sh->acc_done));
            ++ti;
        }
        if (leader) mma_commit(smem_u32(&sh->drain));
        W.drain(smem_u32(&sh->drain), 0);
    } else if (warp >= kWarpEw0) {
        // ------------------------------------------------- P, dS, epilogue
        const int wq = (warp - kWarpEw0) & 3;   // TMEM lane quarter
        const int hf = (warp - kWarpEw0) >> 2;  // query-column part of the tile
        const int c = wq * 32 + lane;           // key row within the tile
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + hf * kColsPerPart;
        const uint32_t tDP = tmem + lane_base + C::kColDP + hf * kColsPerPart;
        const float c2 = p.scale_log2;
        bool ok = true;
        int g = 0;
        int ti = 0;
        for (int t = 0; t < n_mine && ok; ++t) {
            const Tile tl = tile(t);
            const int j = tl.j;
            const int kc = j * kTileN + c;
            for (int n = 0; n < tl.n_items && ok; ++n, ++g) {
                const int i = tl.ilo + n % tl.ni;
                const uint8_t* stage = smem + 2 * C::kTileBytes + (g % C::kStages) * C::kStageKV;
                const float4* lse2 =
                    reinterpret_cast<const float4*>(stage + 2 * C::kTileBytes) + hf * (kColsPerPart / 4);
                const float4* dsum =
                    reinterpret_cast<const float4*>(stage + 2 * C::kTileBytes + C::kVecBytes) + hf * (kColsPerPart / 4);
                if (!(ok = W.wait_warp(smem_u32(&sh->ring_full[g % C::kStages]), (g / C::kStages) & 1))) break;
                if (!(ok = W.wait_warp(smem_u32(&sh->s_full[0]), g & 1))) break;
                tc_fence_after();
                uint32_t s[kChunks][32];
                ld_part(tS, s);
                const bool masked = kMask && tile_needs_mask(p.g, i * kTileM, j);  // uniform over the CTA
                int r_lo = 0, r_hi = kTileM - 1;
                if (masked) key_visible_rows(p.g, kc, i, r_lo, r_hi);
                // P^T: p = 2^(s * scale * log2 e - LSE_q * log2 e), 0 where masked
                auto pt = [&](auto kM) {
                    constexpr bool M = decltype(kM)::value;
#pragma unroll
                    for (int cc = 0; cc < kChunks; ++cc) {
                        uint32_t pk[16];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const float4 l4 = lds_f4(lse2 + cc * 8 + v);
                            float e0, e1, e2, e3;
                            ffma2(e0, e1, u2f(s[cc][4 * v]), u2f(s[cc][4 * v + 1]), c2, c2, -l4.x, -l4.y);
                            ffma2(e2, e3, u2f(s[cc][4 * v + 2]), u2f(s[cc][4 * v + 3]), c2, c2, -l4.z, -l4.w);
                            e0 = ex2(e0);
                            e1 = ex2(e1);
                            e2 = ex2(e2);
                            e3 = ex2(e3);
                            if (M) {
                                const int q = hf * kColsPerPart + cc * 32 + 4 * v;
                                if (q < r_lo || q > r_hi) e0 = 0.f;
                                if (q + 1 < r_lo || q + 1 > r_hi) e1 = 0.f;
                                if (q + 2 < r_lo || q + 2 > r_hi) e2 = 0.f;
                                if (q + 3 < r_lo || q + 3 > r_hi) e3 = 0.f;
                            }
                            s[cc][4 * v] = f2u(e0);
                            s[cc][4 * v + 1] = f2u(e1);
                            s[cc][4 * v + 2] = f2u(e2);
                            s[cc][4 * v + 3] = f2u(e3);
                            pk[2 * v] = pack2<kBf16>(e0, e1);
                            pk[2 * v + 1] = pack2<kBf16>(e2, e3);
                        }
                        tmem_st16(tS + 16 * cc, pk);
                    }
                };
                // Two copies of the loop, one without the per-element test: a tile
                // needs the mask only on the diagonal or a band's edge, and the test
                // kept in the common copy cost the causal backward 12%.
                if (masked) pt(std::true_type{}); else pt(std::false_type{});
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&sh->p_full[0]));
                // dS^T: p * (dP - Dsum_q), written over dP columns of this half already read
                if (!(ok = W.wait_warp(smem_u32(&sh->dp_full[0]), g & 1))) break;
                tc_fence_after();
                uint32_t d[kChunks][32];
                ld_part(tDP, d);
#pragma unroll
                for (int cc = 0; cc < kChunks; ++cc) {
                    uint32_t pk[16];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float4 d4 = lds_f4(dsum + cc * 8 + v);
                        float g0, g1, g2, g3;
                        fadd2(g0, g1, u2f(d[cc][4 * v]), u2f(d[cc][4 * v + 1]), -d4.x, -d4.y);
                        fadd2(g2, g3, u2f(d[cc][4 * v + 2]), u2f(d[cc][4 * v + 3]), -d4.z, -d4.w);
                        fmul2(g0, g1, g0, g1, u2f(s[cc][4 * v]), u2f(s[cc][4 * v + 1]));
                        fmul2(g2, g3, g2, g3, u2f(s[cc][4 * v + 2]), u2f(s[cc][4 * v + 3]));
                        pk[2 * v] = pack2<kBf16>(g0, g1);
                        pk[2 * v + 1] = pack2<kBf16>(g2, g3);
                    }
                    tmem_st16(tDP + 16 * cc, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&sh->ds_full[0]));
            }
            // epilogue: this part's columns of dV and scale * dK for the keys that exist
            const bool live = kc < p.g.N;
            const size_t row = (size_t)row_index(p.layout, tl.b, tl.hk, live ? kc : 0, p.Hkv, p.g.N);
            if (tl.n_items == 0) {
                if (live) {
                    zero_row<D>(p.dv, row, hf);
                    zero_row<D>(p.dk, row, hf);
                }
            } else if (ok && (ok = W.wait_warp(smem_u32(&sh->acc_done), ti & 1))) {
                tc_fence_after();
                store_row<D, kBf16>(tmem + lane_base + C::kColA, p.dv, row, hf, 1.f, live);
                store_row<D, kBf16>(tmem + lane_base + C::kColB, p.dk, row, hf, p.scale, live);
                // the accumulators may now take the next tile's products
                tc_fence_before();
                mbar_arrive(smem_u32(&sh->acc_free));
                ++ti;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMmaB) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ========================================================================= dQ
template <int D, bool kBf16, bool kMask>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    using M = Mma<D, kBf16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sRing = smem_u32(smem);
    BwdCtl* sh = reinterpret_cast<BwdCtl*>(smem + C::kStagesQ * C::kStageQ);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);  // warp-uniform to the compiler
    const int lane = threadIdx.x & 31;

    // CTA -> (b, head, query tile i); consecutive CTAs share a head's K/V
    const int i = blockIdx.x % p.n_tiles;
    const int bh = blockIdx.x / p.n_tiles;
    const int b = bh / p.H, h = bh % p.H, hk = h / p.G;
    const int r0 = i * kTileM;
    int jlo = 0, jhi = 0;
    if (r0 < p.g.N) kv_tile_range(p.g, r0, r0 + kTileM < p.g.N ? r0 + kTileM : p.g.N, jlo, jhi);
    const int n_items = jhi - jlo;

    if (threadIdx.x == 0) init_ctl(sh, 1, kEwThreads / kParts);
    if (warp == kWarpMmaB) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, sh->tmem_base, 0);
    const Waiter W{&sh->abort, p.status, p.wait_limit_ns};

    if (warp == kWarpTmaB && lane == 0 && n_items > 0) {
        // ------------------------------------------------------------ TMA
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        bool ok = true;
        int n = 0;
        for (; n < n_items && ok; ++n) {
            const int st = n % C::kStagesQ;
            if (n >= C::kStagesQ && !(ok = W.wait(smem_u32(&sh->ring_empty[st]), ((n / C::kStagesQ) - 1) & 1))) break;
            const uint32_t full = smem_u32(&sh->ring_full[st]);
            const uint32_t stage = sRing + st * C::kStageQ;
            mbar_arrive_expect_tx(full, 2 * C::kTileBytes);
            load_tile<D>(stage, &p.tm_k, full, p.layout, b, hk, (jlo + n) * kTileN);
            load_tile<D>(stage + C::kTileBytes, &p.tm_v, full, p.layout, b, hk, (jlo + n) * kTileN);
        }
        for (int m = n - C::kStagesQ < 0 ? 0 : n - C::kStagesQ; m < n; ++m)
            W.drain(smem_u32(&sh->ring_full[m % C::kStagesQ]), (m / C::kStagesQ) & 1);
    } else if (warp == kWarpMmaB && n_items > 0) {
        // ------------------------------------------------------------ MMA
        // The whole warp follows one path; the elected lane issues.
        const bool leader = elect_one();
        const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tDQ = tmem + C::kColA;
        const uint32_t tQ = tmem + C::kColQ, tDO = tmem + C::kColDO;
        auto stage = [&](int n) { return sRing + (n % C::kStagesQ) * C::kStageQ; };
        auto ring_full = [&](int n) {
            return W.wait_warp(smem_u32(&sh->ring_full[n % C::kStagesQ]), (n / C::kStagesQ) & 1);
        };
        // S = Q K^T and dP = dO V^T with the stationary A operand read from TMEM
        // (TS products): only K and V come from shared memory, so products of
        // 64 keys keep the tensor core at full rate.  Each column part h (64
        // keys) has its own barriers: part h's next S goes out once its S has
        // been read into registers, its next dP once the dQ product has read
        // its dS, while the other part's elementwise work still runs.
        bool ok = W.wait_warp(smem_u32(&sh->qd_full), 0) && ring_full(0);
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < kParts; ++h) {
                M::rows_part_t(tS, tQ, stage(0), h, leader);                    // S = Q K^T
                if (leader) mma_commit(smem_u32(&sh->s_full[h]));
            }
#pragma unroll
            for (int h = 0; h < kParts; ++h) {
                M::rows_part_t(tDP, tDO, stage(0) + C::kTileBytes, h, leader);  // dP = dO V^T
                if (leader) mma_commit(smem_u32(&sh->dp_full[h]));
            }
        }
        for (int n = 0; n < n_items && ok; ++n) {
            const bool more = n + 1 < n_items;
            if (more) {
                if (!(ok = ring_full(n + 1))) break;
#pragma unroll
                for (int h = 0; h < kParts; ++h) {
                    // the next S may overwrite S once its row loads are done
                    if (!(ok = W.wait_warp(smem_u32(&sh->s_free[h]), n & 1))) break;
                    tc_fence_after();
                    M::rows_part_t(tS, tQ, stage(n + 1), h, leader);
                    if (leader) mma_commit(smem_u32(&sh->s_full[h]));
                }
                if (!ok) break;
            }
#pragma unroll
            for (int h = 0; h < kParts; ++h) {
                if (!(ok = W.wait_warp(smem_u32(&sh->ds_full[h]), n & 1))) break;
                tc_fence_after();
                M::cols_part(tDQ, tDP, stage(n), h, n > 0 || h > 0, leader);     // dQ += dS K
                if (h == kParts - 1 && leader) mma_commit(smem_u32(&sh->ring_empty[n % C::kStagesQ]));
                if (more) {
                    M::rows_part_t(tDP, tDO, stage(n + 1) + C::kTileBytes, h, leader);
                    if (leader) mma_commit(smem_u32(&sh->dp_full[h]));
                }
            }
        }
        if (leader) mma_commit(smem_u32(&sh->acc_done));
        if (leader) mma_commit(smem_u32(&sh->drain));
        W.drain(smem_u32(&sh->drain), 0);
    } else if (warp >= kWarpEw0) {
        // ------------------------------------------------------- dS, epilogue
        const int wq = (warp - kWarpEw0) & 3;   // TMEM lane quarter
        const int hf = (warp - kWarpEw0) >> 2;  // key-column part of the tile
        const int row = wq * 32 + lane;
        const int qi = r0 + row;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + hf * kColsPerPart;
        const uint32_t tDP = tmem + lane_base + C::kColDP + hf * kColsPerPart;
        const size_t vrow = (size_t)bh * p.Npad + qi;
        const float lse2 = p.lse2[vrow];
        const float dsum = p.dsum[vrow];
        const float c2 = p.scale_log2;
        bool ok = true;
        if (n_items > 0) {
            // This thread's row of Q and of dO, its half of the columns, into TMEM as
            // 16-bit pairs (column c holds elements 2c and 2c + 1): the A operands of
            // S = Q K^T and dP = dO V^T.  Rows past N are zeros.
            const bool live_q = qi < p.g.N;
            const size_t qrow = (size_t)row_index(p.layout, b, h, live_q ? qi : 0, p.H, p.g.N);
            constexpr int kWords = D / 4;  // 32-bit words in half a row
            const uint16_t* srcs[2] = {static_cast<const uint16_t*>(p.q), static_cast<const uint16_t*>(p.d_o)};
            const uint32_t dsts[2] = {tmem + lane_base + C::kColQ + hf * kWords,
                                      tmem + lane_base + C::kColDO + hf * kWords};
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const uint4* src = reinterpret_cast<const uint4*>(srcs[x] + qrow * D + hf * (D / 2));
#pragma unroll
                for (int c = 0; c < kWords / 16; ++c) {
                    uint32_t w[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 u = live_q ? src[c * 4 + v] : make_uint4(0, 0, 0, 0);
                        w[4 * v] = u.x;
                        w[4 * v + 1] = u.y;
                        w[4 * v + 2] = u.z;
                        w[4 * v + 3] = u.w;
                    }
                    tmem_st16(dsts[x] + 16 * c, w);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&sh->qd_full));
        }
        for (int n = 0; n < n_items && ok; ++n) {
            const int j = jlo + n;
            if (!(ok = W.wait_warp(smem_u32(&sh->s_full[hf]), n & 1))) break;
            tc_fence_after();
            uint32_t s[kChunks][32];
            ld_part(tS, s);
            tc_fence_before();
            mbar_arrive(smem_u32(&sh->s_free[hf]));
            const bool masked = kMask && tile_needs_mask(p.g, r0, j);  // uniform over the CTA
            int c_lo = 0, c_hi = kTileN - 1;
            if (masked) row_visible_cols(p.g, qi, j, c_lo, c_hi);
            auto pe = [&](auto kM) {
                constexpr bool M = decltype(kM)::value;
#pragma unroll
                for (int cc = 0; cc < kChunks; ++cc)
#pragma unroll
                    for (int v = 0; v < 32; v += 2) {
                        float e0, e1;
                        ffma2(e0, e1, u2f(s[cc][v]), u2f(s[cc][v + 1]), c2, c2, -lse2, -lse2);
                        e0 = ex2(e0);
                        e1 = ex2(e1);
                        if (M) {
                            const int col = hf * kColsPerPart + cc * 32 + v;
                            if (col < c_lo || col > c_hi) e0 = 0.f;
                            if (col + 1 < c_lo || col + 1 > c_hi) e1 = 0.f;
                        }
                        s[cc][v] = f2u(e0);
                        s[cc][v + 1] = f2u(e1);
                    }
            };
            if (masked) pe(std::true_type{}); else pe(std::false_type{});  // as in the dK/dV kernel
            if (!(ok = W.wait_warp(smem_u32(&sh->dp_full[hf]), n & 1))) break;
            tc_fence_after();
            uint32_t d[kChunks][32];
            ld_part(tDP, d);
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    float g0, g1;
                    fadd2(g0, g1, u2f(d[cc][2 * v]), u2f(d[cc][2 * v + 1]), -dsum, -dsum);
                    fmul2(g0, g1, g0, g1, u2f(s[cc][2 * v]), u2f(s[cc][2 * v + 1]));
                    pk[v] = pack2<kBf16>(g0, g1);
                }
                tmem_st16(tDP + 16 * cc, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&sh->ds_full[hf]));
        }
        const bool live = qi < p.g.N;
        const size_t orow = (size_t)row_index(p.layout, b, h, live ? qi : 0, p.H, p.g.N);
        if (n_items == 0) {
            if (live) zero_row<D>(p.dq, orow, hf);
        } else if (ok && W.wait_warp(smem_u32(&sh->acc_done), 0)) {
            tc_fence_after();
            store_row<D, kBf16>(tmem + lane_base + C::kColA, p.dq, orow, hf, p.scale, live);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMmaB) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ===================================================================== pre
// Dsum = rowsum(dO * O) and LSE * log2(e) per row; D/8 lanes take a row,
// 16 bytes of O and of dO each, so a warp covers 32/(D/8) whole rows per
// pass.  Rows past N (up to the padded length) are filled so they contribute
// nothing.
template <bool kBf16, int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint16_t* o, const uint16_t* d_o, const float* lse,
                                                         float* lse2, float* dsum, int B, int H, int N, int Npad,
                                                         int layout) {
    constexpr int kLanes = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanes;
    const long long rows = (long long)B * H * Npad;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanes;
    const int l = lane % kLanes;
    const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRowsPerWarp; r0 < rows;
         r0 += warps * kRowsPerWarp) {
        const long long r = r0 + sub;
        float acc = 0.f;
        float l2 = INFINITY;
        int i = 0;
        long long bh = 0;
        if (r < rows) {
            i = (int)(r % Npad);
            bh = r / Npad;
            if (i < N) {
                const size_t base = (size_t)row_index(layout, (int)(bh / H), (int)(bh % H), i, H, N) * D + 8 * l;
                const uint4 a = *reinterpret_cast<const uint4*>(o + base);
                const uint4 g = *reinterpret_cast<const uint4*>(d_o + base);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    acc = fmaf(lo_half<kBf16>(aw[m]), lo_half<kBf16>(gw[m]), acc);
                    acc = fmaf(hi_half<kBf16>(aw[m]), hi_half<kBf16>(gw[m]), acc);
                }
                const float lv = lse[bh * N + i];
                l2 = lv == -INFINITY ? INFINITY : lv * kLog2e;
            }
        }
#pragma unroll
        for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (l == 0 && r < rows) {
            lse2[bh * Npad + i] = l2;
            dsum[bh * Npad + i] = acc;
        }
    }
}

template <bool kBf16, int D>
void launch_pre_typed(const void* o, const void* d_o, const float* lse, float* lse2, float* dsum, int B, int H, int N,
                      int Npad, int layout, int sms, cudaStream_t s) {
    constexpr int kRowsPerBlock = 8 * (32 / (D / 8));
    const long long rows = (long long)B * H * Npad;
    long long grid = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (grid > 32LL * sms) grid = 32LL * sms;
    fa_bwd_pre_kernel<kBf16, D><<<(int)grid, 256, 0, s>>>(static_cast<const uint16_t*>(o),
                                                          static_cast<const uint16_t*>(d_o), lse, lse2, dsum, B, H,
                                                          N, Npad, layout);
}

// Key tiles per dK/dV CTA for a problem without masks (each key tile then has
// `items` query tiles): the count k that minimises (waves of CTAs) x (k + a),
// one CTA per SM, where a = 4.8 / items is a CTA's fixed cost (set-up and
// last epilogue) in units of one key tile's work, measured at about 0.15 for
// 32 query tiles.  At B = 4, H = 32, N = 4096 on 152 SMs this picks 3 (4,096
// key tiles in 1,366 CTAs, 8.98 waves); measured, 1 to 4 tiles per CTA took
// 2.66, 2.60, 2.54 and 2.58 ms a backward call.
int dkdv_tiles_per_cta(long long n_work, int items) {
    constexpr int kMaxDev = 64;
    static std::atomic<int> sm_count[kMaxDev];
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
    sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 1;
        sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    const double a = 4.8 / (items > 0 ? items : 1);
    int best = 1;
    double best_cost = 0.0;
    for (int k = 1; k <= kDkdvMaxTiles; ++k) {
        const long long ctas = (n_work + k - 1) / k;
        const double cost = (double)((ctas + sms - 1) / sms) * (k + a);
        if (k == 1 || cost < best_cost) {
            best = k;
            best_cost = cost;
        }
    }
    return best;
}

// kMask = false builds both kernels without the element-mask code, for
// problems where no tile needs it (geom_needs_masks); as in the forward, the
// smaller code runs measurably faster.
template <int D, bool kBf16, bool kMask>
cudaError_t launch_bwd_typed(const BwdParams& p, int B, cudaStream_t s) {
    auto kdkdv = fa_bwd_dkdv_kernel<D, kBf16, kMask>;
    auto kdq = fa_bwd_dq_kernel<D, kBf16, kMask>;
    constexpr int sm1 = dkdv_smem_bytes<D>();
    constexpr int sm2 = dq_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(kdkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, sm1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, sm2);
    if (e != cudaSuccess) return e;
    const long long n_work = (long long)B * p.Hkv * p.n_tiles;  // key tiles
    const int per_cta = kMask ? 1 : dkdv_tiles_per_cta(n_work, p.n_tiles * p.G);
    if (n_work > 0x7fffffffLL - per_cta) return cudaErrorInvalidValue;
    kdkdv<<<(unsigned)((n_work + per_cta - 1) / per_cta), kBwdThreads, sm1, s>>>(p, (int)n_work, per_cta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kdq<<<B * p.H * p.n_tiles, kBwdThreads, sm2, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const void* o, const void* d_o, const float* lse, float* lse2, float* dsum, int B, int H,
                           int N, int Npad, int D, int layout, int dtype_code, int sms, cudaStream_t s) {
    const bool bf16 = dtype_code == 1;
    if (D == 64) {
        if (bf16)
            launch_pre_typed<true, 64>(o, d_o, lse, lse2, dsum, B, H, N, Npad, layout, sms, s);
        else
            launch_pre_typed<false, 64>(o, d_o, lse, lse2, dsum, B, H, N, Npad, layout, sms, s);
    } else {
        if (bf16)
            launch_pre_typed<true, 128>(o, d_o, lse, lse2, dsum, B, H, N, Npad, layout, sms, s);
        else
            launch_pre_typed<false, 128>(o, d_o, lse, lse2, dsum, B, H, N, Npad, layout, sms, s);
    }
    return cudaGetLastError();
}

template <int D, bool kBf16>
cudaError_t launch_bwd_masks(const BwdParams& p, int B, cudaStream_t s) {
    return geom_needs_masks(p.g) ? launch_bwd_typed<D, kBf16, true>(p, B, s) : launch_bwd_typed<D, kBf16, false>(p, B, s);
}

cudaError_t launch_bwd(const BwdParams& p, int B, int D, bool bf16, cudaStream_t s) {
    if (D == 64) return bf16 ? launch_bwd_masks<64, true>(p, B, s) : launch_bwd_masks<64, false>(p, B, s);
    return bf16 ? launch_bwd_masks<128, true>(p, B, s) : launch_bwd_masks<128, false>(p, B, s);
}

}  // namespace fa
