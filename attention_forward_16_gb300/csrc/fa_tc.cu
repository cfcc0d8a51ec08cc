// Tensor-core fused attention forward for sm_103a (fp16 / bf16 in, fp32 accumulate).
//
// The method is the tiled, online-softmax attention forward of
// "Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention" (section 1.2: running row max m and row sum l,
// one division at the end; section 3: Q row blocks outer, K/V blocks inner,
// scores kept on chip) and of the ops-transformer walk-through (section
// "online softmax: incremental update").  The Cube/Vector pipelining of
// "FlashAttention extreme optimisation on Ascend NPUs" (optimisation three:
// matrix unit on block i while the vector unit does the softmax of block
// i-1) and the double-buffered loads of its optimisation two become, on
// Blackwell, warp specialisation around tcgen05 + TMEM + TMA:
//
//   warps 0-3   Q tile 0: softmax (thread = one query row), then its epilogue
//   warps 4-7   Q tile 1: same
//   warp  8     TMEM allocator; issues Q tile 0's tcgen05.mma (one elected lane)
//   warp  9     one thread issues the TMA loads of the K/V ring
//   warp  10    issues Q tile 1's tcgen05.mma (one elected lane)
//   warp  11    one thread issues the TMA loads of the two Q tiles
//
// The launch gives 168 registers a thread (12 warps, three per SM
// sub-partition); setmaxnreg then moves 48 from the MMA/TMA warpgroup to the
// softmax warpgroups, for their 64 scores a row plus the epilogue's O chunk
// (192 + 192 + 120 = 3 x 168).
//
// TMEM (512 columns x 128 lanes x 32 bit): S0 | S1 | O0 | O1.  Each S holds
// a 128-key tile as two 64-key halves with their own barriers, and the
// softmax takes each half as an online-softmax step of its own.  P (16-bit)
// overwrites the first half of its S half's columns and feeds the P.V MMA
// straight from TMEM.  Splitting S in two gives every Q tile a second S
// buffer inside the same 512 columns: while a softmax warpgroup turns one
// half into P, the tensor core computes the other half's S or the other Q
// tile's products, so the softmax never waits for its own tile's MMAs.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records a
// timeout in the device status word, lets its in-flight copies and MMAs
// finish, frees TMEM and returns.
#include <cmath>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"
#include "rope_math.cuh"
#include "tc_common.cuh"
#include "tc_softmax.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
// Registers a thread at launch: the 65536-entry file over 384 threads,
// rounded down to the allocation granule of 8 (ptxas reports this count).
constexpr int kLaunchRegs = (65536 / kThreads) & ~7;  // 168
constexpr int kRegSoftmax = 192;  // per thread, warpgroups 0-1
constexpr int kRegOther = 120;    // per thread, warpgroup 2 (MMA, TMA, idle)
// setmaxnreg.inc only draws on the registers the CTA was launched with; a
// split above that total would wait forever.
static_assert(2 * kRegSoftmax + kRegOther <= 3 * kLaunchRegs, "register split exceeds the launch budget");
constexpr int kWarpMma = 8;    // MMA issuer for Q tile 0; TMEM owner
constexpr int kWarpTma = 9;
constexpr int kWarpMma1 = 10;  // MMA issuer for Q tile 1
constexpr int kWarpTmaQ = 11;  // Q tile loads

template <int D>
struct TcCfg {
    static constexpr int kChunks = D / 64;                // 128-byte column chunks per row
    static constexpr int kBoxBytes = kTileM * 64 * 2;     // one TMA box: 128 rows x 64 elements
    static constexpr int kTileBytes = kChunks * kBoxBytes;
    static constexpr int kStages = D == 128 ? 4 : 8;      // K/V ring slots
    static constexpr int kColS0 = 0;
    static constexpr int kColS1 = 128;
    static constexpr int kColO0 = 256;
    static constexpr int kColO1 = 256 + D;
    static constexpr int kTmemCols = 512;
    // Q tiles, the K/V ring, and one 64-column O staging box per Q tile for
    // the epilogue's TMA stores.
    static constexpr int kTileSmem = (2 + kStages) * kTileBytes + 2 * kBoxBytes;
};

constexpr int kUnitRing = 4;  // unit indices handed from the scheduler to the other roles
constexpr int kUnitReaders = 1 + 32 + 32 + 128 + 128;  // K/V thread, two MMA warps, two softmax warpgroups

struct __align__(16) SharedCtl {
    uint4 clc_resp;                  // cluster launch control answer (16-byte aligned)
    int unit_ring[kUnitRing];
    uint64_t u_full[kUnitRing], u_empty[kUnitRing];
    uint64_t clc_bar;
    uint64_t q_full[2], q_empty[2];  // per Q tile
    uint64_t q_ready[2];             // per Q tile: rotated in place (rotary embedding of Q)
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2][2], p_full[2][2];  // per Q tile and S half
    uint64_t pv_done[2][2];               // per Q tile: P.V products completed, by step parity
    uint64_t o_done[2], o_free[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort;
};

template <int D>
constexpr int smem_bytes() {
    return TcCfg<D>::kTileSmem + (int)sizeof(SharedCtl) + 1024;
}

static_assert(smem_bytes<128>() <= 227 * 1024, "shared memory budget (D=128)");
// The MMA issuers wait for K(j+1) before P(j); that is deadlock-free only while
// K(j+1)'s ring slot was last used by K(j-1) or earlier (at least two key steps
// of K/V in the ring), whose S products both tiles issued a step before.
static_assert(TcCfg<128>::kStages >= 4 && TcCfg<64>::kStages >= 4, "K/V ring too short for the issue order");
static_assert(smem_bytes<64>() <= 227 * 1024, "shared memory budget (D=64)");

// ------------------------------------------------------------ TMA producers
// One whole tile (128 rows x D, all column chunks) in one TMA instruction:
// the 5-D map's coordinates are (column, row, chunk, head, batch) in either
// layout.
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int row, int head,
                                          int b) {
    tma_load_5d(dst, tm, bar, 0, row, 0, head, b);
}

// Units are handed out dynamically.  The grid has one CTA per unit, and one
// CTA fits an SM, so 152 run at a time.  A running CTA first takes its own
// unit, then takes each further unit from a CTA of the grid that has not
// started yet: it cancels that CTA's launch with cluster launch control, and
// the cancelled CTA never runs.  CTAs start in index order and units are
// numbered longest first, so faster SMs take more units and every CTA ends
// close to the others (the static round-robin of units left SMs that ran
// slower 10% behind).  The Q thread is the scheduler: it publishes each unit
// index (then -1) into a small ring that every other role reads in order,
// and requests the next index while it loads the current unit's Q.
//
// Q tiles: one thread, one buffer per tile.  Tile t of the next unit is loaded
// as soon as tile t's last S of the current unit has completed, so a tile that
// finishes its key range first (tile 0 under causal and window masks) can
// start its next unit while the other tile finishes this one.  K/V loads have
// their own thread and never wait behind a Q buffer.
template <int D>
__device__ __forceinline__ void tma_q_role(const TcParams& p, const Waiter& W, SharedCtl* sh, uint32_t sQa) {
    using C = TcCfg<D>;
    tma_prefetch_desc(&p.tm_q);
    uint32_t q_it[2] = {0, 0};
    const uint32_t clc_bar = smem_u32(&sh->clc_bar);
    const uint32_t resp = smem_u32(&sh->clc_resp);
    uint32_t asked = 0;  // cancel requests issued (each completes one phase of clc_bar)
    bool ok = true;
    int u = blockIdx.x;
    for (uint32_t k = 0; ok; ++k) {
        const uint32_t slot = k % kUnitRing;
        if (k >= (uint32_t)kUnitRing && !(ok = W.wait(smem_u32(&sh->u_empty[slot]), (k / kUnitRing - 1) & 1)))
            break;
        sh->unit_ring[slot] = u;
        mbar_arrive(smem_u32(&sh->u_full[slot]));
        if (u < 0) break;
        // the next unit, asked for now so that the answer is back by the time
        // this unit's Q is on its way
        mbar_arrive_expect_tx(clc_bar, 16);
        clc_try_cancel(resp, clc_bar);
        ++asked;
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int b = un.bh / p.H, h = un.bh % p.H;
        for (int t = 0; t < 2 && ok; ++t) {
            const uint32_t q_full = smem_u32(&sh->q_full[t]);
            if (q_it[t] > 0 && !(ok = W.wait(smem_u32(&sh->q_empty[t]), (q_it[t] - 1) & 1))) break;
            mbar_arrive_expect_tx(q_full, C::kTileBytes);
            load_tile(sQa + t * C::kTileBytes, &p.tm_q, q_full, un.q0 + t * kTileM, h, b);
            ++q_it[t];
        }
        if (!ok || !(ok = W.wait(clc_bar, (asked - 1) & 1))) break;
        u = clc_query(resp);
        // Pull the next unit's Q tiles into L2 now: their loads wait for this
        // unit's last S products, and would otherwise start with a DRAM latency.
        if (u >= 0) {
            const Unit nx = make_unit(p.g, p.BH, p.order, u);
            const int nb = nx.bh / p.H, nh = nx.bh % p.H;
            for (int t = 0; t < 2; ++t) tma_prefetch_l2_5d(&p.tm_q, 0, nx.q0 + t * kTileM, 0, nh, nb);
        }
    }
    // Let every issued copy (and an answer still on its way) land before
    // shared memory is released (on the normal path too: after an abort
    // elsewhere nobody may wait for them).
    for (int t = 0; t < 2; ++t)
        if (q_it[t] > 0) W.drain(smem_u32(&sh->q_full[t]), (q_it[t] - 1) & 1);
    if (asked > 0) W.drain(clc_bar, (asked - 1) & 1);
}

// The next unit index for a role other than the scheduler (-1: no more), read
// from ring position k; every reading thread then frees its slot.  Warp-
// uniform when kWarp (every lane waits and reads).
template <bool kWarp>
__device__ __forceinline__ int next_unit(SharedCtl* sh, const Waiter& W, uint32_t k, bool& ok) {
    const uint32_t slot = k % kUnitRing;
    const uint32_t full = smem_u32(&sh->u_full[slot]);
    ok = kWarp ? W.wait_warp(full, (k / kUnitRing) & 1) : W.wait(full, (k / kUnitRing) & 1);
    if (!ok) return -1;
    const int u = *reinterpret_cast<volatile int*>(&sh->unit_ring[slot]);
    mbar_arrive(smem_u32(&sh->u_empty[slot]));
    return u;
}

// K/V tiles: one thread filling the ring, K_j then V_j for every key tile in
// the union of the unit's two ranges.
template <int D>
__device__ __forceinline__ void tma_kv_role(const TcParams& p, const Waiter& W, SharedCtl* sh, uint32_t sKVa) {
    using C = TcCfg<D>;
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    uint32_t kv_it = 0;
    bool ok = true;
    for (uint32_t r = 0; ok; ++r) {
        const int u = next_unit<false>(sh, W, r, ok);
        if (u < 0) break;
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int b = un.bh / p.H, h = un.bh % p.H, hk = h / p.G;
        for (int j = un.jlo; j < un.jhi && ok; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
                const int slot = kv_it % C::kStages;
                if (kv_it >= (uint32_t)C::kStages &&
                    !(ok = W.wait(smem_u32(&sh->kv_empty[slot]), ((kv_it / C::kStages) - 1) & 1)))
                    break;
                const uint32_t full = smem_u32(&sh->kv_full[slot]);
                mbar_arrive_expect_tx(full, C::kTileBytes);
                const CUtensorMap* tm = kv ? &p.tm_v : &p.tm_k;
                load_tile(sKVa + slot * C::kTileBytes, tm, full, j * kTileN, hk, b);
                ++kv_it;
            }
        }
    }
    // Let every issued copy land before shared memory is released.
    for (uint32_t s = 0; s < (uint32_t)C::kStages && s < kv_it; ++s) {
        const uint32_t last = kv_it - 1 - ((kv_it - 1 - s) % C::kStages);
        W.drain(smem_u32(&sh->kv_full[s]), (last / C::kStages) & 1);
    }
}

// -------------------------------------------------------------- MMA issuers
// One issuing warp per Q tile t.  Each 128-key tile j is taken in two halves
// of 64 keys, each with its own S columns: S_t,h(j) = Q_t K_j[64h, 64h+64)^T
// and O_t += P_t,h(j) V_j[64h, 64h+64).  P_t,h overwrites S_t,h, so the next
// S_t,h waits for the P.V that reads it, but the other half's S is already
// computed: the softmax of one half runs while the tensor core works on the
// other half (of this tile or of the other Q tile), and no step of the softmax
// waits for its own tile's MMAs.  Issue order per tile (S(lo) is one N = 128
// product that fills both halves):
//   S(lo) | PV(j,0) S(j+1,0) PV(j,1) S(j+1,1) | ...
// A K/V ring slot is released once both warps have arrived (count 2); a tile
// with no work on key tile j still waits for that slot to be full before
// arriving, which keeps the phases of the ring aligned.  Each Q tile's buffer
// is released by its own warp once its last S has completed.
//
// The whole warp runs this role on one path: every wait, counter and shared-
// memory descriptor is warp-uniform, and one elected lane issues the
// tcgen05.mma / commit instructions and the single mbarrier arrivals.  Issue
// from a lone lane of a diverged warp ran at about 100 cycles per MMA, slower
// than the tensor core's 64 cycles for a 128x128x16 product; from a converged
// warp the tensor core stays fed.  Descriptors are formed once and advanced
// by adding encoded offsets (the start address field holds address / 16, and
// every shared address here stays below 256 KiB, so the add never carries out
// of the field).
template <int D, bool kBf16, bool kMask>
__device__ __forceinline__ void mma_role(const TcParams& p, const Waiter& W, SharedCtl* sh, uint32_t sQa,
                                         uint32_t sKVa, uint32_t tmem, int t) {
    using C = TcCfg<D>;
    constexpr int kHalf = kTileN / 2;
    constexpr uint32_t idesc_s = make_idesc(kBf16, kTileM, kHalf, false);
    constexpr uint32_t idesc_o = make_idesc(kBf16, kTileM, D, true);
    const uint32_t dS = tmem + (t ? C::kColS1 : C::kColS0);
    const uint32_t dO = tmem + (t ? C::kColO1 : C::kColO0);
    const uint32_t qa = sQa + t * C::kTileBytes;
    const uint32_t o_done = smem_u32(&sh->o_done[t]);
    const uint32_t o_free = smem_u32(&sh->o_free[t]);
    // With the rotary embedding of Q the tile is released to this warp by its
    // softmax warpgroup once rotated; otherwise as soon as its copy lands.
    const uint32_t q_full = smem_u32(p.rope ? &sh->q_ready[t] : &sh->q_full[t]);
    const uint32_t q_empty = smem_u32(&sh->q_empty[t]);
    const bool leader = elect_one();
    uint32_t kv_it = 0, q_it = 0, o_cnt = 0, pv_it = 0;
    uint32_t p_cnt[2] = {0, 0};
    bool ok = true;

    // S = Q K^T: K = D in steps of 16 (32 bytes inside a 128-byte swizzled row);
    // half h starts 64 key rows (8 swizzle atoms) into each column chunk of K.
    const uint64_t q_desc = make_sdesc(qa, 16, 1024);
    const uint64_t k_desc = make_sdesc(sKVa, 16, 1024);
    const uint64_t v_desc = make_sdesc(sKVa, C::kBoxBytes, 1024);
    // A unit's first S has no P.V to interleave with: one N = 128 product
    // serves both halves, reading Q from shared memory once instead of twice
    // at the point where the unit's loads and the previous epilogue also use
    // shared memory.
    constexpr uint32_t idesc_s2 = make_idesc(kBf16, kTileM, kTileN, false);
    auto issue_s_full = [&](uint32_t slot) {
        const uint64_t kb = k_desc + (uint64_t)(slot * (uint32_t)(C::kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;
            if (leader) mma_ss(dS, q_desc + off, kb + off, idesc_s2, kk > 0);
        }
        if (leader) {
            mma_commit(smem_u32(&sh->s_full[t][0]));
            mma_commit(smem_u32(&sh->s_full[t][1]));
        }
    };
    auto issue_s = [&](uint32_t slot, int h) {
        const uint64_t kb = k_desc + (uint64_t)(slot * (uint32_t)(C::kTileBytes >> 4) + (uint32_t)((h * kHalf * 128) >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;
            if (leader) mma_ss(dS + h * kHalf, q_desc + off, kb + off, idesc_s, kk > 0);
        }
        if (leader) mma_commit(smem_u32(&sh->s_full[t][h]));
    };
    // O += P V: P from TMEM (8 columns = 16 keys per step), V MN-major in
    // shared memory (16 keys = two 8-row swizzle atoms = 2048 bytes per step;
    // the second 64-column chunk of V sits one box further on).  With a split
    // P the low halves (32 columns further on) add a second product.  Every
    // P.V is committed to pv_done by step parity, for the rare O rescale.
    auto issue_pv = [&](uint32_t slot, int h, bool zero, bool split) {
        const uint64_t vb = v_desc + (uint64_t)(slot * (uint32_t)(C::kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk) {
            const uint64_t b = vb + (uint64_t)((h * (kHalf / 16) + kk) * (2048 >> 4));
            if (leader) mma_ts(dO, dS + h * kHalf + kk * 8, b, idesc_o, (zero && kk == 0) ? 0u : 1u);
        }
        if (split) {
#pragma unroll
            for (int kk = 0; kk < kHalf / 16; ++kk) {
                const uint64_t b = vb + (uint64_t)((h * (kHalf / 16) + kk) * (2048 >> 4));
                if (leader) mma_ts(dO, dS + h * kHalf + kHalf / 2 + kk * 8, b, idesc_o, 1u);
            }
        }
        if (leader) mma_commit(smem_u32(&sh->pv_done[t][pv_it & 1]));
        ++pv_it;
    };
    auto wait_kv = [&](uint32_t idx) {
        const bool r = W.wait_warp(smem_u32(&sh->kv_full[idx % C::kStages]), (idx / C::kStages) & 1);
        tc_fence_after();
        return r;
    };
    // Give back a slot this tile does not read.
    auto skip_kv = [&](uint32_t idx) {
        if (!wait_kv(idx)) return false;
        if (leader) mbar_arrive(smem_u32(&sh->kv_empty[idx % C::kStages]));
        return true;
    };

    for (uint32_t r = 0; ok; ++r) {
        const int u = next_unit<true>(sh, W, r, ok);
        if (u < 0) break;
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        if (!(ok = W.wait_warp(q_full, q_it & 1))) break;
        ++q_it;
        tc_fence_after();
        const uint32_t kbase = kv_it;  // ring index of K_jlo; V_j follows K_j
        kv_it += 2 * (un.jhi - un.jlo);
        const int lo = t ? un.lo[1] : un.lo[0];
        const int hi = t ? un.hi[1] : un.hi[0];
        auto kidx = [&](int j) { return kbase + 2 * (uint32_t)(j - un.jlo); };
        if (lo == hi) {
            if (leader) mbar_arrive(q_empty);
            for (int j = un.jlo; j < un.jhi && ok; ++j) ok = skip_kv(kidx(j)) && skip_kv(kidx(j) + 1);
            continue;
        }
        const bool split = kBf16 && kMask && tile_split_p(p.g, un.q0 + t * kTileM);
        for (int j = un.jlo; j < lo && ok; ++j) ok = skip_kv(kidx(j)) && skip_kv(kidx(j) + 1);
        if (!ok || !(ok = wait_kv(kidx(lo)))) break;
        issue_s_full(kidx(lo) % C::kStages);
        if (leader) mma_commit(smem_u32(&sh->kv_empty[kidx(lo) % C::kStages]));
        for (int j = lo; j < hi && ok; ++j) {
            const uint32_t v = kidx(j) + 1;
            if (j == hi - 1 && leader) mma_commit(q_empty);  // this tile's last S is issued
            // Every other condition of this step is met before P_j is waited
            // for, so the MMAs go out as soon as each half of P_j lands: V_j;
            // K_(j+1) for the S issued right after each P.V (its ring slot was
            // freed by S(j-1) of both tiles, issued at least one step earlier,
            // so it never waits on this step); and the O accumulator at a
            // unit's first step (freed by the previous epilogue, which precedes
            // this unit's first P).
            if (!(ok = wait_kv(v))) break;
            if (j + 1 < hi && !(ok = wait_kv(kidx(j + 1)))) break;
            const bool first = j == lo;
            if (first && o_cnt > 0 && !(ok = W.wait_warp(o_free, (o_cnt - 1) & 1))) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!(ok = W.wait_warp(smem_u32(&sh->p_full[t][h]), p_cnt[h] & 1))) break;
                ++p_cnt[h];
                tc_fence_after();
                issue_pv(v % C::kStages, h, first && h == 0, split);
                if (h == 1 && leader) mma_commit(smem_u32(&sh->kv_empty[v % C::kStages]));
                if (j + 1 < hi) {
                    const uint32_t k = kidx(j + 1) % C::kStages;
                    issue_s(k, h);
                    if (h == 1 && leader) mma_commit(smem_u32(&sh->kv_empty[k]));
                } else if (h == 1) {
                    if (leader) mma_commit(o_done);
                    ++o_cnt;
                }
            }
        }
        for (int j = hi; j < un.jhi && ok; ++j) ok = skip_kv(kidx(j)) && skip_kv(kidx(j) + 1);
    }
    // Every issued MMA must complete before TMEM is released.
    const uint32_t drain = smem_u32(&sh->drain[t]);
    if (leader) mma_commit(drain);
    W.drain(drain, 0);
}

// ------------------------------------------------------ softmax + epilogue
template <int D, bool kBf16, bool kPosScale, bool kMask>
__device__ __forceinline__ void softmax_role(const TcParams& p, const Waiter& W, SharedCtl* sh, uint32_t tmem,
                                             uint8_t* sQ, uint32_t sStg, int warp, int lane) {
    using C = TcCfg<D>;
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_base + (t ? C::kColO1 : C::kColO0);
    const uint32_t o_done = smem_u32(&sh->o_done[t]);
    const uint32_t o_free = smem_u32(&sh->o_free[t]);
    const float c2 = p.scale_log2;
    uint32_t sc = 0;  // key tiles whose two S halves were taken
    uint32_t u_cnt = 0, q_cnt = 0, g = 0;  // g: S halves taken so far (P.V steps)
    uint32_t e_cnt = 0;                    // O chunks staged so far
    bool ok = true;
    for (uint32_t r = 0; ok; ++r) {
        const int u = next_unit<true>(sh, W, r, ok);
        if (u < 0) break;
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int jlo_t = t ? un.lo[1] : un.lo[0];
        const int jhi_t = t ? un.hi[1] : un.hi[0];
        const int r0 = un.q0 + t * kTileM;
        const int qi = r0 + row;
        if (p.rope) {
            // Rotate this thread's row of the tile once it has landed, make the
            // stores visible to the tensor core, and release the tile (every
            // unit, so the issuer's phases stay aligned even for an empty tile).
            if (!(ok = W.wait_warp(smem_u32(&sh->q_full[t]), q_cnt & 1))) break;
            ++q_cnt;
            if (jlo_t < jhi_t && qi < p.g.N) {
                const long long pos = (long long)p.rope_pos0 + qi;
                rope_q_row<D, kBf16, C::kBoxBytes>(sQ + t * C::kTileBytes, row, p.rope_cos + pos * (D / 2),
                                                   p.rope_sin + pos * (D / 2), p.rope_style);
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&sh->q_ready[t]));
        }
        if (jlo_t == jhi_t) continue;
        const bool split = kBf16 && kMask && tile_split_p(p.g, r0);
        float m_ref = -INFINITY;
        float l = 0.f;
        for (int j = jlo_t; j < jhi_t && ok; ++j) {
            // With masks, bf16 carries the split-P path as well: with both
            // halves inlined its softmax code outgrows the instruction cache,
            // so the halves share one copy there (the other builds keep the
            // unrolled pair, which schedules better).
#pragma unroll((kBf16 && kMask) ? 1 : 2)
            for (int h = 0; h < 2; ++h) {
                if (!(ok = W.wait_warp(smem_u32(&sh->s_full[t][h]), sc & 1))) break;
                sc += (uint32_t)h;
                tc_fence_after();
                // The P.V of the previous half is the only product that can
                // still be adding into O here.
                const uint32_t gp = g - 1;
                auto wait_pv = [&]() { return W.wait_warp(smem_u32(&sh->pv_done[t][gp & 1]), (gp >> 1) & 1); };
                float lsum;
                if (!(ok = softmax_half<D, kBf16, kPosScale, kMask>(p.g, tS + h * (kTileN / 2), tO, c2, r0, qi, j, h,
                                                             j == jlo_t && h == 0, split, m_ref, l, lsum, wait_pv)))
                    break;
                mbar_arrive(smem_u32(&sh->p_full[t][h]));
                l += lsum;
                ++g;
            }
        }
        if (!ok) break;

        // Epilogue: O / l, LSE = ln 2 * (m + log2 l), once the last P.V landed.
        if (!(ok = W.wait_warp(o_done, u_cnt & 1))) break;
        ++u_cnt;
        tc_fence_after();
        const float inv = 1.f / l;
        const bool live = qi < p.g.N;
        const size_t lrow = (size_t)un.bh * p.g.N + (size_t)(live ? qi : 0);
        if (p.o_f32) {
            const size_t orow = (size_t)row_index(p.layout, un.bh / p.H, un.bh % p.H, live ? qi : 0, p.H, p.g.N);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
                if (live) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(u2f(o[4 * i]) * inv, u2f(o[4 * i + 1]) * inv, u2f(o[4 * i + 2]) * inv,
                                             u2f(o[4 * i + 3]) * inv);
                }
            }
            tc_fence_before();
            mbar_arrive(o_free);
        } else {
            // 16-bit O: each warp stages its 32 rows of a 64-column chunk in
            // its own quarter of the tile's box (128-byte swizzled rows, the
            // layout of the O tensor map) and writes them with one TMA store
            // of its own, so the write-back is whole-box copies rather than
            // 16-byte stores that touch a cache line per row, and no warp
            // waits for another.  Lane 0 waits for its store to have read the
            // quarter only when the quarter is wanted again.  The O columns
            // are released to the next unit's P.V as soon as the last chunk
            // has been read out of tensor memory.
            const uint32_t stg = sStg + t * C::kBoxBytes + wq * (C::kBoxBytes / 4);
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t oa[32], ob[32];
                tmem_ld32(tO + c * 64, oa);
                tmem_ld32(tO + c * 64 + 32, ob);
                tmem_wait_ld();
                if (c == D / 64 - 1) {
                    tc_fence_before();
                    mbar_arrive(o_free);
                }
                if (e_cnt > 0) {
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                }
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) {
                    const uint32_t* w = uu < 4 ? oa + 8 * uu : ob + 8 * (uu - 4);
                    const uint4 v = make_uint4(pack2<kBf16>(u2f(w[0]) * inv, u2f(w[1]) * inv),
                                               pack2<kBf16>(u2f(w[2]) * inv, u2f(w[3]) * inv),
                                               pack2<kBf16>(u2f(w[4]) * inv, u2f(w[5]) * inv),
                                               pack2<kBf16>(u2f(w[6]) * inv, u2f(w[7]) * inv));
                    st_shared_v4(stg + lane * 128 + (((uint32_t)uu ^ (uint32_t)(lane & 7)) << 4), v);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_5d(&p.tm_o, stg, 0, r0 + wq * 32, c, un.bh % p.H, un.bh / p.H);
                    bulk_commit_group();
                }
                ++e_cnt;
            }
            if (!ok) break;
        }
        if (live && p.lse) p.lse[lrow] = (m_ref + log2f(l)) * kLn2;
    }
    // Every TMA store of O has finished before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_group<0>();
}

template <int D, bool kBf16, bool kPosScale, bool kMask>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_tc_kernel(const __grid_constant__ TcParams p) {
    using C = TcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SharedCtl* sh = reinterpret_cast<SharedCtl*>(smem + C::kTileSmem);
    const uint32_t sQa = smem_u32(smem);
    const uint32_t sKVa = sQa + 2 * C::kTileBytes;

    // Warp index through a shuffle, so the compiler sees it as warp-uniform.
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&sh->q_full[t]), 1);
            mbar_init(smem_u32(&sh->q_empty[t]), 1);
            mbar_init(smem_u32(&sh->q_ready[t]), 128);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&sh->kv_full[s]), 1);
            mbar_init(smem_u32(&sh->kv_empty[s]), 2);
        }
        for (int t = 0; t < 2; ++t) {
            for (int h = 0; h < 2; ++h) {
                mbar_init(smem_u32(&sh->s_full[t][h]), 1);
                mbar_init(smem_u32(&sh->p_full[t][h]), 128);
                mbar_init(smem_u32(&sh->pv_done[t][h]), 1);
            }
            mbar_init(smem_u32(&sh->o_done[t]), 1);
            mbar_init(smem_u32(&sh->o_free[t]), 128);
        }
        mbar_init(smem_u32(&sh->drain[0]), 1);
        mbar_init(smem_u32(&sh->drain[1]), 1);
        for (int k = 0; k < kUnitRing; ++k) {
            mbar_init(smem_u32(&sh->u_full[k]), 1);
            mbar_init(smem_u32(&sh->u_empty[k]), kUnitReaders);
        }
        mbar_init(smem_u32(&sh->clc_bar), 1);
        sh->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, sh->tmem_base, 0);
    const Waiter W{&sh->abort, p.status, p.wait_limit_ns};

    // setmaxnreg is warpgroup-wide: all four warps of a group run the same one.
    if (warp >= 8)
        setmaxnreg_dec<kRegOther>();
    else
        setmaxnreg_inc<kRegSoftmax>();

    if (warp < 8) {
        softmax_role<D, kBf16, kPosScale, kMask>(p, W, sh, tmem, smem, sKVa + C::kStages * C::kTileBytes, warp, lane);
    } else if (warp == kWarpMma || warp == kWarpMma1) {
        mma_role<D, kBf16, kMask>(p, W, sh, sQa, sKVa, tmem, warp == kWarpMma ? 0 : 1);
    } else if (warp == kWarpTma) {
        if (lane == 0) tma_kv_role<D>(p, W, sh, sKVa);
    } else if (warp == kWarpTmaQ) {
        if (lane == 0) tma_q_role<D>(p, W, sh, sQa);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kBf16, bool kPos, bool kMask>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t s) {
    auto kern = fa_fwd_tc_kernel<D, kBf16, kPos, kMask>;
    constexpr int smem = smem_bytes<D>();
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    // Refuse to launch if the registers the CTA starts with cannot cover the
    // setmaxnreg split (the increase would never be granted).
    if (3 * attr.numRegs < 2 * kRegSoftmax + kRegOther) return cudaErrorLaunchOutOfResources;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// Problems with no mask or split P anywhere (and a positive scale, the usual
// case) take the build without those paths; every other one the full build.
template <int D, bool kBf16>
cudaError_t launch_dt(const TcParams& p, bool pos_scale, int grid, cudaStream_t s) {
    if (pos_scale && !geom_needs_masks(p.g)) return launch_one<D, kBf16, true, false>(p, grid, s);
    return pos_scale ? launch_one<D, kBf16, true, true>(p, grid, s) : launch_one<D, kBf16, false, true>(p, grid, s);
}

}  // namespace

cudaError_t launch_tc(const TcParams& p, int D, bool bf16, bool pos_scale, int grid, cudaStream_t s) {
    if (D == 128) return bf16 ? launch_dt<128, true>(p, pos_scale, grid, s) : launch_dt<128, false>(p, pos_scale, grid, s);
    return bf16 ? launch_dt<64, true>(p, pos_scale, grid, s) : launch_dt<64, false>(p, pos_scale, grid, s);
}

}  // namespace fa
