// Tensor-core fused attention forward over CTA pairs (sm_103a, D = 128,
// fp16 / bf16 in, fp32 accumulate).
//
// The method is that of fa_tc.cu -- the tiled online-softmax forward of
// "Ascend C advanced practice: high-performance FlashAttention-2-style
// tile-level fused attention" (sections 1.2 and 3), with the Cube/Vector
// pipelining of "FlashAttention extreme optimisation on Ascend NPUs"
// (optimisation three: the matrix unit works on block j+1 while the vector
// unit does the softmax of block j) -- laid out for two SMs at a time.
//
// The two CTAs of a cluster run on neighbouring SMs.  A unit is 256 query
// rows of one (b, h): 128 in each CTA.  One tcgen05.mma.cta_group::2 of
// M = 256 serves both: each CTA holds its own 128 rows of Q and of the
// accumulators, and half of every K tile (64 keys) and of every V tile (64 of
// the 128 columns); each SM's tensor core reads the other half from the
// peer's shared memory.  Splitting B this way keeps a 128-row tile per SM as
// cheap in shared-memory traffic as two tiles sharing full K/V tiles, which
// leaves tensor memory for three S buffers per tile: S(j+3) is computed
// while the softmax works through steps j+1 and j+2, so the softmax is never
// waiting for the products that follow its own P (the chain softmax(j) ->
// P.V(j) -> S(j+1) -> softmax(j+1) of a single S buffer is gone).  The products run as one
// stream across units, so the next unit's first scores are ready when the
// softmax reaches it.
//
//   warps 0-7   softmax: warp w takes 16 rows of TMEM lane quarter w % 4,
//               two lanes a row, each lane 64 of the row's 128 key columns;
//               the halves of a row combine their maxima by a shuffle
//   warps 8-11  per unit: release this CTA's Q tile to the products
//               (rotating it in place first when the rotary embedding of Q
//               is on) and, once the unit's last P.V lands, the epilogue
//               (O / l and LSE); the softmax warps go straight on
//   warp  12    TMEM allocator (both CTAs); in the first CTA, one elected
//               lane issues every product
//   warp  13    one thread: this CTA's halves of the K tiles (TMA, own ring)
//   warp  14    one thread: this CTA's halves of the V tiles (TMA, own ring)
//   warp  15    one thread: this CTA's Q tile of each unit (TMA, two buffers)
//
// Barriers that collect a warpgroup's work take one arrival per warp: the
// lanes finish (and fence) their own stores, the warp synchronises, and lane
// 0 arrives with release semantics.  Per-thread arrivals on a barrier in the
// other CTA cost a shared-memory transaction each across the pair.
//
// TMEM per CTA: S buffers 0, 1, 2 | O (128 columns each, all 512); P
// (16-bit) overwrites the first half of its S buffer (the second half too
// for a split bf16 P).
//
// Registers: 512 threads launch with 128 each; setmaxnreg gives the softmax
// warpgroups (64 scores a thread) 160, and the Q-release/epilogue and the
// MMA/TMA warpgroups 96 each (2 x 160 + 96 + 96 = 4 x 128).
//
// Every wait is bounded; a timeout in either CTA stops both (each raises the
// other's abort flag), and each lets its issued copies and products land
// before the pair frees tensor memory together.
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_softmax.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kLaunchRegs = (65536 / kThreads) & ~7;  // 128
constexpr int kRegSoftmax = 160;  // warpgroups 0-1
constexpr int kRegEpi = 96;       // warpgroup 2
constexpr int kRegCtl = 96;       // warpgroup 3 (MMA issue, TMA)
static_assert(2 * kRegSoftmax + kRegEpi + kRegCtl <= 4 * kLaunchRegs, "register split exceeds the launch budget");
constexpr int kWarpMma = 12;  // TMEM owner; the issuer in the first CTA
constexpr int kWarpK = 13;   // K tile loads
constexpr int kWarpV = 14;   // V tile loads
constexpr int kWarpQ = 15;
constexpr uint16_t kBothCtas = 0x3;
constexpr int kSoftmaxWarps = 8;
constexpr int kEpiWarps = 4;

struct PairCfg {
    static constexpr int D = 128;
    static constexpr int kQBox = kTileM * 64 * 2;   // 128 rows x 64 columns: 16 KiB
    static constexpr int kQTile = 2 * kQBox;        // this CTA's 128 x 128 Q tile
    static constexpr int kKBox = 64 * 64 * 2;       // 64 keys x 64 columns: 8 KiB
    static constexpr int kStage = 16384;            // half a K tile (two boxes) or half a V tile (one)
    static constexpr int kStagesK = 5;
    static constexpr int kStagesV = 4;
    static constexpr int kQBytes = 2 * kQTile;      // two buffers
    static constexpr int kTileSmem = kQBytes + (kStagesK + kStagesV) * kStage;
    static constexpr int kSBufs = 3;                // S buffers: S(g) in buffer g % 3
    static constexpr int kColS = 0;                 // S buffer b at kColS + 128 b
    static constexpr int kColO = 384;
    static constexpr int kTmemCols = 512;
};

struct __align__(16) PairCtl {
    uint64_t q_land[2];                  // [buffer] this CTA's Q tile landed (1 + bytes)
    uint64_t q_ready[2];                 // first CTA: both CTAs' tiles ready for the products (8 warps)
    uint64_t q_empty[2];                 // both: the unit's last S completed (1)
    uint64_t k_full[PairCfg::kStagesK];  // first CTA: both halves of the stage's K tile landed (1 + bytes)
    uint64_t k_empty[PairCfg::kStagesK]; // both: the S reading it completed (1)
    uint64_t v_full[PairCfg::kStagesV];  // first CTA: the same for V tiles
    uint64_t v_empty[PairCfg::kStagesV]; // both: the P.V reading it completed (1)
    uint64_t s_full[PairCfg::kSBufs];    // both: S in buffer b (1)
    uint64_t p_full[PairCfg::kSBufs];    // first CTA: P of both CTAs in buffer b (16 warps)
    uint64_t pv_done[2];                 // both: P.V of a step of this parity completed (1)
    uint64_t o_done;                     // both: the unit's last P.V completed (1)
    uint64_t o_free;                     // first CTA: both CTAs have read O out (8 warps)
    uint64_t st_full[2];                 // [unit parity] this CTA: row statistics written (8 warps)
    uint64_t drain;                      // first CTA
    uint32_t tmem_base;
    int abort;
    float2 stats[2][kTileM];             // [unit parity][row]: (reference max, row sum)
};

constexpr int smem_bytes_pair() { return PairCfg::kTileSmem + (int)sizeof(PairCtl) + 1024; }
static_assert(smem_bytes_pair() <= 227 * 1024, "shared memory budget");
// S(g+3) is issued right after P.V(g): its K stage was last read by S(g+3-kStagesK),
// issued (and waited for) earlier, so the K ring needs at least four stages
// to keep S three steps ahead; V stages are read in order.
static_assert(PairCfg::kStagesK >= 4 && PairCfg::kStagesV >= 2, "K or V ring too short for the issue order");

// Arrive on the first CTA's copy of barrier `bar`: a plain arrival there;
// from the second CTA through the shared-memory window, with a cluster-scope
// release when the arrival publishes shared-memory stores (kPublishSmem), the
// default release when it publishes tensor memory (see mbar_arrive_remote).
template <bool kPublishSmem>
__device__ __forceinline__ void arrive_first(uint32_t bar, uint32_t rank) {
    if (rank == 0)
        mbar_arrive(bar);
    else if (kPublishSmem)
        mbar_arrive_cluster(mapa_shared(bar, 0));
    else
        mbar_arrive_remote(mapa_shared(bar, 0));
}

// ------------------------------------------------------------- Q producer
// This CTA's Q tile of every unit, rows [q0 + 128 rank, +128), into buffer
// (unit count & 1); a buffer is refilled once the last S of the unit two
// back has completed.
__device__ __forceinline__ void q_role(const TcParams& p, const PairWaiter& W, PairCtl* sh, uint32_t sQ,
                                       uint32_t rank, int cl, int ncl) {
    using C = PairCfg;
    tma_prefetch_desc(&p.tm_q);
    int last0 = -1, last1 = -1;  // unit count of each buffer's latest load
    bool ok = true;
    int k = 0;
    for (int r = 0, u; (u = sched_unit(r, cl, ncl)) < p.n_units && ok; ++r, ++k) {
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int b = un.bh / p.H, h = un.bh % p.H;
        const uint32_t buf = (uint32_t)k & 1;
        if (k >= 2 && !(ok = W.wait(smem_u32(&sh->q_empty[buf]), ((k >> 1) - 1) & 1))) break;
        const uint32_t land = smem_u32(&sh->q_land[buf]);
        mbar_arrive_expect_tx(land, C::kQTile);
        tma_load_5d(sQ + buf * C::kQTile, &p.tm_q, land, 0, un.q0 + kTileM * (int)rank, 0, h, b);
        if (buf)
            last1 = k;
        else
            last0 = k;
    }
    // Let every issued copy land before shared memory is released (on the
    // normal path too: after an abort nobody may wait for them).
    const uint64_t t0 = globaltimer_ns();
    if (last0 >= 0) W.drain(smem_u32(&sh->q_land[0]), (last0 >> 1) & 1, t0);
    if (last1 >= 0) W.drain(smem_u32(&sh->q_land[1]), (last1 >> 1) & 1, t0);
}

// ----------------------------------------------------------- K, V producers
// Two threads, one per ring: this CTA's half of K_j (keys [64 rank, +64), two
// 64 x 64 boxes) or of V_j (columns [64 rank, +64), one 128 x 64 box) for
// every key tile of every unit.  Separate rings let each run as far ahead as
// its own stages allow: S(g) reads K three steps before P.V(g) reads V, so
// with one ring K loads would queue behind V's later-released stages.  Both
// halves of a tile complete on the first CTA's barrier, which the first CTA's
// producer arms with the bytes of both.
template <bool kIsV>
__device__ __forceinline__ void ring_role(const TcParams& p, const PairWaiter& W, uint64_t* full_bar,
                                          uint64_t* empty_bar, uint32_t sRing, uint32_t rank, int cl, int ncl) {
    using C = PairCfg;
    constexpr int kN = kIsV ? C::kStagesV : C::kStagesK;
    const CUtensorMap* tm = kIsV ? &p.tm_v : &p.tm_k;
    tma_prefetch_desc(tm);
    uint32_t n = 0, s = 0, ph = 0;  // tiles issued; stage and phase bit of tile n
    bool ok = true;
    for (int r = 0, u; (u = sched_unit(r, cl, ncl)) < p.n_units && ok; ++r) {
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int b = un.bh / p.H, hk = (un.bh % p.H) / p.G;
        for (int j = un.jlo; j < un.jhi; ++j) {
            // the stage's previous tile (n - kN) has been read
            if (n >= (uint32_t)kN && !(ok = W.wait(smem_u32(&empty_bar[s]), ph ^ 1))) break;
            const uint32_t full = smem_u32(&full_bar[s]);
            if (rank == 0) mbar_arrive_expect_tx(full, 2 * C::kStage);
            const uint32_t full_first = mapa_shared(full, 0);
            const uint32_t dst = sRing + s * C::kStage;
            // one instruction per half tile: K keys [64 rank, +64) x both chunks,
            // V keys [0, 128) x chunk `rank`
            if (!kIsV)
                tma_load_5d_pair(dst, tm, full_first, 0, j * kTileN + 64 * (int)rank, 0, hk, b);
            else
                tma_load_5d_pair(dst, tm, full_first, 0, j * kTileN, (int)rank, hk, b);
            ++n;
            if (++s == (uint32_t)kN) {
                s = 0;
                ph ^= 1;
            }
        }
    }
    // This CTA's copies complete on the first CTA's barriers, so wait instead
    // until the products have released every stage they were loaded into: on
    // the normal path that means they landed and were read; after an abort
    // the bounded wait covers their flight.  Tile m sits in stage m % kN and
    // its release completes phase m / kN of that stage's empty barrier.
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t st = 0; st < (uint32_t)kN && st < n; ++st) {
        const uint32_t last = n - 1 - ((n - 1 - st) % kN);
        W.drain(smem_u32(&empty_bar[st]), (last / kN) & 1, t0);
    }
}

// A position in the stream of key steps: unit (round r, unit index u, count
// k of units taken) and key tile j.  Step g (counted over all units) keeps S
// in buffer g & 1 and uses ring stages 2g (K) and 2g + 1 (V).
struct StepCursor {
    int r, u, k, j;
    Unit un;
    __device__ __forceinline__ bool valid(const TcParams& p) const { return u < p.n_units; }
    __device__ __forceinline__ void start(const TcParams& p, int cl, int ncl) {
        r = 0;
        k = 0;
        u = sched_unit(0, cl, ncl);
        if (u < p.n_units) {
            un = make_unit(p.g, p.BH, p.order, u);
            j = un.jlo;
        }
    }
    __device__ __forceinline__ void next(const TcParams& p, int cl, int ncl) {
        if (++j < un.jhi) return;
        ++r;
        ++k;
        u = sched_unit(r, cl, ncl);
        if (u < p.n_units) {
            un = make_unit(p.g, p.BH, p.order, u);
            j = un.jlo;
        }
    }
};

// --------------------------------------------------------------- MMA issuer
// First CTA only.  S(g) = Q K_j^T into buffer g % 3 runs three steps ahead
// of O += P(g) V_j: after P.V(g) the issuer puts out S(g + 3), which reuses
// the buffer P.V(g) just read (products of one thread execute in order), so
// the softmax has two more steps of scores in hand while that P.V and S run.
// The stream runs across units, so S of a unit's first steps follows the
// last P.V of the unit before.
template <bool kBf16>
__device__ __forceinline__ void mma_role(const TcParams& p, const PairWaiter& W, PairCtl* sh, uint32_t sQ,
                                         uint32_t sK, uint32_t sV, uint32_t tmem, int cl, int ncl) {
    using C = PairCfg;
    constexpr uint32_t idesc_s = make_idesc(kBf16, 2 * kTileM, kTileN, false);
    constexpr uint32_t idesc_o = make_idesc(kBf16, 2 * kTileM, C::D, true);
    const uint32_t dO = tmem + C::kColO;
    const bool leader = elect_one();
    // K half: 64 keys, K-major, 128-byte swizzle, D in two 64-column boxes;
    // Q: 128 rows, two 16 KiB boxes; V half: 128 keys x 64 columns, MN-major.
    const uint64_t k_desc = make_sdesc(sK, 16, 1024);
    const uint64_t v_desc = make_sdesc(sV, C::kStage, 1024);
    bool ok = true;

    StepCursor sc, pc;  // next S, next P.V
    sc.start(p, cl, ncl);
    pc.start(p, cl, ncl);
    uint32_t gs = 0, gp = 0;  // steps whose S / P.V have been issued
    uint32_t sbuf = 0, sph = 0;  // buffer of S(gs), and the phase bit of its barriers
    uint32_t pbuf = 0, pph = 0;  // the same for P(gp)
    int q_seen = -1;          // last unit whose Q this issuer has waited for
    uint32_t o_units = 0;     // units whose last P.V has been issued

    uint32_t ks = 0, kph = 0, vs = 0, vph = 0;  // ring stage and phase bit of K(gs) and V(gp)
    // S for the step at the S cursor.
    auto issue_s = [&]() {
        if (sc.k != q_seen) {
            const uint32_t qb = (uint32_t)sc.k & 1;
            if (!W.wait_warp<true>(smem_u32(&sh->q_ready[qb]), (sc.k >> 1) & 1)) return false;
            q_seen = sc.k;
        }
        if (!W.wait_warp(smem_u32(&sh->k_full[ks]), kph)) return false;
        tc_fence_after();
        const uint32_t dS = tmem + C::kColS + 128 * sbuf;
        const uint64_t kb = k_desc + (uint64_t)(ks * (uint32_t)(C::kStage >> 4));
        const uint64_t qd = make_sdesc(sQ + ((uint32_t)sc.k & 1) * C::kQTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
            const uint32_t oq = ((kk / 4) * C::kQBox + (kk % 4) * 32) >> 4;
            const uint32_t okk = ((kk / 4) * C::kKBox + (kk % 4) * 32) >> 4;
            if (leader) mma_ss_pair(dS, qd + oq, kb + okk, idesc_s, kk > 0);
        }
        if (leader) mma_commit_pair_mc(smem_u32(&sh->s_full[sbuf]), kBothCtas);
        if (leader) mma_commit_pair_mc(smem_u32(&sh->k_empty[ks]), kBothCtas);
        if (++ks == (uint32_t)C::kStagesK) {
            ks = 0;
            kph ^= 1;
        }
        // the unit's last S: its Q buffer may be refilled once this completes
        if (sc.j == sc.un.jhi - 1 && leader) mma_commit_pair_mc(smem_u32(&sh->q_empty[sc.k & 1]), kBothCtas);
        ++gs;
        if (++sbuf == (uint32_t)C::kSBufs) {
            sbuf = 0;
            sph ^= 1;
        }
        sc.next(p, cl, ncl);
        return true;
    };

    for (int i = 0; i < C::kSBufs && ok && sc.valid(p); ++i) ok = issue_s();
    while (ok && pc.valid(p)) {
        const bool first = pc.j == pc.un.jlo;
        const bool split = kBf16 && slot_split_p(p.g, pc.un.q0);
        if (!(ok = W.wait_warp(smem_u32(&sh->v_full[vs]), vph))) break;
        if (first && o_units > 0 && !(ok = W.wait_warp(smem_u32(&sh->o_free), (o_units - 1) & 1))) break;
        if (!(ok = W.wait_warp(smem_u32(&sh->p_full[pbuf]), pph))) break;
        tc_fence_after();
        // O += P V: P from tensor memory (8 columns = 16 keys a step), V's 16
        // keys = two 8-row swizzle atoms = 2048 bytes a step; a split P adds
        // the low halves (64 columns on) in a second pass.
        const uint32_t dP = tmem + C::kColS + 128 * pbuf;
        const uint64_t vb = v_desc + (uint64_t)(vs * (uint32_t)(C::kStage >> 4));
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
            const uint64_t b = vb + (uint64_t)(kk * (2048 >> 4));
            if (leader) mma_ts_pair(dO, dP + kk * 8, b, idesc_o, (first && kk == 0) ? 0u : 1u);
        }
        if (split) {
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk) {
                const uint64_t b = vb + (uint64_t)(kk * (2048 >> 4));
                if (leader) mma_ts_pair(dO, dP + 64 + kk * 8, b, idesc_o, 1u);
            }
        }
        if (leader) mma_commit_pair_mc(smem_u32(&sh->pv_done[gp & 1]), kBothCtas);
        if (leader) mma_commit_pair_mc(smem_u32(&sh->v_empty[vs]), kBothCtas);
        if (++vs == (uint32_t)C::kStagesV) {
            vs = 0;
            vph ^= 1;
        }
        if (pc.j == pc.un.jhi - 1) {
            if (leader) mma_commit_pair_mc(smem_u32(&sh->o_done), kBothCtas);
            ++o_units;
        }
        ++gp;
        if (++pbuf == (uint32_t)C::kSBufs) {
            pbuf = 0;
            pph ^= 1;
        }
        pc.next(p, cl, ncl);
        if (sc.valid(p)) ok = issue_s();
    }
    // Every issued product must complete before tensor memory is released.
    const uint32_t drain = smem_u32(&sh->drain);
    if (leader) mma_commit_pair(drain);
    W.drain(drain, 0, globaltimer_ns());
}

// ------------------------------------------------------------------ softmax
// Warp w holds 16 rows: TMEM lane quarter w % 4, the upper or lower 16 of it
// by w / 4.  Lane l takes row (l % 16) of those, key columns [64 h, 64 h + 64)
// with h = l / 16 (the .16x32bx2 access shape), so the two halves of a row
// sit in one warp and combine their maxima and sums with one shuffle.  The
// online softmax is that of the one-CTA kernel (tc_softmax.cuh).
template <bool kBf16, bool kPosScale>
__device__ __forceinline__ void softmax_role(const TcParams& p, const PairWaiter& W, PairCtl* sh, uint32_t tmem,
                                             uint32_t rank, int warp, int lane, int cl, int ncl) {
    using C = PairCfg;
    const int row = 32 * (warp & 3) + 16 * (warp >> 2) + (lane & 15);
    const int hf = lane >> 4;
    const int col0 = 64 * hf;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3) + 16 * (warp >> 2)) << 16;
    const uint32_t tO = tmem + lanes + C::kColO;
    const float c2 = p.scale_log2;
    uint32_t g = 0;              // key steps done
    uint32_t sb = 0, sph = 0;    // S buffer of step g (g % 3) and the phase bit of its barriers
    bool ok = true;
    int k = 0;
    for (int r = 0, u; (u = sched_unit(r, cl, ncl)) < p.n_units && ok; ++r, ++k) {
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int r0 = un.q0 + (int)rank * kTileM;
        const int qi = r0 + row;
        const bool split = kBf16 && slot_split_p(p.g, un.q0);
        float m_ref = -INFINITY;
        float l = 0.f;
        for (int j = un.jlo; j < un.jhi; ++j, ++g) {
            if (!(ok = W.wait_warp(smem_u32(&sh->s_full[sb]), sph))) break;
            tc_fence_after();
            const uint32_t tS = tmem + lanes + C::kColS + 128 * sb;
            uint32_t s[2][32];
            tmem_ld32_x2<64>(tS, s[0]);
            tmem_ld32_x2<64>(tS + 32, s[1]);
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
            if (tile_needs_mask(p.g, r0, j)) {
                int c_lo, c_hi;
                row_visible_cols(p.g, qi, j, c_lo, c_hi);
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = col0 + c * 32 + i;
                        if (col < c_lo || col > c_hi) s[c][i] = f2u(-INFINITY);
                    }
            }
            float mxk[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mxk[q] = fmaxf(u2f(s[0][2 * q]), u2f(s[0][2 * q + 1]));
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int i = (c == 0 ? 16 : 0); i < 32; i += 2) {
                    const int q = (i >> 1) & 7;
                    mxk[q] = max3(mxk[q], u2f(s[c][i]), u2f(s[c][i + 1]));
                }
            float mx = fmaxf(max3(mxk[0], mxk[1], mxk[2]), max3(max3(mxk[3], mxk[4], mxk[5]), mxk[6], mxk[7]));
            // Both halves end with the same row max, hence the same decisions.
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = kPosScale ? mx * c2 : mx;
            const bool first = j == un.jlo;
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
            // P for keys [col0, col0 + 64) goes to columns [col0 / 2, +32) of the
            // buffer (16-bit pairs); a split bf16 P puts the low parts 64
            // columns further on.  S is all in registers (the ld above waited),
            // so P may overwrite it.
            if (!split) {
                float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float a, b;
                        if (kPosScale)
                            ffma2(a, b, u2f(s[c][i]), u2f(s[c][i + 1]), c2, c2, neg_m, neg_m);
                        else
                            fadd2(a, b, u2f(s[c][i]), u2f(s[c][i + 1]), neg_m, neg_m);
                        a = ex2(a);
                        b = ex2(b);
                        pk[16 * c + (i >> 1)] = pack2<kBf16>(a, b);
                        const int q = (i >> 1) & 3;
                        fadd2(acc[q][0], acc[q][1], acc[q][0], acc[q][1], a, b);
                    }
                }
                tmem_st32_x2<32>(tS, pk);
                l0 = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
                l1 = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
            } else {
                uint32_t hw[32], lw[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float a = kPosScale ? ex2(fmaf(u2f(s[c][i]), c2, neg_m)) : ex2(u2f(s[c][i]) + neg_m);
                        const float b =
                            kPosScale ? ex2(fmaf(u2f(s[c][i + 1]), c2, neg_m)) : ex2(u2f(s[c][i + 1]) + neg_m);
                        const uint32_t w = pack2<kBf16>(a, b);
                        hw[16 * c + (i >> 1)] = w;
                        lw[16 * c + (i >> 1)] = pack2<kBf16>(a - lo_half<kBf16>(w), b - hi_half<kBf16>(w));
                        l0 += a;
                        l1 += b;
                    }
                }
                tmem_st32_x2<32>(tS, hw);
                tmem_st32_x2<32>(tS + 64, lw);
            }
            if (!first && __any_sync(0xffffffffu, resc)) {
                // Rare: the running max moved by more than kTau; rescale this
                // lane's half of the row of O, once the previous P.V, which
                // writes O, has completed (its commit also covers the P.V
                // before it).  P.V of odd and even steps commit to separate
                // barriers, and waiting only here is safe: S(g) has completed,
                // so P.V(g-3) (issued before it) has too, and P.V(g+1) needs a
                // later P, so the barrier of P.V(g-1) sits in that P.V's phase
                // or the one after.
                if (!(ok = W.wait_warp(smem_u32(&sh->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32_x2<64>(tO + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                    tmem_st32_x2<64>(tO + c * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_first<false>(smem_u32(&sh->p_full[sb]), rank);
            l += l0 + l1;
            if (++sb == (uint32_t)C::kSBufs) {
                sb = 0;
                sph ^= 1;
            }
        }
        if (!ok) break;
        // Hand the row's statistics to the epilogue warps.
        const float lrow = l + __shfl_xor_sync(0xffffffffu, l, 16);
        if (hf == 0) sh->stats[k & 1][row] = make_float2(m_ref, lrow);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->st_full[k & 1]));
    }
}

// ---------------------------------------------- Q release and epilogue
template <bool kBf16>
__device__ __forceinline__ void epi_role(const TcParams& p, const PairWaiter& W, PairCtl* sh, uint8_t* sQg,
                                         uint32_t tmem, uint32_t rank, int warp, int lane, int cl, int ncl) {
    using C = PairCfg;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;

    // Unit k's Q tile: wait for this CTA's copy, rotate this thread's row in
    // place when the rotary embedding of Q is on, make the stores visible to
    // the tensor core, and tell the first CTA's issuer.
    auto release_q = [&](int k, const Unit& un) {
        const uint32_t buf = (uint32_t)k & 1;
        if (!W.wait_warp(smem_u32(&sh->q_land[buf]), (k >> 1) & 1)) return false;
        if (p.rope) {
            const int qi = un.q0 + (int)rank * kTileM + row;
            if (qi < p.g.N) {
                const long long pos = (long long)p.rope_pos0 + qi;
                rope_q_row<C::D, kBf16, C::kQBox>(sQg + buf * C::kQTile, row, p.rope_cos + pos * (C::D / 2),
                                                   p.rope_sin + pos * (C::D / 2), p.rope_style);
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) arrive_first<true>(smem_u32(&sh->q_ready[buf]), rank);
        return true;
    };

    int k = 0;
    {
        const int u0 = sched_unit(0, cl, ncl);
        if (u0 < p.n_units) ok = release_q(0, make_unit(p.g, p.BH, p.order, u0));
    }
    for (int r = 0, u; (u = sched_unit(r, cl, ncl)) < p.n_units && ok; ++r, ++k) {
        const Unit un = make_unit(p.g, p.BH, p.order, u);
        const int un_next = sched_unit(r + 1, cl, ncl);
        if (un_next < p.n_units && !(ok = release_q(k + 1, make_unit(p.g, p.BH, p.order, un_next)))) break;
        if (!(ok = W.wait_warp(smem_u32(&sh->o_done), k & 1))) break;
        if (!(ok = W.wait_warp(smem_u32(&sh->st_full[k & 1]), (k >> 1) & 1))) break;
        tc_fence_after();
        const float2 s0 = sh->stats[k & 1][row];
        const float lsum = s0.y;
        const float inv = 1.f / lsum;
        const int b = un.bh / p.H, h = un.bh % p.H;
        const int qi = un.q0 + (int)rank * kTileM + row;
        const bool live = qi < p.g.N;
        const size_t orow = (size_t)row_index(p.layout, b, h, live ? qi : 0, p.H, p.g.N);
        const uint32_t tO = tmem + lane_base + C::kColO;
#pragma unroll 1
        for (int c = 0; c < C::D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_wait_ld();
            if (!live) continue;
            if (p.o_f32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * C::D + c * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_float4(u2f(o[4 * i]) * inv, u2f(o[4 * i + 1]) * inv, u2f(o[4 * i + 2]) * inv,
                                         u2f(o[4 * i + 3]) * inv);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * C::D + c * 16);
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    dst[i] = make_uint4(pack2<kBf16>(u2f(o[8 * i]) * inv, u2f(o[8 * i + 1]) * inv),
                                        pack2<kBf16>(u2f(o[8 * i + 2]) * inv, u2f(o[8 * i + 3]) * inv),
                                        pack2<kBf16>(u2f(o[8 * i + 4]) * inv, u2f(o[8 * i + 5]) * inv),
                                        pack2<kBf16>(u2f(o[8 * i + 6]) * inv, u2f(o[8 * i + 7]) * inv));
            }
        }
        if (live && p.lse) p.lse[(size_t)un.bh * p.g.N + qi] = (s0.x + log2f(lsum)) * kLn2;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_first<false>(smem_u32(&sh->o_free), rank);
    }
}

template <bool kBf16, bool kPosScale>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_tc2_kernel(const __grid_constant__ TcParams p) {
    using C = PairCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairCtl* sh = reinterpret_cast<PairCtl*>(smem + C::kTileSmem);
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + C::kQBytes;
    const uint32_t sV = sK + C::kStagesK * C::kStage;
    const uint32_t rank = cluster_ctarank();
    const int cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sh->q_land[b]), 1);
            mbar_init(smem_u32(&sh->q_ready[b]), 2 * kEpiWarps);
            mbar_init(smem_u32(&sh->q_empty[b]), 1);
            mbar_init(smem_u32(&sh->st_full[b]), kSoftmaxWarps);
            mbar_init(smem_u32(&sh->pv_done[b]), 1);
        }
        for (int s = 0; s < C::kStagesK; ++s) {
            mbar_init(smem_u32(&sh->k_full[s]), 1);
            mbar_init(smem_u32(&sh->k_empty[s]), 1);
        }
        for (int s = 0; s < C::kStagesV; ++s) {
            mbar_init(smem_u32(&sh->v_full[s]), 1);
            mbar_init(smem_u32(&sh->v_empty[s]), 1);
        }
        for (int b = 0; b < C::kSBufs; ++b) {
            mbar_init(smem_u32(&sh->s_full[b]), 1);
            mbar_init(smem_u32(&sh->p_full[b]), 2 * kSoftmaxWarps);
        }
        mbar_init(smem_u32(&sh->o_done), 1);
        mbar_init(smem_u32(&sh->o_free), 2 * kEpiWarps);
        mbar_init(smem_u32(&sh->drain), 1);
        sh->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc_pair(smem_u32(&sh->tmem_base), C::kTmemCols);
        tmem_relinquish_pair();
    }
    // Both CTAs' barriers and tensor memory exist before either touches the
    // other's.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, sh->tmem_base, 0);
    const PairWaiter W{&sh->abort, mapa_generic(&sh->abort, rank ^ 1u), p.status, p.wait_limit_ns};

    if (warp >= 12)
        setmaxnreg_dec<kRegCtl>();
    else if (warp >= 8)
        setmaxnreg_dec<kRegEpi>();
    else
        setmaxnreg_inc<kRegSoftmax>();

    if (warp < 8) {
        softmax_role<kBf16, kPosScale>(p, W, sh, tmem, rank, warp, lane, cl, ncl);
    } else if (warp < 12) {
        epi_role<kBf16>(p, W, sh, smem, tmem, rank, warp, lane, cl, ncl);
    } else if (warp == kWarpMma) {
        if (rank == 0) mma_role<kBf16>(p, W, sh, sQ, sK, sV, tmem, cl, ncl);
    } else if (warp == kWarpK) {
        if (lane == 0) ring_role<false>(p, W, sh->k_full, sh->k_empty, sK, rank, cl, ncl);
    } else if (warp == kWarpV) {
        if (lane == 0) ring_role<true>(p, W, sh->v_full, sh->v_empty, sV, rank, cl, ncl);
    } else if (warp == kWarpQ) {
        if (lane == 0) q_role(p, W, sh, sQ, rank, cl, ncl);
    }

    // The first CTA's products read the second CTA's shared memory and write
    // its tensor memory: both wait here until they have all completed.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

template <bool kBf16, bool kPos>
cudaError_t launch_pair(const TcParams& p, int clusters, cudaStream_t s) {
    auto kern = fa_fwd_tc2_kernel<kBf16, kPos>;
    constexpr int smem = smem_bytes_pair();
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    // Refuse to launch if the registers the CTA starts with cannot cover the
    // setmaxnreg split (the increase would never be granted).
    if (4 * attr.numRegs < 2 * kRegSoftmax + kRegEpi + kRegCtl) return cudaErrorLaunchOutOfResources;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_pair(const TcParams& p, bool bf16, bool pos_scale, int clusters, cudaStream_t s) {
    if (bf16) return pos_scale ? launch_pair<true, true>(p, clusters, s) : launch_pair<true, false>(p, clusters, s);
    return pos_scale ? launch_pair<false, true>(p, clusters, s) : launch_pair<false, false>(p, clusters, s);
}

}  // namespace fa
