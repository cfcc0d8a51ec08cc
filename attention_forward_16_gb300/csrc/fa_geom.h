// Tile geometry shared by the host planner and the kernels: which key tiles a
// block of query rows must visit under a mask, which of those need
// per-element masking, and how persistent CTAs enumerate work units.
//
// Mask semantics ("Ascend C advanced practice: high-performance
// FlashAttention-2-style tile-level fused attention", section 4.2 for causal;
// "FlashAttention under the catlass template", section "Usage" for the
// (window_left, window_right) tuple): key j is visible to query i iff
//     (win_l < 0 || j >= i - win_l) && (win_r < 0 || j <= i + win_r) && j < N.
// Causal is the window (-1, 0) and no mask is (-1, -1).  Skipping key tiles
// that are wholly masked is the causal block skip of that page's section 6,
// generalised to the window.
#pragma once

#ifdef __CUDACC__
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int kTileM = 128;  // query rows per Q tile (one tcgen05 M=128 accumulator)
constexpr int kTileN = 128;  // keys per K/V tile

// Unit enumeration orders (longest-first for masks whose work grows with q).
// ORDER_GRP_Q_DESC takes the heads in groups of heads_per_group(N), each
// group longest first: the group's K/V stays in L2 while its units run.
enum UnitOrder { ORDER_HEAD_MAJOR = 0, ORDER_Q_DESC = 1, ORDER_Q_ASC = 2, ORDER_GRP_Q_DESC = 3 };

// Heads per group of ORDER_GRP_Q_DESC: a group's keys and values (N keys of
// D = 128 at 16 bits, 2 MB a head at N = 4,096) fill about half of the 126 MB
// L2; with units handed out dynamically, 32 heads at N = 4,096 measured
// fastest among 16, 24, 32, 48, 64 and all 128.
FA_HD int heads_per_group(int N) {
    const long long g = (32LL * 4096) / (N > 0 ? N : 1);
    return g < 1 ? 1 : (int)g;
}

struct Geom {
    int N;       // sequence length (queries == keys)
    int win_l;   // -1 = unbounded
    int win_r;   // -1 = unbounded
};

// Key-tile range [lo, hi) that rows [r0, r1) (r0 < r1 <= N) must visit.
FA_HD void kv_tile_range(const Geom& g, int r0, int r1, int& lo, int& hi) {
    int kmin = g.win_l < 0 ? 0 : r0 - g.win_l;
    if (kmin < 0) kmin = 0;
    long long kmax = g.win_r < 0 ? (long long)g.N - 1 : (long long)(r1 - 1) + g.win_r;
    if (kmax > g.N - 1) kmax = g.N - 1;
    lo = kmin / kTileN;
    hi = (int)(kmax / kTileN) + 1;
}

// True if key tile j (keys [j*kTileN, +kTileN)) holds a masked element for
// some row of [r0, r0 + kTileM): ragged tail, left or right band edge.
FA_HD bool tile_needs_mask(const Geom& g, int r0, int j) {
    long long k0 = (long long)j * kTileN;
    if (k0 + kTileN > g.N) return true;
    if (g.win_l >= 0 && k0 < (long long)r0 + (kTileM - 1) - g.win_l) return true;
    if (g.win_r >= 0 && k0 + (kTileN - 1) > (long long)r0 + g.win_r) return true;
    return false;
}

// Visible column interval [c_lo, c_hi] (tile-local, may be empty) of query row i
// inside key tile j.
FA_HD void row_visible_cols(const Geom& g, int i, int j, int& c_lo, int& c_hi) {
    long long k0 = (long long)j * kTileN;
    long long lo = g.win_l < 0 ? 0 : (long long)i - g.win_l - k0;
    long long hi = g.win_r < 0 ? (long long)kTileN - 1 : (long long)i + g.win_r - k0;
    long long tail = (long long)g.N - 1 - k0;
    if (hi > tail) hi = tail;
    if (lo < 0) lo = 0;
    if (hi > kTileN - 1) hi = kTileN - 1;
    c_lo = (int)(lo > kTileN ? kTileN : lo);
    c_hi = (int)(hi < -1 ? -1 : hi);
}

// Query-tile range [lo, hi) holding a row that sees some key of key tile j
// (the transpose of kv_tile_range, for passes that hold a key tile and walk
// the query tiles); lo == hi when no row sees any of its keys.
FA_HD void q_tile_range(const Geom& g, int j, int& lo, int& hi) {
    const long long c0 = (long long)j * kTileN;
    long long c1 = c0 + kTileN - 1;
    if (c1 > g.N - 1) c1 = g.N - 1;
    long long rmin = g.win_r < 0 ? 0 : c0 - g.win_r;
    long long rmax = g.win_l < 0 ? (long long)g.N - 1 : c1 + g.win_l;
    if (rmin < 0) rmin = 0;
    if (rmax > g.N - 1) rmax = g.N - 1;
    if (c0 > g.N - 1 || rmin > rmax) {
        lo = hi = 0;
        return;
    }
    lo = (int)(rmin / kTileM);
    hi = (int)(rmax / kTileM) + 1;
}

// Visible row interval [r_lo, r_hi] (tile-local, may be empty) of key kc
// inside query tile i: rows r with kc - win_r <= r <= kc + win_l, r < N.
FA_HD void key_visible_rows(const Geom& g, int kc, int i, int& r_lo, int& r_hi) {
    const long long r0 = (long long)i * kTileM;
    long long lo = g.win_r < 0 ? 0 : (long long)kc - g.win_r - r0;
    long long hi = g.win_l < 0 ? (long long)kTileM - 1 : (long long)kc + g.win_l - r0;
    const long long tail = (long long)g.N - 1 - r0;
    if (hi > tail) hi = tail;
    if (kc > g.N - 1) hi = -1;
    if (lo < 0) lo = 0;
    if (hi > kTileM - 1) hi = kTileM - 1;
    r_lo = (int)(lo > kTileM ? kTileM : lo);
    r_hi = (int)(hi < -1 ? -1 : hi);
}

// Fewest visible keys over rows [r0, r1) (r0 < r1 <= N).  The count per row,
// min(N-1, i+win_r) - max(0, i-win_l) + 1, is concave in i, so the minimum
// sits at one end of the range.
FA_HD long long min_visible_keys(const Geom& g, int r0, int r1) {
    long long best = -1;
    const int ends[2] = {r0, r1 - 1};
    for (int e = 0; e < 2; ++e) {
        const long long i = ends[e];
        long long lo = g.win_l < 0 ? 0 : i - g.win_l;
        if (lo < 0) lo = 0;
        long long hi = g.win_r < 0 ? (long long)g.N - 1 : i + g.win_r;
        if (hi > g.N - 1) hi = g.N - 1;
        const long long c = hi - lo + 1;
        if (best < 0 || c < best) best = c;
    }
    return best;
}

// Rows that see fewer keys than this carry the bf16 probabilities as an
// unevaluated hi + lo pair (two P.V products): with few keys the 2^-8
// relative rounding of a single bf16 P does not average out.
constexpr int kSplitKeys = 512;

FA_HD bool tile_split_p(const Geom& g, int r0) {
    if (r0 >= g.N) return false;
    const int r1 = r0 + kTileM < g.N ? r0 + kTileM : g.N;
    return min_visible_keys(g, r0, r1) < kSplitKeys;
}

// False when no tile of the problem needs an element mask or a split P: no
// window or causal bound, whole key tiles only (N a multiple of kTileN), and
// every row sees all N >= kSplitKeys keys.  tile_needs_mask and tile_split_p
// are then false everywhere, and the forward kernel can be built without
// those paths.
FA_HD bool geom_needs_masks(const Geom& g) {
    return g.win_l >= 0 || g.win_r >= 0 || g.N % kTileN != 0 || g.N < kSplitKeys;
}

// One persistent work unit: two consecutive 128-row Q tiles of one (b, h).
struct Unit {
    int bh;      // b * H + h
    int q0;      // first query row of tile 0
    int lo[2];   // key-tile range per Q tile; lo == hi means the tile is empty
    int hi[2];
    int jlo;     // union of both ranges
    int jhi;
};

FA_HD int n_pairs_for(int N) { return (N + 2 * kTileM - 1) / (2 * kTileM); }

// Units of the CTA-pair kernel: four 128-row Q tiles, two 256-row slots.
// Slot t covers rows [q0 + 256 t, q0 + 256 t + 256): its first 128 rows sit
// in the pair's first CTA and the next 128 in the second, and one M = 256
// product serves both, so both visit every key tile any of the 256 rows needs.
constexpr int kSlotRowsPair = 2 * kTileM;
FA_HD int n_quads_for(int N) { return (N + 2 * kSlotRowsPair - 1) / (2 * kSlotRowsPair); }

// Unit u in enumeration order `order`, with slots of `slot_rows` query rows.
FA_HD Unit make_unit_rows(const Geom& g, int BH, int order, int u, int slot_rows) {
    const int np = (g.N + 2 * slot_rows - 1) / (2 * slot_rows);
    int bh, pair;
    if (order == ORDER_HEAD_MAJOR) {
        bh = u / np;
        pair = u % np;
    } else if (order == ORDER_GRP_Q_DESC) {
        const int G = heads_per_group(g.N) < BH ? heads_per_group(g.N) : BH;
        const int grp = u / (G * np), v = u % (G * np);
        const int g0 = grp * G, gh = BH - g0 < G ? BH - g0 : G;
        pair = np - 1 - v / gh;
        bh = g0 + v % gh;
    } else if (order == ORDER_Q_DESC) {
        pair = np - 1 - u / BH;
        bh = u % BH;
    } else {
        pair = u / BH;
        bh = u % BH;
    }
    Unit un;
    un.bh = bh;
    un.q0 = pair * 2 * slot_rows;
    un.jlo = 0x7fffffff;
    un.jhi = 0;
    for (int t = 0; t < 2; ++t) {
        int r0 = un.q0 + t * slot_rows;
        if (r0 >= g.N) {
            un.lo[t] = un.hi[t] = 0;
            continue;
        }
        int r1 = r0 + slot_rows < g.N ? r0 + slot_rows : g.N;
        kv_tile_range(g, r0, r1, un.lo[t], un.hi[t]);
        if (un.lo[t] < un.jlo) un.jlo = un.lo[t];
        if (un.hi[t] > un.jhi) un.jhi = un.hi[t];
    }
    return un;
}

FA_HD Unit make_unit(const Geom& g, int BH, int order, int u) { return make_unit_rows(g, BH, order, u, kTileM); }
FA_HD Unit make_unit_pair(const Geom& g, int BH, int order, int u) {
    return make_unit_rows(g, BH, order, u, kSlotRowsPair);
}

// bf16 split of P for a 256-row slot of the pair kernel: both CTAs take the
// same decision (one product reads both halves), split if either half needs it.
FA_HD bool slot_split_p(const Geom& g, int r0) {
    return tile_split_p(g, r0) || tile_split_p(g, r0 + kTileM);
}

// The unit a persistent CTA takes in round r: rounds hand out `ctas`
// consecutive units, in CTA order on even rounds and in reverse order on odd
// ones.  Units come longest first under masks whose work varies by query
// tile, so plain round robin would give the low CTAs the longer unit of every
// round; alternating the direction pairs a longer unit with a shorter one and
// evens out the total per CTA.  Once r * ctas + (unit offset) passes the last
// unit, no later round has one for this CTA either.
FA_HD int sched_unit(int r, int cta, int ctas) {
    const long long u = (long long)r * ctas + ((r & 1) ? ctas - 1 - cta : cta);
    return u > 0x7fffffffLL ? 0x7fffffff : (int)u;  // past any unit count
}

FA_HD int unit_order_for(const Geom& g) {
    if (g.win_r >= 0 && g.win_l < 0) return ORDER_GRP_Q_DESC;  // causal-like: later rows see more keys
    if (g.win_r >= 0) return ORDER_Q_DESC;   // band: the edge units at the start are shorter
    if (g.win_l >= 0) return ORDER_Q_ASC;    // earlier rows see more keys
    return ORDER_HEAD_MAJOR;                 // uniform work: keep one head's K/V hot in L2
}

}  // namespace fa
