// Internal (non-ABI) declarations shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_geom.h"

namespace fa {

// Status codes written by kernels into the device status word.
enum DeviceStatus { DEV_OK = 0, DEV_TIMEOUT = 1 };

// Parameters of the tensor-core kernel (passed as one __grid_constant__).
// Memory layouts of Q, K, V and O.
enum Layout { LAYOUT_BHND = 0, LAYOUT_BNHD = 1 };

// Row offset (in elements / D) of query or key row i of head h, batch b.
FA_HD long long row_index(int layout, int b, int h, int i, int H, int N) {
    return layout == LAYOUT_BHND ? ((long long)b * H + h) * N + i : ((long long)b * N + i) * H + h;
}

struct TcParams {
    CUtensorMap tm_q;   // 5-D maps {64 columns, rows, D/64 chunks, heads, batch} of either layout,
    CUtensorMap tm_k;   // 16-bit, 128-byte swizzle; one box is a whole tile (all chunks of
    CUtensorMap tm_v;   // 128 rows; the pair kernel's K and V halves: see launch_tc_pair)
    CUtensorMap tm_o;   // O with Q's map shape, box 64 columns x 32 rows: each softmax warp of
                        // the one-CTA kernel stores its rows of 16-bit O through it (unused
                        // for fp32 O)
    void* o;            // O in Q's layout, 16-bit or fp32 (o_f32)
    float* lse;         // [B, H, N] or null
    Geom g;
    int BH;
    int H;              // query heads
    int G;              // query heads per K/V head (H / H_kv)
    int layout;
    int n_units;
    int order;
    float scale_log2;   // scale * log2(e)
    int o_f32;
    unsigned long long wait_limit_ns;
    int* status;        // device status word
    // Rotary embedding of Q applied in the kernel (rope != 0): query row i
    // sits at position rope_pos0 + i of the fp32 [n_pos, D/2] cos/sin tables.
    const float* rope_cos;
    const float* rope_sin;
    int rope;
    int rope_style;     // RopeStyle
    int rope_pos0;
};

struct SimtParams {
    const float* q;
    const float* k;
    const float* v;
    float* o;
    float* lse;
    Geom g;
    int BH;
    int D;
    float scale;
    int H = 1;          // query heads
    int G = 1;          // query heads per K/V head
    int layout = LAYOUT_BHND;
};

// Split-K decode: a few queries (the last Nq positions) against an Nk-key cache.
constexpr int kDecodeMaxQ = 16;   // queries per (b, h) the decode kernels accept
constexpr int kDecodeMinKeysPerSplit = 256;

struct DecodeParams {
    const void* q;      // [B, H, Nq, D] or [B, Nq, H, D]
    const void* k;      // [B, H_kv, Nk, D] or [B, Nk, H_kv, D]
    const void* v;
    void* o;            // Q's shape and layout
    float* lse;         // [B, H, Nq] or null
    float* part_o;      // [B*H_kv, n_splits, G*Nq, D] fp32 partial outputs (n_splits > 1)
    float* part_lse;    // [B*H_kv, n_splits, G*Nq]
    long long BH;       // B * H_kv: one CTA group per (batch, K/V head)
    int Nq;
    int Nk;
    int D;
    float scale_log2;
    int win_l;          // -1 = unbounded; positions: query i sits at key Nk - Nq + i
    int win_r;
    int n_splits;
    int chunk;          // keys per split (multiple of 4)
    int G = 1;          // query heads per K/V head; a CTA takes all G * Nq query rows of its K/V head
    int Hkv = 1;        // K/V heads (read only for [B, N, H, D])
    int layout = LAYOUT_BHND;
    // Paged cache (block_table != null): k, v are [num_pages, page_size, Hkv, D];
    // position j of sequence b is row j % page_size of page block_table[b][j / page_size];
    // sequence b has seq_lens[b] positions (clamped to [0, Nk]); Nk is the longest.
    const int* block_table = nullptr;
    const int* seq_lens = nullptr;
    int page_shift = 0;  // log2(page_size)
    int max_pages = 0;   // row stride of block_table
    int num_pages = 0;   // page indices are clamped to [0, num_pages)
};

// Split count and key chunk for a decode problem (n_req <= 0: choose).
//
// With ctas_per_sm > 0 (the decode kernel's resident CTAs per SM, so one wave
// is ctas_per_sm * sms CTAs) the choice is the split count, at most two
// waves' worth, whose last wave is fullest; ties go to fewer splits.  With
// one_wave_first (the tensor-core kernel, whose CTAs carry a larger fixed
// cost: Q fragments, ring fill, merge) the split count whose single wave is
// fullest wins instead whenever that wave is at least kDecodeOneWaveFill full:
// every CTA of a second wave pays the fixed cost again, and for that kernel a
// wave 84% full measured faster than two waves 98% full, while the one-row
// kernel, with more and lighter CTAs, measured faster with two full waves.
// With ctas_per_sm == 0 it is the older rule of about eight CTAs per SM.
constexpr double kDecodeOneWaveFill = 0.75;
inline void decode_plan(long long BH, int Nk, int sms, int n_req, int* n_splits, int* chunk, int ctas_per_sm = 0,
                        bool one_wave_first = false) {
    const long long cap = (Nk + kDecodeMinKeysPerSplit - 1) / kDecodeMinKeysPerSplit;
    long long s = n_req > 0 ? n_req : (8LL * sms + BH - 1) / BH;
    if (n_req <= 0 && ctas_per_sm > 0) {
        const long long slots = (long long)ctas_per_sm * sms;
        long long best = 1;
        double best_eff = -1.0;
        for (long long t = 1; one_wave_first && t <= cap && BH * t <= slots; ++t) {
            const double eff = (double)(BH * t) / (double)slots;
            if (eff > best_eff + 1e-9) {
                best_eff = eff;
                best = t;
            }
        }
        if (best_eff < kDecodeOneWaveFill) {
            best = 1;
            best_eff = -1.0;
            for (long long t = 1; t <= cap && BH * t <= 2 * slots; ++t) {
                const long long waves = (BH * t + slots - 1) / slots;
                const double eff = (double)(BH * t) / (double)(waves * slots);
                if (eff > best_eff + 1e-9) {
                    best_eff = eff;
                    best = t;
                }
            }
        }
        s = best;
    }
    if (n_req <= 0 && s > cap) s = cap;
    if (s > Nk) s = Nk;
    if (s > 1024) s = 1024;
    if (s < 1) s = 1;
    long long c = (Nk + s - 1) / s;
    c = (c + 3) / 4 * 4;
    *chunk = (int)c;
    *n_splits = (int)((Nk + c - 1) / c);
}

// Bytes of fp32 partials a decode with n_splits splits needs (0 for one split).
inline unsigned long long decode_workspace_bytes(long long BH, int Nq, int D, int n_splits) {
    if (n_splits <= 1) return 0;
    const unsigned long long rows = (unsigned long long)BH * n_splits * Nq;
    const unsigned long long o_bytes = (rows * D * 4 + 255) / 256 * 256;
    return o_bytes + (rows * 4 + 255) / 256 * 256;
}

// Backward pass (dQ, dK, dV).  Rows are padded to a whole number of 128-row
// tiles in the per-row vectors so the kernels copy them without tail checks.
struct BwdParams {
    CUtensorMap tm_q;   // whole-tile 5-D maps as in TcParams: Q and dO with H heads,
    CUtensorMap tm_k;   // K and V with H_kv heads
    CUtensorMap tm_v;
    CUtensorMap tm_do;
    const void* q;      // Q and dO as plain pointers too (Q's shape and layout): the dQ
    const void* d_o;    // kernel reads its rows of them straight into TMEM
    void* dq;           // Q's shape and layout, input element type
    void* dk;           // K's shape and layout
    void* dv;
    const float* lse2;  // [B*H, Npad]: LSE * log2(e); +inf where a row sees no key and on padding
    const float* dsum;  // [B*H, Npad]: rowsum(dO * O); 0 on padding
    Geom g;
    int H;              // query heads
    int G;              // query heads per K/V head
    int Hkv;
    int layout;
    int Npad;           // rows rounded up to kTileM
    int n_tiles;        // Npad / kTileM
    float scale;
    float scale_log2;
    unsigned long long wait_limit_ns;
    int* status;
};

// Rotary position embedding of Q and K (one pass in HBM before attention).
enum RopeStyle { ROPE_HALF = 0, ROPE_INTERLEAVED = 1 };

struct RopeParams {
    const void* x[2];   // Q, K (null: that tensor is skipped)
    void* y[2];         // rotated outputs (may equal x)
    int n[2];           // rows per (b, h): Nq, Nk
    int heads[2];       // H, H_kv
    int pos0[2];        // position of row 0
    const float* cos;   // [n_pos, D/2]
    const float* sin;
    int B;
    int D;              // multiple of 16
    int style;
    int layout;
};

// Records `e` as this host thread's last CUDA error (the text
// fa_last_cuda_error returns) and returns FA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Launchers (return the CUDA error of the launch, if any).
cudaError_t launch_decode(const DecodeParams& p, int dtype_code, cudaStream_t s);
// Resident CTAs per SM of the decode kernel that `rows` query rows per (b, K/V
// head) select, at head dimension D (0 if the runtime cannot say).
int decode_ctas_per_sm(int rows, int D);
cudaError_t launch_tc(const TcParams& p, int D, bool bf16, bool pos_scale, int grid, cudaStream_t s);
// The CTA-pair forward (D = 128): `clusters` persistent 2-CTA clusters over
// p.n_units 256-row units; tm_k's box is 64 keys x 128 columns (one CTA's
// half of a K tile), tm_v's 128 keys x 64 columns (half of a V tile).
cudaError_t launch_tc_pair(const TcParams& p, bool bf16, bool pos_scale, int clusters, cudaStream_t s);
cudaError_t launch_simt_f32(const SimtParams& p, cudaStream_t s);
cudaError_t launch_bwd_pre(const void* o, const void* d_o, const float* lse, float* lse2, float* dsum, int B,
                           int H, int N, int Npad, int D, int layout, int dtype_code, int sms, cudaStream_t s);
cudaError_t launch_bwd(const BwdParams& p, int B, int D, bool bf16, cudaStream_t s);
cudaError_t launch_rope(const RopeParams& p, int dtype_code, int sms, cudaStream_t s);
cudaError_t launch_rope_tables(float* cos_tab, float* sin_tab, int n_pos, int D, double base, int sms,
                               cudaStream_t s);
cudaError_t launch_selftest_timeout(int* status, unsigned long long limit_ns, cudaStream_t s);

}  // namespace fa
