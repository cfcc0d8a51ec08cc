// C ABI of libfa: argument validation, mask normalisation, TMA descriptor
// encoding, kernel dispatch, device status word.
//
// The two-phase "workspace size + execute" call of the ops-transformer
// walk-through (section "the complete operator in ops-transformer", aclnn
// FlashAttention call) is not needed here: the kernels use no workspace, so
// one call enqueues the whole forward on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

thread_local char g_last_cuda_err[256] = "no error";
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_fwd_kernel{FA_FWD_AUTO};

__device__ int g_status_word;

struct DeviceInfo {
    std::once_flag once;
    int sms = 0;
    int* status = nullptr;
    cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;

int cuda_fail(cudaError_t e) {
    std::snprintf(g_last_cuda_err, sizeof(g_last_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return FA_ERR_CUDA;
}

int cuda_fail_msg(const char* msg) {
    std::snprintf(g_last_cuda_err, sizeof(g_last_cuda_err), "%s", msg);
    return FA_ERR_CUDA;
}

// Per-device facts, resolved once with that device current.
int device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail_msg("device ordinal out of range");
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) d.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
    });
    if (d.err != cudaSuccess) return cuda_fail(d.err);
    *out = &d;
    return FA_OK;
}

int encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess) g_encode_err = cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (g_encode_err != cudaSuccess || !g_encode) return cuda_fail(g_encode_err);
    *fn = g_encode;
    return FA_OK;
}

// 5-D view {64 columns, rows, D / 64 column chunks, heads, batch} of a 16-bit
// [B, H, N, D] or [B, N, H, D] tensor, so that one TMA instruction moves a
// whole box of `box_rows` rows x (64 * box_chunks) columns into shared memory
// as box_chunks blocks of box_rows x 128 bytes (128-byte swizzle), the
// layout the tensor-core descriptors read.  Whole tiles per instruction
// matter: a TMA load costs about the same fixed time per instruction up to
// at least 32 KiB, so two 16 KiB boxes take twice as long as one 32 KiB box.
int make_tile_map(CUtensorMap* m, const void* base, bool bf16, int layout, int B, int Hx, int N, int D,
                  int box_rows, int box_chunks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = encoder(&enc);
    if (rc != FA_OK) return rc;
    const cuuint64_t e = 2;
    const cuuint64_t row = layout == fa::LAYOUT_BHND ? (cuuint64_t)D * e : (cuuint64_t)Hx * D * e;
    const cuuint64_t head = layout == fa::LAYOUT_BHND ? (cuuint64_t)N * D * e : (cuuint64_t)D * e;
    cuuint64_t dims[5] = {64, (cuuint64_t)N, (cuuint64_t)(D / 64), (cuuint64_t)Hx, (cuuint64_t)B};
    cuuint64_t strides[4] = {row, 128, head, (cuuint64_t)Hx * N * D * e};
    cuuint32_t box[5] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_err, sizeof(g_last_cuda_err), "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Normalised mask: causal == window(-1, 0), none == window(-1, -1).
int normalise_mask(int mask_kind, int win_l, int win_r, int N, fa::Geom* g) {
    g->N = N;
    switch (mask_kind) {
        case FA_MASK_NONE: g->win_l = -1; g->win_r = -1; return FA_OK;
        case FA_MASK_CAUSAL: g->win_l = -1; g->win_r = 0; return FA_OK;
        case FA_MASK_WINDOW:
            if (win_l < -1 || win_r < -1) return FA_ERR_ARG;
            g->win_l = win_l;
            g->win_r = win_r;
            return FA_OK;
        default: return FA_ERR_ARG;
    }
}

int validate(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H, int N,
             int D, float scale, int mask_kind, int win_l, int win_r, int dtype, int o_dtype, fa::Geom* g) {
    if (!q || !k || !v || !o) return FA_ERR_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || D <= 0) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    int rc = normalise_mask(mask_kind, win_l, win_r, N, g);
    if (rc != FA_OK) return rc;
    const long long bh = (long long)B * H;
    if (bh > 0x7fffffffLL) return FA_ERR_ARG;
    const double elems = (double)bh * N * D;
    if (elems > 4.0e18) return FA_ERR_ARG;
    switch (dtype) {
        case FA_F16:
        case FA_BF16:
            if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
            if (o_dtype != dtype && o_dtype != FA_F32) return FA_ERR_UNSUPPORTED;
            break;
        case FA_F32:
            if (D > 128) return FA_ERR_UNSUPPORTED;
            if (o_dtype != FA_F32) return FA_ERR_UNSUPPORTED;
            break;
        default: return FA_ERR_UNSUPPORTED;
    }
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return FA_ERR_ALIGN;
    if (lse && !aligned(lse, 4)) return FA_ERR_ALIGN;
    return FA_OK;
}

}  // namespace

namespace fa {
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
}  // namespace fa

namespace {

// Rotary embedding of Q inside the forward (null tables: none).
struct RopeQ {
    const float* cos = nullptr;
    const float* sin = nullptr;
    int style = 0;
    int pos0 = 0;
};

int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
               int D, float scale, int mask_kind, int win_l, int win_r, int dtype, int o_dtype, int layout,
               const RopeQ& rope, void* stream) {
    fa::Geom g;
    int rc = validate(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, &g);
    if (rc != FA_OK) return rc;
    if (H_kv <= 0 || H_kv > H || H % H_kv != 0) return FA_ERR_ARG;
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_ARG;
    if (rope.cos && dtype == FA_F32) return FA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    if ((rc = device_info(&dev)) != FA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int BH = B * H;

    if (dtype == FA_F32) {
        fa::SimtParams p;
        p.q = static_cast<const float*>(q);
        p.k = static_cast<const float*>(k);
        p.v = static_cast<const float*>(v);
        p.o = static_cast<float*>(o);
        p.lse = lse;
        p.g = g;
        p.BH = BH;
        p.D = D;
        p.scale = scale;
        p.H = H;
        p.G = H / H_kv;
        p.layout = layout;
        cudaError_t e = fa::launch_simt_f32(p, s);
        return e == cudaSuccess ? FA_OK : cuda_fail(e);
    }

    const bool bf16 = dtype == FA_BF16;
    // The one-CTA kernel unless the caller asked for the CTA pair (D = 128).
    const int sel = g_fwd_kernel.load(std::memory_order_relaxed);
    const bool pair = D == 128 && sel == FA_FWD_CTA_PAIR && dev->sms >= 2;
    fa::TcParams p;
    std::memset(&p, 0, sizeof(p));
    // Whole tiles per TMA instruction: Q and K/V tiles of 128 rows x D in the
    // one-CTA kernel; in the pair kernel each CTA's K half is 64 keys x D and
    // its V half 128 keys x 64 columns (one chunk).
    const int chunks = D / 64;
    if ((rc = make_tile_map(&p.tm_q, q, bf16, layout, B, H, N, D, fa::kTileM, chunks)) != FA_OK) return rc;
    if ((rc = make_tile_map(&p.tm_k, k, bf16, layout, B, H_kv, N, D, pair ? fa::kTileN / 2 : fa::kTileN, chunks)) !=
        FA_OK)
        return rc;
    if ((rc = make_tile_map(&p.tm_v, v, bf16, layout, B, H_kv, N, D, fa::kTileN, pair ? 1 : chunks)) != FA_OK)
        return rc;
    // 16-bit O leaves the one-CTA kernel by TMA stores of 64-column boxes
    if (o_dtype != FA_F32 && (rc = make_tile_map(&p.tm_o, o, bf16, layout, B, H, N, D, 32, 1)) != FA_OK)
        return rc;
    p.o = o;
    p.lse = lse;
    p.g = g;
    p.BH = BH;
    p.H = H;
    p.G = H / H_kv;
    p.layout = layout;
    const long long units = (long long)BH * fa::n_pairs_for(N);  // 256 query rows each (both kernels)
    if (units > 0x7fffffffLL) return FA_ERR_ARG;
    p.n_units = (int)units;
    p.order = fa::unit_order_for(g);
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.o_f32 = o_dtype == FA_F32 ? 1 : 0;
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.status = dev->status;
    if (rope.cos) {
        p.rope = 1;
        p.rope_cos = rope.cos;
        p.rope_sin = rope.sin;
        p.rope_style = rope.style;
        p.rope_pos0 = rope.pos0;
    }
    cudaError_t e;
    if (pair) {
        const int clusters = p.n_units < dev->sms / 2 ? p.n_units : dev->sms / 2;
        e = fa::launch_tc_pair(p, bf16, scale > 0.f, clusters, s);
    } else {
        // One CTA per unit: the CTAs that run take the units of those that
        // have not started yet (cluster launch control), so as many run as fit.
        e = fa::launch_tc(p, D, bf16, scale > 0.f, p.n_units, s);
    }
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
               int D, float scale, int mask_kind, int win_l, int win_r, int dtype, int o_dtype, int layout,
               void* stream) {
    return fwd_common(q, k, v, o, lse, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, layout,
                      RopeQ{}, stream);
}

int fa_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, const float* cos_tab,
                const float* sin_tab, int n_pos, int q_pos0, int style, int B, int H, int H_kv, int N, int D,
                float scale, int mask_kind, int win_l, int win_r, int dtype, int o_dtype, int layout, void* stream) {
    if (!cos_tab || !sin_tab || n_pos <= 0 || q_pos0 < 0) return FA_ERR_ARG;
    if (N > 0 && (long long)q_pos0 + N > n_pos) return FA_ERR_ARG;
    if (style != fa::ROPE_HALF && style != fa::ROPE_INTERLEAVED) return FA_ERR_ARG;
    if (!aligned(cos_tab, 16) || !aligned(sin_tab, 16)) return FA_ERR_ALIGN;
    RopeQ r;
    r.cos = cos_tab;
    r.sin = sin_tab;
    r.style = style;
    r.pos0 = q_pos0;
    return fwd_common(q, k, v, o, lse, B, H, H_kv, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, layout, r,
                      stream);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
              float scale, int mask_kind, int win_l, int win_r, int dtype, int o_dtype, void* stream) {
    return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, D, scale, mask_kind, win_l, win_r, dtype, o_dtype, FA_LAYOUT_BHND,
                      stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D, float scale,
           int mask_kind, int win_l, int win_r, int dtype, void* stream) {
    return fa_fwd_ex(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, dtype, dtype, stream);
}

int fa_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
               float scale, int mask_kind, int win_l, int win_r, void* stream) {
    return fa_fwd(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, FA_F16, stream);
}

int fa_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                float scale, int mask_kind, int win_l, int win_r, void* stream) {
    return fa_fwd(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, FA_BF16, stream);
}

int fa_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
               float scale, int mask_kind, int win_l, int win_r, void* stream) {
    return fa_fwd(q, k, v, o, lse, B, H, N, D, scale, mask_kind, win_l, win_r, FA_F32, stream);
}

int fa_device_status(void* stream) {
    DeviceInfo* dev;
    int rc = device_info(&dev);
    if (rc != FA_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cuda_fail(e);
        return FA_ERR_DEVICE;
    }
    int word = 0;
    e = cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return FA_ERR_DEVICE;
    }
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cuda_fail(e);
            return FA_ERR_DEVICE;
        }
        return FA_ERR_TIMEOUT;
    }
    return FA_OK;
}

int fa_select_fwd_kernel(int which) {
    if (which != FA_FWD_AUTO && which != FA_FWD_ONE_CTA && which != FA_FWD_CTA_PAIR) return FA_ERR_ARG;
    return g_fwd_kernel.exchange(which);
}

unsigned long long fa_set_wait_limit_ns(unsigned long long ns) {
    if (ns < FA_MIN_WAIT_LIMIT_NS) ns = FA_MIN_WAIT_LIMIT_NS;
    return g_wait_limit_ns.exchange(ns);
}

int fa_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
    DeviceInfo* dev;
    int rc = device_info(&dev);
    if (rc != FA_OK) return rc;
    cudaError_t e = fa::launch_selftest_timeout(dev->status, limit_ns, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_decode_plan_gqa(int B, int H, int H_kv, int Nq, int Nk, int D, int n_splits, int* n_splits_out,
                       unsigned long long* workspace_bytes) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return FA_ERR_ARG;
    if (H_kv <= 0 || H_kv > H || H % H_kv != 0) return FA_ERR_ARG;
    DeviceInfo* dev;
    int rc = device_info(&dev);
    if (rc != FA_OK) return rc;
    int ns, chunk;
    const long long groups = (long long)B * H_kv;
    fa::decode_plan(groups, Nk, dev->sms, n_splits, &ns, &chunk, fa::decode_ctas_per_sm((H / H_kv) * Nq, D),
                    (H / H_kv) * Nq > 1);
    if (n_splits_out) *n_splits_out = ns;
    if (workspace_bytes) *workspace_bytes = fa::decode_workspace_bytes(groups, (H / H_kv) * Nq, D, ns);
    return FA_OK;
}

int fa_decode_plan(int B, int H, int Nq, int Nk, int D, int n_splits, int* n_splits_out,
                   unsigned long long* workspace_bytes) {
    return fa_decode_plan_gqa(B, H, H, Nq, Nk, D, n_splits, n_splits_out, workspace_bytes);
}

int fa_decode_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int Nq,
                  int Nk, int D, float scale, int mask_kind, int win_l, int win_r, int dtype, int layout,
                  int n_splits, void* workspace, unsigned long long workspace_bytes, void* stream) {
    if (!q || !k || !v || !o) return FA_ERR_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || D <= 0 || Nq > Nk) return FA_ERR_ARG;
    if (H_kv <= 0 || H_kv > H || H % H_kv != 0) return FA_ERR_ARG;
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    fa::Geom g;
    int rc = normalise_mask(mask_kind, win_l, win_r, Nk, &g);
    if (rc != FA_OK) return rc;
    if ((long long)B * H > 0x7fffffffLL) return FA_ERR_ARG;
    const int G = H / H_kv;
    if (dtype < FA_F16 || dtype > FA_F32 || (D != 64 && D != 128) || (long long)G * Nq > fa::kDecodeMaxQ)
        return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return FA_ERR_ALIGN;
    if (lse && !aligned(lse, 4)) return FA_ERR_ALIGN;
    DeviceInfo* dev;
    if ((rc = device_info(&dev)) != FA_OK) return rc;
    fa::DecodeParams p{};
    p.BH = (long long)B * H_kv;
    p.G = G;
    p.Hkv = H_kv;
    p.layout = layout;
    fa::decode_plan(p.BH, Nk, dev->sms, n_splits, &p.n_splits, &p.chunk, fa::decode_ctas_per_sm(G * Nq, D),
                    G * Nq > 1);
    const unsigned long long need = fa::decode_workspace_bytes(p.BH, G * Nq, D, p.n_splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FA_ERR_ARG;
        if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
        p.part_o = static_cast<float*>(workspace);
        p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              ((unsigned long long)p.BH * p.n_splits * G * Nq * D * 4 + 255) / 256 * 256);
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
    p.win_l = g.win_l;
    p.win_r = g.win_r;
    cudaError_t e = fa::launch_decode(p, dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                    const int* seq_lens, void* o, float* lse, int B, int H, int H_kv, int Nq, int max_seq_len,
                    int page_size, int max_pages, int num_pages, int D, float scale, int mask_kind, int win_l,
                    int win_r, int dtype, int layout, int n_splits, void* workspace,
                    unsigned long long workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return FA_ERR_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || D <= 0 || max_seq_len <= 0 || max_pages <= 0 || num_pages <= 0)
        return FA_ERR_ARG;
    if (page_size <= 0 || (page_size & (page_size - 1)) != 0) return FA_ERR_ARG;
    if ((long long)max_pages * page_size < max_seq_len) return FA_ERR_ARG;
    if ((long long)num_pages * page_size * H_kv * D > (1LL << 46)) return FA_ERR_ARG;
    if (H_kv <= 0 || H_kv > H || H % H_kv != 0) return FA_ERR_ARG;
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    fa::Geom g;
    int rc = normalise_mask(mask_kind, win_l, win_r, max_seq_len, &g);
    if (rc != FA_OK) return rc;
    if ((long long)B * H > 0x7fffffffLL) return FA_ERR_ARG;
    const int G = H / H_kv;
    if (dtype < FA_F16 || dtype > FA_F32 || (D != 64 && D != 128) || (long long)G * Nq > fa::kDecodeMaxQ)
        return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16)) return FA_ERR_ALIGN;
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4))) return FA_ERR_ALIGN;
    DeviceInfo* dev;
    if ((rc = device_info(&dev)) != FA_OK) return rc;
    fa::DecodeParams p{};
    p.BH = (long long)B * H_kv;
    p.G = G;
    p.Hkv = H_kv;
    p.layout = layout;
    fa::decode_plan(p.BH, max_seq_len, dev->sms, n_splits, &p.n_splits, &p.chunk,
                    fa::decode_ctas_per_sm(G * Nq, D), G * Nq > 1);
    const unsigned long long need = fa::decode_workspace_bytes(p.BH, G * Nq, D, p.n_splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FA_ERR_ARG;
        if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
        p.part_o = static_cast<float*>(workspace);
        p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              ((unsigned long long)p.BH * p.n_splits * G * Nq * D * 4 + 255) / 256 * 256);
    }
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.o = o;
    p.lse = lse;
    p.Nq = Nq;
    p.Nk = max_seq_len;
    p.D = D;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.win_l = g.win_l;
    p.win_r = g.win_r;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    int shift = 0;
    while ((1 << shift) < page_size) ++shift;
    p.page_shift = shift;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    cudaError_t e = fa::launch_decode(p, dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int D,
              float scale, int mask_kind, int win_l, int win_r, int dtype, int n_splits, void* workspace,
              unsigned long long workspace_bytes, void* stream) {
    return fa_decode_gqa(q, k, v, o, lse, B, H, H, Nq, Nk, D, scale, mask_kind, win_l, win_r, dtype, FA_LAYOUT_BHND,
                         n_splits, workspace, workspace_bytes, stream);
}

namespace {
// Padded rows and the workspace split of the backward pass: LSE*log2(e) then
// Dsum, each [B*H, Npad] fp32 on a 256-byte boundary.
long long bwd_npad(int N) { return ((long long)N + fa::kTileM - 1) / fa::kTileM * fa::kTileM; }
unsigned long long bwd_vec_bytes(int B, int H, int N) {
    return ((unsigned long long)B * H * bwd_npad(N) * 4 + 255) / 256 * 256;
}
}  // namespace

int fa_bwd_workspace_bytes(int B, int H, int N, unsigned long long* bytes) {
    if (B <= 0 || H <= 0 || N <= 0 || !bytes) return FA_ERR_ARG;
    *bytes = 2 * bwd_vec_bytes(B, H, N);
    return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int H_kv, int N, int D, float scale, int mask_kind, int win_l,
           int win_r, int dtype, int layout, void* workspace, unsigned long long workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !d_o || !lse || !dq || !dk || !dv) return FA_ERR_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || D <= 0) return FA_ERR_ARG;
    if (H_kv <= 0 || H_kv > H || H % H_kv != 0) return FA_ERR_ARG;
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    fa::Geom g;
    int rc = normalise_mask(mask_kind, win_l, win_r, N, &g);
    if (rc != FA_OK) return rc;
    const long long n_tiles = bwd_npad(N) / fa::kTileM;
    if ((long long)B * H * n_tiles > 0x7fffffffLL) return FA_ERR_ARG;
    if ((dtype != FA_F16 && dtype != FA_BF16) || (D != 64 && D != 128)) return FA_ERR_UNSUPPORTED;
    const void* p16[] = {q, k, v, o, d_o, dq, dk, dv};
    for (const void* ptr : p16)
        if (!aligned(ptr, 16)) return FA_ERR_ALIGN;
    if (!aligned(lse, 4)) return FA_ERR_ALIGN;
    const unsigned long long vb = bwd_vec_bytes(B, H, N);
    if (!workspace || workspace_bytes < 2 * vb) return FA_ERR_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
    DeviceInfo* dev;
    if ((rc = device_info(&dev)) != FA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf16 = dtype == FA_BF16;
    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int chunks = D / 64;
    if ((rc = make_tile_map(&p.tm_q, q, bf16, layout, B, H, N, D, fa::kTileM, chunks)) != FA_OK) return rc;
    if ((rc = make_tile_map(&p.tm_k, k, bf16, layout, B, H_kv, N, D, fa::kTileN, chunks)) != FA_OK) return rc;
    if ((rc = make_tile_map(&p.tm_v, v, bf16, layout, B, H_kv, N, D, fa::kTileN, chunks)) != FA_OK) return rc;
    if ((rc = make_tile_map(&p.tm_do, d_o, bf16, layout, B, H, N, D, fa::kTileM, chunks)) != FA_OK) return rc;
    float* lse2 = static_cast<float*>(workspace);
    float* dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + vb);
    p.q = q;
    p.d_o = d_o;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.lse2 = lse2;
    p.dsum = dsum;
    p.g = g;
    p.H = H;
    p.G = H / H_kv;
    p.Hkv = H_kv;
    p.layout = layout;
    p.Npad = (int)bwd_npad(N);
    p.n_tiles = (int)n_tiles;
    p.scale = scale;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.status = dev->status;
    cudaError_t e = fa::launch_bwd_pre(o, d_o, lse, lse2, dsum, B, H, N, p.Npad, D, layout, dtype, dev->sms, s);
    if (e == cudaSuccess) e = fa::launch_bwd(p, B, D, bf16, s);
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_rope(const void* q, const void* k, void* q_out, void* k_out, const float* cos_tab, const float* sin_tab,
            int B, int H, int H_kv, int Nq, int Nk, int D, int q_pos0, int k_pos0, int n_pos, int style, int dtype,
            int layout, void* stream) {
    if (!q && !k) return FA_ERR_ARG;
    if ((q == nullptr) != (q_out == nullptr) || (k == nullptr) != (k_out == nullptr)) return FA_ERR_ARG;
    if (!cos_tab || !sin_tab) return FA_ERR_ARG;
    if (B <= 0 || D <= 0 || D % 16 != 0 || D > 1024 || n_pos <= 0) return FA_ERR_ARG;
    if (style != fa::ROPE_HALF && style != fa::ROPE_INTERLEAVED) return FA_ERR_ARG;
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_ARG;
    if (q && (H <= 0 || Nq <= 0 || q_pos0 < 0 || (long long)q_pos0 + Nq > n_pos)) return FA_ERR_ARG;
    if (k && (H_kv <= 0 || Nk <= 0 || k_pos0 < 0 || (long long)k_pos0 + Nk > n_pos)) return FA_ERR_ARG;
    if (dtype < FA_F16 || dtype > FA_F32) return FA_ERR_UNSUPPORTED;
    if ((q && (!aligned(q, 16) || !aligned(q_out, 16))) || (k && (!aligned(k, 16) || !aligned(k_out, 16))) ||
        !aligned(cos_tab, 16) || !aligned(sin_tab, 16))
        return FA_ERR_ALIGN;
    DeviceInfo* dev;
    int rc = device_info(&dev);
    if (rc != FA_OK) return rc;
    fa::RopeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x[0] = q;
    p.y[0] = q_out;
    p.n[0] = q ? Nq : 0;
    p.heads[0] = q ? H : 0;
    p.pos0[0] = q_pos0;
    p.x[1] = k;
    p.y[1] = k_out;
    p.n[1] = k ? Nk : 0;
    p.heads[1] = k ? H_kv : 0;
    p.pos0[1] = k_pos0;
    p.cos = cos_tab;
    p.sin = sin_tab;
    p.B = B;
    p.D = D;
    p.style = style;
    p.layout = layout;
    cudaError_t e = fa::launch_rope(p, dtype, dev->sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_rope_tables(float* cos_tab, float* sin_tab, int n_pos, int D, double base, void* stream) {
    if (!cos_tab || !sin_tab || n_pos <= 0 || D <= 0 || D % 2 != 0 || D > 1024) return FA_ERR_ARG;
    if (!(base > 0.0) || !std::isfinite(base)) return FA_ERR_ARG;
    if (!aligned(cos_tab, 16) || !aligned(sin_tab, 16)) return FA_ERR_ALIGN;
    DeviceInfo* dev;
    int rc = device_info(&dev);
    if (rc != FA_OK) return rc;
    cudaError_t e = fa::launch_rope_tables(cos_tab, sin_tab, n_pos, D, base, dev->sms,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_plan_units(int B, int H, int N, int mask_kind, int win_l, int win_r, int* out, int cap) {
    if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_ARG;
    fa::Geom g;
    int rc = normalise_mask(mask_kind, win_l, win_r, N, &g);
    if (rc != FA_OK) return rc;
    const long long units = (long long)B * H * fa::n_pairs_for(N);
    if (units > 0x7fffffffLL) return FA_ERR_ARG;
    const int order = fa::unit_order_for(g);
    for (int u = 0; out && u < cap && u < units; ++u) {
        fa::Unit un = fa::make_unit(g, B * H, order, u);
        int* r = out + 6 * u;
        r[0] = un.bh;
        r[1] = un.q0;
        r[2] = un.lo[0];
        r[3] = un.hi[0];
        r[4] = un.lo[1];
        r[5] = un.hi[1];
    }
    return (int)units;
}

int fa_tile_needs_mask(int N, int mask_kind, int win_l, int win_r, int r0, int j) {
    fa::Geom g;
    if (normalise_mask(mask_kind, win_l, win_r, N, &g) != FA_OK) return FA_ERR_ARG;
    return fa::tile_needs_mask(g, r0, j) ? 1 : 0;
}

int fa_geom_needs_masks(int N, int mask_kind, int win_l, int win_r) {
    fa::Geom g;
    if (normalise_mask(mask_kind, win_l, win_r, N, &g) != FA_OK) return FA_ERR_ARG;
    return fa::geom_needs_masks(g) ? 1 : 0;
}

const char* fa_strerror(int code) {
    switch (code) {
        case FA_OK: return "ok";
        case FA_ERR_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported dtype or head dimension";
        case FA_ERR_ALIGN: return "pointer not aligned (16 bytes for q/k/v/o, 4 for lse)";
        case FA_ERR_CUDA: return "CUDA error (see fa_last_cuda_error)";
        case FA_ERR_TIMEOUT: return "a kernel wait timed out";
        case FA_ERR_DEVICE: return "device error reported by the stream";
        case FA_ERR_SCRATCH: return "partial results exceed the library's fixed scratch array";
        default: return "unknown error code";
    }
}

const char* fa_last_cuda_error(void) { return g_last_cuda_err; }

int fa_version(void) { return 100; }

}  // extern "C"
