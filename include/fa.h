/*
 * libfa -- fused attention forward for NVIDIA GB300 (sm_103a), C ABI.
 *
 * Computes, for every batch b and head h,
 *
 *     S   = scale * Q K^T              (scores, never written to memory)
 *     S_ij = -inf where the mask hides key j from query i
 *     O   = softmax_rows(S) V
 *     LSE_i = ln sum_j exp(S_ij)       (natural log, fp32)
 *
 * Definition: "Ascend C advanced practice: high-performance
 * FlashAttention-2-style tile-level fused attention", section 1.1 (the MHA
 * definition) and section 1.2 (the online-softmax identity the kernels use);
 * the causal rule follows its section 4.2 kernel (a key after the query is
 * masked); the (window_left, window_right) sliding window follows "FlashAttention
 * under the catlass template", section "Usage" (full / causal / window masks
 * handled by one kernel), read as the inclusive band i - win_l <= j <= i + win_r.
 *
 * Layout: Q, K, V and O are contiguous [B, H, N, D] row-major tensors (D is
 * the fastest axis), as in the ops-transformer walk-through's aclnn call
 * ({B, H, S, D} ND tensors).  LSE is a contiguous [B, H, N] fp32 tensor.
 *
 * Ownership: every pointer is caller-owned CUDA device memory; the library
 * allocates nothing and keeps no reference after the kernel finishes (the
 * decode and backward entry points take a caller workspace sized by their
 * planning calls).  Pointers must be 16-byte aligned.  O must not alias Q, K
 * or V.  The later sections declare the decode, layout / grouped-head,
 * backward and rotary-embedding entry points, each with its own layouts.
 *
 * Asynchrony: a return of FA_OK means the work was enqueued on `stream`
 * (a cudaStream_t, or 0 for the legacy default stream).  Kernel-side
 * failures (a bounded wait that timed out) are reported through
 * fa_device_status().
 *
 * Thread safety: the entry points may be called from several host threads
 * on different streams.  The only global state is one device status word
 * (see fa_device_status) and a per-device cache of the SM count.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Mask kinds. CAUSAL == WINDOW(-1, 0); NONE == WINDOW(-1, -1). */
enum {
    FA_MASK_NONE = 0,    /* every key visible                                  */
    FA_MASK_CAUSAL = 1,  /* key j visible to query i iff j <= i                */
    FA_MASK_WINDOW = 2   /* visible iff i - win_l <= j <= i + win_r; a bound of
                            -1 means unbounded on that side                    */
};

/* Memory layouts (fa_fwd_gqa).  BHND: contiguous [B, H, N, D].  BNHD:
 * contiguous [B, N, H, D] -- the "[total_tokens, H, D]" per-batch layout of
 * the Ascend C page's section 4.1 parameter struct, i.e. projection outputs
 * used without a transposing copy. */
enum { FA_LAYOUT_BHND = 0, FA_LAYOUT_BNHD = 1 };

/* Element types of Q, K, V (and O unless fa_fwd_ex overrides it). */
enum { FA_F16 = 0, FA_BF16 = 1, FA_F32 = 2 };

/* Return codes. Negative codes mean nothing was launched. */
enum {
    FA_OK = 0,
    FA_ERR_ARG = -1,          /* null pointer, B/H/N <= 0, non-finite scale,
                                 window bound < -1, unknown mask kind, or a
                                 size whose element count overflows 2^62       */
    FA_ERR_UNSUPPORTED = -2,  /* f16/bf16 need D in {64, 128}; f32 needs
                                 1 <= D <= 128; unknown dtype                  */
    FA_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned              */
    FA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed; see
                                 fa_last_cuda_error()                          */
    FA_ERR_TIMEOUT = -5,      /* (fa_device_status) a kernel wait timed out    */
    FA_ERR_DEVICE = -6,       /* (fa_device_status) the stream reported a CUDA
                                 error                                         */
    FA_ERR_SCRATCH = -7       /* (fa_decode_noalloc) the problem's partial
                                 results do not fit the library's fixed
                                 scratch array                                 */
};

/*
 * fa_fwd -- fused attention forward, O and LSE from Q, K, V.
 *
 *   q, k, v   [B, H, N, D] device pointers of element type `dtype`.
 *   o         [B, H, N, D] device pointer, same element type as q.
 *   lse       [B, H, N] fp32 device pointer, or NULL to skip it.
 *   B, H, N   batch, heads, sequence length (queries == keys == N), all >= 1.
 *   D         head dimension (see FA_ERR_UNSUPPORTED).
 *   scale     multiplies Q K^T before masking; any finite value (0 is legal:
 *             every visible key then gets equal weight).
 *   mask_kind FA_MASK_NONE / FA_MASK_CAUSAL / FA_MASK_WINDOW.
 *   win_l, win_r  window bounds (>= -1), read only for FA_MASK_WINDOW.
 *   dtype     FA_F16 / FA_BF16 (tensor-core kernel) or FA_F32 (fp32 FFMA kernel).
 *   stream    cudaStream_t to enqueue on.
 *
 * Accumulation is fp32 throughout; for 16-bit inputs the softmax
 * probabilities are rounded to the input type before the P.V product.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int D, float scale,
           int mask_kind, int win_l, int win_r, int dtype, void* stream);

/* Typed conveniences with exactly the argument list of the method's call:
 * fa_fwd(q,k,v,o,lse,B,H,N,D,scale,mask_kind,win_l,win_r,stream). */
int fa_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int D, float scale,
               int mask_kind, int win_l, int win_r, void* stream);
int fa_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int N, int D, float scale,
                int mask_kind, int win_l, int win_r, void* stream);
int fa_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int D, float scale,
               int mask_kind, int win_l, int win_r, void* stream);

/*
 * fa_fwd_ex -- as fa_fwd, but O is written with element type `o_dtype`
 * (FA_F32 lets a caller see the fp32 accumulator divided by the row sum
 * before any 16-bit output rounding; otherwise o_dtype must equal dtype).
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int D, float scale,
              int mask_kind, int win_l, int win_r, int dtype, int o_dtype,
              void* stream);

/*
 * Decode against a key/value cache (split-K).
 *
 * The KV-cache incremental decode of "FlashAttention extreme optimisation on
 * Ascend NPUs" (optimisation four): Nq new queries (1 <= Nq <= 16, Nq <= Nk)
 * attend to an Nk-entry cache; query i sits at key position Nk - Nq + i, so
 * FA_MASK_CAUSAL lets it see keys 0 .. Nk - Nq + i and FA_MASK_WINDOW applies
 * the same band rule around that position.  The cache is split into chunks
 * handled in parallel; each produces a normalised partial output and its
 * log-sum-exp, merged exactly as LSE = ln sum_s e^{LSE_s},
 * O = sum_s e^{LSE_s - LSE} O_s (the page's running-average merge is replaced
 * by this softmax-correct one).
 *
 * Two-phase call, as in the ops-transformer walk-through's aclnn
 * FlashAttention API (workspace size query, then execute):
 *
 * fa_decode_plan -- for the current device, the number of splits a decode of
 *   this shape uses (n_splits <= 0: chosen from how many CTAs of the decode
 *   kernel this shape takes fit on an SM, as the count of at most two waves
 *   whose last wave is fullest, never more than ceil(Nk / 256); > 0: that
 *   many, capped at Nk) and the workspace it needs in bytes (0 when one split
 *   suffices).  The choice does not depend on the element type, and is fixed
 *   for a device and shape.  Returns FA_OK or FA_ERR_ARG.
 *
 * fa_decode -- q [B, H, Nq, D], k and v [B, H, Nk, D], o [B, H, Nq, D] (element
 *   type dtype: FA_F16, FA_BF16 or FA_F32; D in {64, 128}), lse [B, H, Nq] fp32
 *   or NULL.  `workspace` is caller-owned device memory of at least the size
 *   fa_decode_plan reported for the same n_splits (256-byte aligned; may be
 *   NULL when that size is 0); it holds fp32 partial results and must not be
 *   shared with another call in flight.  Errors: FA_ERR_ARG (null pointer,
 *   Nq > Nk, a size <= 0, non-finite scale, bad mask, workspace missing or too
 *   small), FA_ERR_UNSUPPORTED (Nq > 16, D not 64/128, bad dtype),
 *   FA_ERR_ALIGN (q/k/v/o not 16-byte aligned, workspace not 256-byte
 *   aligned), FA_ERR_CUDA.  Asynchronous on `stream`.
 */
int fa_decode_plan(int B, int H, int Nq, int Nk, int D, int n_splits, int* n_splits_out,
                   unsigned long long* workspace_bytes);
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int Nq, int Nk, int D, float scale,
              int mask_kind, int win_l, int win_r, int dtype,
              int n_splits, void* workspace, unsigned long long workspace_bytes,
              void* stream);

/*
 * fa_decode_plan_gqa / fa_decode_gqa -- decode with grouped K/V heads and a
 * choice of layout.  q and o have H heads, k and v H_kv heads (H a multiple
 * of H_kv; query head h reads K/V head h / (H / H_kv)); `layout` is
 * FA_LAYOUT_BHND (q [B, H, Nq, D], k/v [B, H_kv, Nk, D]) or FA_LAYOUT_BNHD
 * (q [B, Nq, H, D], k/v [B, Nk, H_kv, D]); lse is [B, H, Nq].  One CTA group
 * serves all H / H_kv query heads of a K/V head, so the cache is read once
 * per K/V head; (H / H_kv) * Nq must be at most 16 (FA_ERR_UNSUPPORTED
 * otherwise).  Workspace rules and the other errors as for fa_decode, plus
 * FA_ERR_ARG for a bad H_kv or layout.  fa_decode / fa_decode_plan are these
 * with H_kv == H and FA_LAYOUT_BHND.
 */
int fa_decode_plan_gqa(int B, int H, int H_kv, int Nq, int Nk, int D, int n_splits, int* n_splits_out,
                       unsigned long long* workspace_bytes);
int fa_decode_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int H_kv, int Nq, int Nk, int D, float scale,
                  int mask_kind, int win_l, int win_r, int dtype, int layout,
                  int n_splits, void* workspace, unsigned long long workspace_bytes,
                  void* stream);

/*
 * fa_decode_paged -- fa_decode_gqa against a paged K/V cache.  "Ascend C
 * advanced practice: high-performance FlashAttention-2-style tile-level fused
 * attention", section 9 ("Extensions: integration with RoPE and a paged KV
 * cache"), replaces the K/V block loads with a gather from a paged cache; the
 * page gives no format, so this takes the common one:
 *   k_cache, v_cache: [num_pages, page_size, H_kv, D] (dtype as q);
 *   block_table: int [B, max_pages]; position j of sequence b is row
 *     j % page_size of page block_table[b * max_pages + j / page_size];
 *   seq_lens: int [B]; sequence b has seq_lens[b] cached positions (values
 *     outside [0, max_seq_len] are clamped), and its Nq new queries sit at
 *     positions seq_lens[b] - Nq + i, which set the causal and window masks
 *     (a query whose position is negative sees no key: O = 0, LSE = -inf).
 * q, o and lse as in fa_decode_gqa (`layout` applies to q and o only).
 * block_table and seq_lens are device memory the library only reads; a
 * page index outside [0, num_pages) is clamped, so a bad table gives wrong
 * values, never an out-of-bounds read.  page_size must be a power of two
 * with max_pages * page_size >= max_seq_len.  The split plan and workspace are
 * fa_decode_plan_gqa(B, H, H_kv, Nq, max_seq_len, D, n_splits); splits past a
 * sequence's length contribute nothing.  Errors as for fa_decode_gqa, plus
 * FA_ERR_ARG for the page arguments and FA_ERR_ALIGN for a block table or
 * length array not 4-byte aligned.
 */
int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                    const int* seq_lens, void* o, float* lse,
                    int B, int H, int H_kv, int Nq, int max_seq_len, int page_size, int max_pages, int num_pages,
                    int D, float scale, int mask_kind, int win_l, int win_r, int dtype, int layout,
                    int n_splits, void* workspace, unsigned long long workspace_bytes, void* stream);

/*
 * fa_decode_noalloc -- fa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for code that
 * must not call cudaMalloc / cudaFree (or any allocating routine) where it
 * runs: inside an allocator or memory-pool callback, in a runtime that owns all
 * device memory through its own pool, or in a plugin that is handed only its
 * input and output buffers.  It computes what fa_decode computes, with the same
 * arguments minus the workspace: the split-K partial results go to a fixed
 * 16 MiB array compiled into the library (fa_decode_noalloc_scratch_bytes()),
 * which every GPU that loads the library holds until the process exits.
 *
 * Returns FA_ERR_SCRATCH when the partials of this shape and split count would
 * not fit (for an explicit n_splits, fa_decode_plan's workspace size above the
 * array's size; a smaller n_splits or a call to fa_decode with a workspace is
 * the way out), otherwise the codes of fa_decode.  It allocates nothing.  With
 * n_splits <= 0 it picks its own split count, about eight CTAs per SM with at
 * most ceil(Nk / 256) splits, which can differ from fa_decode_plan's choice.
 *
 * The first call on a device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture.
 * All calls on a device share the one array, and it keeps the last call's
 * contents: calls whose kernels can overlap on the GPU (different streams
 * without ordering between them) race on it and must be serialised by the
 * caller.  Nothing in it needs clearing: every partial is written before it is
 * read.
 */
int fa_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int Nq, int Nk, int D, float scale,
                      int mask_kind, int win_l, int win_r, int dtype, int n_splits,
                      void* stream);
unsigned long long fa_decode_noalloc_scratch_bytes(void);

/*
 * fa_fwd_gqa -- fa_fwd_ex with grouped K/V heads and a choice of layout.
 *
 * Q and O have H heads, K and V have H_kv heads (1 <= H_kv <= H, H a multiple
 * of H_kv); query head h attends with K/V head h / (H / H_kv) (grouped-query
 * attention; H_kv == H is ordinary multi-head attention).  `layout` is
 * FA_LAYOUT_BHND or FA_LAYOUT_BNHD for all of Q, K, V and O; LSE is always
 * [B, H, N].  Same element types, head dimensions, masks, alignment and error
 * codes as fa_fwd_ex, plus FA_ERR_ARG for a bad H_kv or layout.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int H_kv, int N, int D, float scale,
               int mask_kind, int win_l, int win_r, int dtype, int o_dtype, int layout,
               void* stream);

/*
 * fa_bwd -- gradients dQ, dK, dV of the attention above for an upstream
 * gradient dO of O.  The ops-transformer walk-through's closing remarks say
 * the operator also has a backward pass, without writing it out; this is the
 * chain rule through the definition of "Ascend C advanced practice:
 * high-performance FlashAttention-2-style tile-level fused attention",
 * section 1.1, with P recomputed from the forward's LSE:
 *     P = exp(scale * Q K^T + mask - LSE)      Dsum_i = sum_d dO_id O_id
 *     dV = P^T dO     dS = P * (dO V^T - Dsum)
 *     dQ = scale * dS K      dK = scale * dS^T Q
 * Grouped K/V heads (H_kv < H) sum the gradients of the query heads that
 * share a K/V head.  The LSE output itself is not differentiated.
 *
 * q, o, d_o, dq: [B, H, N, D] (or [B, N, H, D] for FA_LAYOUT_BNHD); k, v,
 * dk, dv: [B, H_kv, N, D] / [B, N, H_kv, D]; lse: [B, H, N] fp32 as fa_fwd_gqa
 * returned it.  dtype FA_F16 or FA_BF16 for every tensor (O as the forward
 * wrote it in that type); D = 64 or 128.  P and dS enter the tensor-core
 * products rounded to dtype; everything else is fp32.  The three outputs are
 * written in full (rows no query sees get zeros) and must not overlap any
 * input.  `workspace` is caller-owned device memory of at least
 * fa_bwd_workspace_bytes(B, H, N) bytes, 256-byte aligned, used by this call
 * only; other pointers 16-byte aligned (lse 4).
 *
 * Returns FA_OK (enqueued on `stream`), FA_ERR_ARG (bad size, mask, H_kv,
 * layout, scale, a NULL pointer, a small workspace), FA_ERR_UNSUPPORTED
 * (FA_F32 or another D), FA_ERR_ALIGN or FA_ERR_CUDA; kernel wait timeouts
 * are reported by fa_device_status().
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int D, float scale,
           int mask_kind, int win_l, int win_r, int dtype, int layout,
           void* workspace, unsigned long long workspace_bytes, void* stream);

/* Workspace fa_bwd needs for B x H rows of length N (two fp32 values per row,
 * rows padded to a multiple of 128).  FA_OK or FA_ERR_ARG. */
int fa_bwd_workspace_bytes(int B, int H, int N, unsigned long long* bytes);

/* Pairings of the rotary embedding (fa_rope). */
enum {
    FA_ROPE_HALF = 0,        /* pair i is (i, i + D/2): rotate-half form     */
    FA_ROPE_INTERLEAVED = 1  /* pair i is (2i, 2i + 1)                       */
};

/*
 * fa_rope -- rotary position embedding of Q and/or K, run before fa_fwd_gqa
 * or fa_decode_gqa.  "Ascend C advanced practice: high-performance
 * FlashAttention-2-style tile-level fused attention", section 9 ("Extensions:
 * integration with RoPE and a paged KV cache"), rotates the Q and K blocks as
 * they are loaded, using a cos/sin table.  The page gives no formula; this is
 * the standard rotary embedding.  Row n of Q sits at position p = q_pos0 + n
 * (of K: k_pos0 + n), and each of its D/2 pairs (x_a, x_b), pair i, becomes
 *     x_a' = x_a cos_tab[p][i] - x_b sin_tab[p][i]
 *     x_b' = x_b cos_tab[p][i] + x_a sin_tab[p][i]
 * in fp32 (x_b sin and x_a sin rounded once, the rest fused), rounded once
 * to the element type.  This entry point is one streaming pass over Q and/or
 * K in device memory.  For the forward, fa_fwd_rope rotates Q inside the
 * attention kernel as its tiles arrive (Q is loaded once per work unit, so
 * nothing is repeated); K stays a pass of its own here, because each K tile
 * is loaded by every CTA of its head and a rotation at the load would be
 * repeated N/256 times per head.
 *
 * q, q_out: [B, H, Nq, D] (FA_LAYOUT_BHND) or [B, Nq, H, D] (FA_LAYOUT_BNHD).
 * k, k_out: [B, H_kv, Nk, D] or [B, Nk, H_kv, D].  dtype: FA_F16, FA_BF16 or
 * FA_F32 for all four.  cos_tab, sin_tab: fp32 [n_pos, D/2] row-major
 * (fa_rope_tables fills them).  Either q or k may be NULL to skip that tensor
 * (its out pointer must then be NULL as well; its sizes are ignored).  In
 * place is allowed (q_out == q, k_out == k); any other overlap is not.  All
 * pointers are caller-owned device memory, 16-byte aligned.
 *
 * Returns FA_OK (enqueued on `stream`), FA_ERR_ARG (a size <= 0, D not a
 * multiple of 16 or above 1024, a position outside [0, n_pos), bad style or
 * layout, missing pointers), FA_ERR_UNSUPPORTED (dtype), FA_ERR_ALIGN or
 * FA_ERR_CUDA.
 */
int fa_rope(const void* q, const void* k, void* q_out, void* k_out, const float* cos_tab, const float* sin_tab,
            int B, int H, int H_kv, int Nq, int Nk, int D, int q_pos0, int k_pos0, int n_pos,
            int style, int dtype, int layout, void* stream);

/*
 * fa_fwd_rope -- fa_fwd_gqa with the rotary embedding of Q applied inside the
 * kernel, as "Ascend C advanced practice: high-performance
 * FlashAttention-2-style tile-level fused attention", section 9, describes:
 * each 128-row Q tile is rotated in shared memory right after its copy lands
 * and before its first Q K^T product.  Query row i sits at position
 * q_pos0 + i and is rotated exactly as fa_rope rotates it (same formula, same
 * rounding, so the result equals fa_rope on Q followed by fa_fwd_gqa bit for
 * bit).  K must already be rotated (fa_rope with q = NULL, or a cache of
 * rotated keys); V is not rotated.
 *
 * cos_tab, sin_tab: fp32 [n_pos, D/2] device tables (fa_rope_tables), 16-byte
 * aligned; style FA_ROPE_HALF or FA_ROPE_INTERLEAVED.  The other arguments,
 * layouts and outputs are those of fa_fwd_gqa; dtype FA_F16 or FA_BF16.
 *
 * Returns FA_OK, FA_ERR_ARG (missing table, n_pos <= 0, q_pos0 < 0,
 * q_pos0 + N > n_pos, bad style, or any fa_fwd_gqa argument error),
 * FA_ERR_UNSUPPORTED (FA_F32, or fa_fwd_gqa's limits), FA_ERR_ALIGN or
 * FA_ERR_CUDA.
 */
int fa_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse,
                const float* cos_tab, const float* sin_tab, int n_pos, int q_pos0, int style,
                int B, int H, int H_kv, int N, int D, float scale,
                int mask_kind, int win_l, int win_r, int dtype, int o_dtype, int layout,
                void* stream);

/*
 * fa_rope_tables -- fill cos_tab and sin_tab (fp32 [n_pos, D/2], caller-owned
 * device memory, 16-byte aligned) with cos and sin of p * base^(-2i/D) for
 * position p and pair i, each computed in double precision and rounded once.
 * Returns FA_OK, FA_ERR_ARG (n_pos <= 0, D odd, <= 0 or above 1024, base not
 * a positive finite number, NULL table), FA_ERR_ALIGN or FA_ERR_CUDA.
 */
int fa_rope_tables(float* cos_tab, float* sin_tab, int n_pos, int D, double base, void* stream);

/*
 * fa_device_status -- synchronise `stream`, then report and clear the
 * library's device status word.  Returns FA_OK, FA_ERR_TIMEOUT (a kernel
 * wait ran past its limit; the kernel stopped early and its outputs are
 * undefined) or FA_ERR_DEVICE (the stream synchronisation itself failed).
 */
int fa_device_status(void* stream);

/* Forward kernels (fa_select_fwd_kernel). */
enum {
    FA_FWD_AUTO = 0,      /* the one-CTA kernel (measured the faster of the two on every benchmark shape) */
    FA_FWD_ONE_CTA = 1,   /* one CTA per SM, two 128-row Q tiles, M = 128 products */
    FA_FWD_CTA_PAIR = 2   /* 2-CTA clusters, M = 256 products over an SM pair (D = 128 only;
                             other head sizes still take the one-CTA kernel) */
};

/*
 * fa_select_fwd_kernel -- choose the tensor-core forward kernel that later
 * fa_fwd* / fa_fwd_gqa / fa_fwd_rope calls launch (process-wide; default
 * FA_FWD_AUTO).  Both compute the same result by the same method; they
 * differ in how work maps onto SMs.  The one-CTA kernel runs one CTA per SM
 * with two 128-row query tiles and M = 128 tcgen05 products.  The CTA-pair
 * kernel runs 2-CTA clusters whose M = 256 products
 * (tcgen05.mma.cta_group::2) split every K and V tile between the two SMs,
 * halving the per-SM shared-memory traffic.  Returns the previous choice, or
 * FA_ERR_ARG for an unknown value.  Host-only.
 */
int fa_select_fwd_kernel(int which);

/* Smallest wait limit fa_set_wait_limit_ns accepts, in nanoseconds. */
#define FA_MIN_WAIT_LIMIT_NS 1000ull

/* Wait limit, in nanoseconds, for every bounded wait inside the kernels
 * (default 2e9), taken by launches enqueued after the call.  Values below
 * FA_MIN_WAIT_LIMIT_NS are raised to it.  Returns the previous value.
 *
 * A wait that runs past the limit makes the kernel stop early: it records
 * FA_ERR_TIMEOUT for fa_device_status, and before it frees its tensor memory
 * and shared memory it waits for the copies and tensor-core products it has
 * already issued.  That final wait has its own fixed bound of one second (or
 * the limit set here, if longer), so a short limit cannot end it while that
 * work is still writing.  A limit below the time a launch's ordinary waits
 * take (microseconds) therefore aborts the launch, with undefined outputs,
 * but leaves the context usable. */
unsigned long long fa_set_wait_limit_ns(unsigned long long ns);

/*
 * fa_selftest_wait_timeout -- enqueue a one-CTA kernel that waits on an
 * mbarrier nothing ever arrives at, bounded by `limit_ns`; it records
 * FA_ERR_TIMEOUT in the device status word and returns.  Exists so a test
 * can check the watchdog path without touching the attention kernels.
 */
int fa_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * fa_plan_units -- host-side view of the work decomposition the tensor-core
 * kernel uses (no GPU needed).  Units are pairs of 128-row query tiles of one
 * (b, h), in the order the kernel hands them out (longest first where their
 * lengths differ; the CTAs that run take the next unit as they become free).
 * If `out` is not NULL,
 * writes min(cap, n_units) records of 6 ints {bh, q0, lo0, hi0, lo1, hi1}:
 * query rows [q0, q0+128) visit key tiles [lo0, hi0), rows [q0+128, q0+256)
 * visit [lo1, hi1) (key tile j = keys [128 j, 128 j + 128)); lo == hi marks a
 * tile past the end of the sequence.  Returns n_units or FA_ERR_ARG.
 */
int fa_plan_units(int B, int H, int N, int mask_kind, int win_l, int win_r, int* out, int cap);

/* 1 if key tile j holds a masked element for some row of the 128-row query
 * tile starting at r0 (the kernel then applies per-element masks), 0 if the
 * whole tile is visible, FA_ERR_ARG on a bad mask.  No GPU needed. */
int fa_tile_needs_mask(int N, int mask_kind, int win_l, int win_r, int r0, int j);

/* 1 if some tile of an N-position problem under this mask may need an element
 * mask or a split P (a window or causal bound, N not a multiple of 128, or
 * N < 512), 0 if none does -- the tensor-core forward then runs a build
 * without those paths -- FA_ERR_ARG on a bad mask.  No GPU needed. */
int fa_geom_needs_masks(int N, int mask_kind, int win_l, int win_r);

/* Human-readable text for a return code. Never NULL. */
const char* fa_strerror(int code);

/* The CUDA error string of the last FA_ERR_CUDA on this host thread. */
const char* fa_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
