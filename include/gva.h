/*
 * gva.h -- C ABI of libgva.so: Grouped Value Attention (GVA) decode on one B300 GPU.
 *
 * GVA caches only the grouped values V[.., G, d_h] and one shared, already-rotated
 * positional key K_rope[.., d_r] per token.  Each query head h owns a map
 * M_h in R^{d_h x d_n}; its content key K_h = V_{g(h)} M_h is never materialised.
 * Instead the query is absorbed once per step, q~_h = q_h^nope M_h^T, and every
 * cached position j is scored as q~_h . v_{j,g(h)} + q_h^rope . k_rope_j, followed
 * by a softmax and the weighted sum of the same V.
 *
 * Sources (web pages, cited by title and section):
 *   [A] "GVA：KV 缓存里的 Key 其实可以不存——从 Value 里"现算"出来就行": 第二次尝试
 *       (K_h = V_{g(h)} M_h), 关键技巧一 (absorption), 关键技巧二 (decoupled shared
 *       RoPE), 缓存账本 (N_GVA = T G d_h + T d_r).
 *   [S] "Grouped Value Attention: Efficient KV Caching via On-Demand Key
 *       Reconstruction": the positional key is cached already rotated; the
 *       absorption is exact.
 *   [K] "KV Cache 优化（一）：从 MHA 到 MQA 与 GQA": §1 (append the current token,
 *       then attend over all history), §4 (GQA), §6.2 (decode shapes), §7 (paging
 *       moves bytes, not maths).
 *
 * Conventions (all entry points):
 *   - Every pointer argument named "device" is CUDA device memory owned by the
 *     caller.  The library never allocates or frees memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and return after enqueueing.  The return value covers host-side
 *     argument validation and launch errors (cudaGetLastError after the launches).
 *   - Device pointers must be 16-byte aligned; otherwise GVA_ERR_ARG.
 *   - No call throws.  Device-side checks (a length beyond the cache capacity, a
 *     block-table entry out of range, a position beyond the RoPE table) never trap:
 *     the offending token or sequence is skipped, and the first such code is kept
 *     in a per-device status word that gva_get_device_status() reads and clears.
 *   - Head grouping: head h reads value group g(h) = h / (H/G) (contiguous blocks).
 *   - Positions are 0-based.  A decode over L_b cached tokens puts the query at
 *     position t = L_b - 1 (the current token is appended before attending, [K] §1).
 *   - RoPE: interleaved pairs (x[2i], x[2i+1]), theta_i = base^(-2i/d_r),
 *     Rot(p): y0 = x0 cos(p theta_i) - x1 sin(p theta_i), y1 = x0 sin + x1 cos.
 *   - Thread safety: calls on different streams may run concurrently; calls that
 *     share a workspace must be ordered by the caller.
 */
#ifndef GVA_H
#define GVA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GVA_ABI_VERSION 6

typedef enum {
    GVA_OK = 0,
    GVA_ERR_ARG = -1,          /* invalid argument (null, misaligned, inconsistent) */
    GVA_ERR_UNSUPPORTED = -2,  /* valid, but a shape / dtype this build does not run */
    GVA_ERR_CUDA = -3,         /* a CUDA runtime call or a launch failed */
    GVA_ERR_WORKSPACE = -4,    /* workspace NULL, too small or not 256-byte aligned */
    GVA_ERR_DEVICE_CHECK = -5  /* returned by gva_get_device_status(): a device check tripped */
} gva_status;

/* Device-side check codes kept in the status word (see gva_get_device_status). */
typedef enum {
    GVA_DEV_OK = 0,
    GVA_DEV_BAD_LENGTH = 1,    /* seq_len[b] < 0 or beyond the sequence's capacity */
    GVA_DEV_BAD_PAGE = 2,      /* block-table entry outside [0, num_rows/page_size) */
    GVA_DEV_BAD_POSITION = 3,  /* append position out of range, or beyond the RoPE table */
    GVA_DEV_TIMEOUT = 4        /* a bounded wait inside a kernel gave up */
} gva_device_check;

typedef enum { GVA_F32 = 0, GVA_BF16 = 1 } gva_dtype;

typedef enum {
    GVA_LAYOUT_CONTIGUOUS = 0, /* row = b * T_cap + j */
    GVA_LAYOUT_RAGGED = 1,     /* row = offsets[b] + j */
    GVA_LAYOUT_PAGED = 2       /* row = block_table[b][j / page_size] * page_size + j % page_size */
} gva_layout;

/* Problem shape.  Supported: H % G == 0 with r = H/G in 1..8; d_h in {32, 64, 128};
 * H * d_h <= 4096; d_n in 8..256, a multiple of 8; d_r in {0, 8, 16, 24, 32};
 * 1 <= B <= 4096; cache_dtype and q_dtype each GVA_F32 or GVA_BF16. */
typedef struct {
    int B;            /* sequences in the batch */
    int H;            /* query heads */
    int G;            /* value groups (GVA) or KV heads (GQA) */
    int d_h;          /* value width (and GQA key width) */
    int d_n;          /* content-query width (GVA) */
    int d_r;          /* positional width (GVA); 0 = no positional slice */
    int cache_dtype;  /* gva_dtype of the cache rows */
    int q_dtype;      /* gva_dtype of the queries */
} gva_dims;

/* Where logical token j of sequence b is stored. */
typedef struct {
    int layout;              /* gva_layout */
    long long num_rows;      /* rows allocated behind every row pointer of the cache */
    long long T_cap;         /* contiguous: rows per sequence (capacity) */
    const int *offsets;      /* ragged: device [B+1], row starts; capacity offsets[b+1]-offsets[b] */
    const int *block_table;  /* paged: device [B][max_pages] physical page ids; capacity
                                max_pages * page_size; pages hold page_size rows */
    int max_pages;           /* paged: columns of block_table */
    int page_size;           /* paged: tokens per page, a positive multiple of 16 */
} gva_rows;

/* GVA cache ([A] 缓存账本; [S]): V rows [G][d_h], K_rope rows [d_r] (already rotated to
 * the row's own position), both cache_dtype, both laid out by `rows`. */
typedef struct {
    gva_rows rows;
    void *V;                 /* device */
    void *K_rope;            /* device; may be NULL when d_r == 0 */
} gva_cache;

/* Matched GQA cache for the comparator ([K] §4): explicit K and V rows [G][d_h]. */
typedef struct {
    gva_rows rows;
    void *K;                 /* device */
    void *V;                 /* device */
} gva_kv_cache;

typedef enum {
    GVA_PATH_AUTO = 0,       /* tensor-core kernels where they apply, else CUDA cores */
    GVA_PATH_SIMT = 1,       /* CUDA-core kernel (fp32 FMA); every supported shape */
    GVA_PATH_MMA = 2         /* separate absorb, bf16 tensor-core split-K and combine
                                kernels (bf16 cache only) */
} gva_path;

/* Query RMSNorm before absorption (the "scale-matched + query RMSNorm" variant named
 * in [A] 实验 and [S]'s results table; the pages give no formula, the reading is):
 *   q_nope[b,h,:] <- gain * q_nope[b,h,:] / sqrt(mean_k q_nope[b,h,k]^2 + eps)
 * per head over its d_n values; the positional query is not normalised. */
#define GVA_FLAG_QUERY_RMSNORM 1

typedef struct {
    int path;                /* gva_path */
    int num_ctas;            /* decode grid size; 0 = the library's choice for this GPU */
    int flags;               /* 0 or GVA_FLAG_QUERY_RMSNORM; other bits: GVA_ERR_ARG */
    float q_norm_eps;        /* with GVA_FLAG_QUERY_RMSNORM: eps >= 0 (finite) */
    const float *q_norm_gain;/* with GVA_FLAG_QUERY_RMSNORM: device fp32 [d_n], shared by
                                all heads, or NULL for ones */
} gva_decode_opts;

/* ------------------------------------------------------------------------- */

/* Human-readable name of a gva_status or gva_device_check value (static string). */
const char *gva_status_string(int status);

/* GVA_ABI_VERSION of the loaded library. */
int gva_abi_version(void);

/* Fill a HOST table [max_pos][d_r/2][2] of fp32 (cos, sin)(p * theta_i),
 * theta_i = base^(-2i/d_r), each computed in double and rounded once.  The caller
 * copies it to the device and passes it as `rope_tab` below.  Reading of [A]
 * 关键技巧二 (the pages name only the relative rotation R_{j-t}).  With d_r = 0 there
 * is nothing to fill and host_tab may be NULL.
 * Errors: GVA_ERR_ARG for a NULL table (d_r > 0), max_pos < 1, odd or negative d_r,
 * base <= 0. */
int gva_rope_table_fill(float *host_tab, int max_pos, int d_r, double base);

/* Query absorption ([A] 关键技巧一, [S]):
 *   q_tilde[b,h,:]    = scale * q_nope[b,h,:] M_h^T         M: device fp32 [H][d_h][d_n]
 *   q_rope_rot[b,h,:] = scale * Rot(L_b - 1) q_rope[b,h,:]  (position 0 when L_b = 0)
 * q_nope [B][H][d_n], q_rope [B][H][d_r] (q_dtype), seq_len device int [B],
 * rope_tab device [rope_max_pos][d_r/2][2]; outputs device fp32 [B][H][d_h] and
 * [B][H][d_r] (q_rope_rot may be NULL when d_r == 0).  gva_decode_attention runs
 * the same step internally; this entry point exposes it for reuse and testing. */
int gva_absorb_query(void *stream, const gva_dims *dims, const void *q_nope,
                     const void *q_rope, const float *M, const int *seq_len,
                     const float *rope_tab, int rope_max_pos, float scale,
                     float *q_tilde, float *q_rope_rot);

/* gva_absorb_query with options: only opts->flags (GVA_FLAG_QUERY_RMSNORM), q_norm_eps
 * and q_norm_gain are read; opts may be NULL. */
int gva_absorb_query_ex(void *stream, const gva_dims *dims, const void *q_nope,
                        const void *q_rope, const float *M, const int *seq_len,
                        const float *rope_tab, int rope_max_pos, float scale,
                        float *q_tilde, float *q_rope_rot, const gva_decode_opts *opts);

/* Cache append ([S]: cached already rotated; [K] §1: append, then attend):
 *   V[row(b, pos[b])]      = v_new[b]                   (rounded once to cache_dtype)
 *   K_rope[row(b, pos[b])] = Rot(pos[b]) k_rope_new[b]
 * The rotated key is computed in fp32 in a fixed order with no fused multiply-add,
 * y0 = (x0*c) - (x1*s), y1 = (x0*s) + (x1*c), c/s from rope_tab, then rounded once
 * (RNE) to the cache dtype, so the stored bytes are reproducible bit for bit.
 * v_new device fp32 [B][G][d_h]; k_rope_new device fp32 [B][d_r] (unrotated);
 * pos device int [B]; seq_len_out (optional, device int [B]) receives pos[b] + 1
 * and may alias pos.  A position outside the sequence's capacity or the RoPE
 * table skips that sequence and sets GVA_DEV_BAD_POSITION. */
int gva_append_cache(void *stream, const gva_dims *dims, const float *v_new,
                     const float *k_rope_new, const int *pos, int *seq_len_out,
                     const gva_cache *cache, const float *rope_tab, int rope_max_pos);

/* Bytes of device workspace gva_decode_attention / gva_gqa_decode_attention need for
 * `dims` on the current device (split-K partials and the absorbed queries).
 * 0 on invalid dims. */
size_t gva_decode_workspace_size(const gva_dims *dims);

/* GVA decode attention over a contiguous, ragged or paged cache ([A] 关键技巧一/二;
 * [K] §1, §6.2).  For every sequence b and head h, with t = L_b - 1 = seq_len[b] - 1:
 *   z_j = scale * (q~_h . v_{j,g(h)} + Rot(t) q_rope_h . k_rope_j),  j < L_b
 *   out[b,h,:] = sum_j softmax(z)_j v_{j,g(h)}     (device fp32 [B][H][d_h])
 *   lse[b,h]   = ln sum_j exp(z_j)                 (device fp32 [B][H], or NULL)
 * L_b = 0 gives out = 0 and lse = -inf.  Split-K flash-decoding over 16-token slabs
 * spread evenly over the GPU, then a log-sum-exp merge of the splits: three kernels
 * (absorb, split-K partial, combine).  The workspace (device,
 * >= gva_decode_workspace_size(dims), 256-byte aligned) is scratch only: every value
 * the call reads there it wrote first.  q_nope/q_rope/M/seq_len/rope_tab as in
 * gva_absorb_query. */
int gva_decode_attention(void *stream, const gva_dims *dims, const void *q_nope,
                         const void *q_rope, const float *M, const int *seq_len,
                         const gva_cache *cache, const float *rope_tab, int rope_max_pos,
                         float scale, float *out, float *lse, void *workspace,
                         size_t ws_bytes);

/* gva_decode_attention with kernel options (path selection, grid size, query RMSNorm);
 * opts may be NULL.  GVA_ERR_UNSUPPORTED when the requested path cannot run `dims`. */
int gva_decode_attention_ex(void *stream, const gva_dims *dims, const void *q_nope,
                            const void *q_rope, const float *M, const int *seq_len,
                            const gva_cache *cache, const float *rope_tab,
                            int rope_max_pos, float scale, float *out, float *lse,
                            void *workspace, size_t ws_bytes, const gva_decode_opts *opts);

/* Bytes of device workspace gva_prefill_attention needs for a chunk of n queries per
 * sequence over `rows` on the current device.  0 on invalid arguments or a layout the
 * prefill does not take (a ragged cache when the tcgen05 prefill kernel does not take
 * the shape). */
size_t gva_prefill_workspace_size(const gva_dims *dims, int n, const gva_rows *rows);

/* Causal chunked prefill ([K] §1: every new token attends to the cached history and to
 * the chunk up to and including itself; [K] §6.1: the chunk's tokens enter together and
 * a group's query heads share its rows; [A] 关键技巧一/二 for the scores).  Sequence b
 * holds L0[b] tokens (device int [B]); its n new tokens go to positions
 * p = L0[b] + i, i < n.  The call appends all of them, exactly as gva_append_cache
 * would one by one (v_new device fp32 [B][n][G][d_h], k_rope_new device fp32
 * [B][n][d_r], unrotated), then for query i of sequence b computes the decode of
 * gva_decode_attention over positions 0..p with the positional query rotated by p:
 *   out[b,i,h,:] (device fp32 [B][n][H][d_h]), lse[b,i,h] (device fp32 [B][n][H] or NULL).
 * q_nope [B][n][H][d_n], q_rope [B][n][H][d_r] (q_dtype); M, rope_tab, scale and opts
 * as in gva_decode_attention_ex.  L0 is not updated (the caller adds n).
 * Paths: GVA_PATH_AUTO runs, for bf16 caches with d_h 64 or 128, a tensor-core prefill
 * kernel that loads each tile of a sequence's rows once and scores it against all of the
 * chunk's queries (split over the history, merged by log-sum-exp): the tcgen05 kernel
 * when a value group's chunk rows n * H / G fit one product (<= 64, or <= 128 at
 * d_h = 64), else an mma.sync kernel; every
 * other case, and GVA_PATH_SIMT / _MMA, runs each query as one entry of a
 * decode batch of B*n entries reading sequence b's rows (a paged view of the cache).
 * Layouts: paged, and contiguous with T_cap a positive multiple of 16; ragged only on
 * GVA_PATH_AUTO when the tcgen05 kernel takes the shape (it reads the caller's rows; the
 * other paths need page-aligned rows), else GVA_ERR_UNSUPPORTED.  B*n <= 4096 (else GVA_ERR_ARG).  Workspace: device, 256-byte
 * aligned, >= gva_prefill_workspace_size(dims, n, &cache->rows), scratch only, one call
 * in flight per workspace (the tcgen05 kernel's merge counters live in it and are reset
 * by the call itself).  A chunk that does not fit the capacity or the RoPE table
 * sets GVA_DEV_BAD_POSITION / GVA_DEV_BAD_LENGTH for the queries concerned. */
int gva_prefill_attention(void *stream, const gva_dims *dims, int n, const void *q_nope,
                          const void *q_rope, const float *M, const int *L0,
                          const float *v_new, const float *k_rope_new,
                          const gva_cache *cache, const float *rope_tab, int rope_max_pos,
                          float scale, float *out, float *lse, void *workspace,
                          size_t ws_bytes, const gva_decode_opts *opts);

/* Matched GQA decode, the comparator ([K] §4): out[b,h] = softmax(scale q_h K_g^T) V_g
 * with explicit K and V rows [G][d_h] (cache_dtype).  q device [B][H][d_h] (q_dtype);
 * dims.d_n and dims.d_r are ignored.  Same split-K design, workspace and outputs as
 * gva_decode_attention; opts may be NULL (GVA_FLAG_QUERY_RMSNORM: GVA_ERR_UNSUPPORTED). */
int gva_gqa_decode_attention(void *stream, const gva_dims *dims, const void *q,
                             const int *seq_len, const gva_kv_cache *cache, float scale,
                             float *out, float *lse, void *workspace, size_t ws_bytes,
                             const gva_decode_opts *opts);

/* MLA-shaped decode: the second reference point at matched cache bytes ([A] 问题 and
 * 对 MLA 的优势: a latent cache of T (d_c + d_r) scalars against GVA's T (G d_h + d_r); the
 * KV-cache compression survey's MLA sections: per-head up-projections of one latent).
 * Cache rows hold a latent c_j [d_c] and one shared, already-rotated positional key [d_r]
 * (gva_cache with V -> the latent rows).  Head h's key is [c_j W_uk_h ; k_rope_j] with
 * W_uk_h in R^{d_c x d_n}, its value c_j W_uv_h with W_uv_h in R^{d_c x d_h}; the query is
 * [q_nope ; Rot(t) q_rope], t = L_b - 1:
 *   z_j = scale (q_nope . c_j W_uk_h + Rot(t) q_rope . k_rope_j)
 *   out[b,h,:] = sum_j softmax(z)_j c_j W_uv_h,   lse[b,h] = ln sum_j exp(z_j)
 * computed as the absorbed decode over the latent rows followed by the up-projection:
 * q~_h = q_nope W_uk_h^T, o~ = sum_j softmax(z)_j c_j, out = o~ W_uv_h.
 * Supported: bf16 cache; d_c in {128, 256}; H a multiple of 4 with H / 4 <= 8; d_n in
 * 8..256 (multiple of 8); d_r in {0, 8, 16, 24, 32}; d_h in {32, 64, 128, 256}. */
typedef struct {
    int B;            /* sequences */
    int H;            /* query heads */
    int d_c;          /* latent width of a cache row */
    int d_n;          /* content-query width */
    int d_r;          /* positional width */
    int d_h;          /* output (value) width per head */
    int cache_dtype;  /* gva_dtype of the cache rows (GVA_BF16 runs; GVA_F32: UNSUPPORTED) */
    int q_dtype;      /* gva_dtype of the queries */
} gva_mla_dims;

/* Bytes of device workspace gva_mla_decode_attention needs on the current device (0 on
 * invalid dims). */
size_t gva_mla_workspace_size(const gva_mla_dims *dims);

/* MLA-shaped decode (see gva_mla_dims).  q_nope device [B][H][d_n], q_rope [B][H][d_r]
 * (q_dtype); W_uk device fp32 [H][d_c][d_n]; W_uv device fp32 [H][d_c][d_h]; seq_len device
 * int [B]; cache: latent rows [d_c] in cache->V, positional keys [d_r] in cache->K_rope,
 * laid out by cache->rows; rope_tab as in gva_absorb_query; out device fp32 [B][H][d_h];
 * lse device fp32 [B][H] or NULL; workspace device, 256-byte aligned, >=
 * gva_mla_workspace_size(dims) (scratch only).  Errors as gva_decode_attention. */
int gva_mla_decode_attention(void *stream, const gva_mla_dims *dims, const void *q_nope,
                             const void *q_rope, const float *W_uk, const float *W_uv,
                             const int *seq_len, const gva_cache *cache, const float *rope_tab,
                             int rope_max_pos, float scale, float *out, float *lse,
                             void *workspace, size_t ws_bytes);

/* ------------------------------------------------------------------------- */
/* Decode of the variant with ordinary RoPE on the reconstructed key.           */
/* The agihunt summary (results discussion) describes a scale-matched GVA row   */
/* that rotates the rebuilt key K_h = V_g M_h itself with plain RoPE, so that   */
/* M_h can no longer be folded into the query; the analysis page (关键技巧二)   */
/* explains why: the relative rotation would sit between q and M_h^T.  The     */
/* pages give no formula; this library reads it as                              */
/*   z_j = scale * (Rot(t) q_h) . (Rot(j) v_{j,g} M_h),  t = L_b - 1,             */
/*   out[b,h] = sum_j softmax(z)_j v_{j,g},  lse[b,h] = logsumexp_j z_j,          */
/* with Rot over d_n dimensions in interleaved pairs (theta_i over d_n) and no  */
/* separate positional key.  Each token costs d_h * d_n multiply-adds per head  */
/* on the tensor cores.                                                          */
/* ------------------------------------------------------------------------- */

/* Bytes of device workspace gva_rope_keys_decode_attention needs for `dims` on the
 * current device (0 on invalid dims).  dims->d_r must be 0. */
size_t gva_rope_keys_workspace_size(const gva_dims *dims);

/* Decode of the variant above, one new query per sequence.
 *   q        device [B][H][d_n] (dims->q_dtype), the whole query of each head
 *   M        device fp32 [H][d_h][d_n]
 *   seq_len  device int [B]; L_b = 0 gives out = 0, lse = -inf
 *   cache    value rows [G][d_h] in cache->V (bf16 runs; fp32 returns
 *            GVA_ERR_UNSUPPORTED), laid out by cache->rows; cache->K_rope is not read
 *   rope_tab device fp32 [rope_max_pos][d_n/2][2] (cos, sin)(p theta_i), theta_i =
 *            base^(-2i/d_n) (gva_rope_table_fill with d_r = d_n); rope_max_pos >= 128
 *            and >= every L_b (a longer sequence counts as empty and sets
 *            GVA_DEV_BAD_POSITION)
 *   out      device fp32 [B][H][d_h]; lse device fp32 [B][H] or NULL
 *   workspace device, 256-byte aligned, >= gva_rope_keys_workspace_size(dims); scratch only
 * Runs for d_h and d_n in {64, 128} (else GVA_ERR_UNSUPPORTED).  All device buffers are
 * caller-owned and 16-byte aligned; asynchronous on `stream`.  Errors as
 * gva_decode_attention. */
int gva_rope_keys_decode_attention(void *stream, const gva_dims *dims, const void *q,
                                   const float *M, const int *seq_len, const gva_cache *cache,
                                   const float *rope_tab, int rope_max_pos, float scale,
                                   float *out, float *lse, void *workspace, size_t ws_bytes);

/* Size of the fixed device array behind gva_decode_attention_static (24 MiB). */
#define GVA_STATIC_SCRATCH_BYTES (24u << 20)

/* gva_decode_attention without a caller-provided workspace, for callers that cannot
 * allocate device memory where they decode: plugins or embedded runtimes handed no
 * allocator and no scratch buffer, engines whose device memory is planned once at
 * start-up and may not grow afterwards, and latency-critical loops that forbid
 * allocator calls because those can block or synchronise the device.  The source pages
 * have no counterpart to this entry point; it exists for deployment only.
 *   - Scratch is one fixed array of GVA_STATIC_SCRATCH_BYTES in device memory, held by
 *     every GPU that loads the library until the process exits.  Shapes whose
 *     workspace (gva_decode_workspace_size) exceeds it return GVA_ERR_WORKSPACE.
 *   - Nothing is allocated or freed: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device resolves the array's device address (set-up); make
 *     that first call before any stream capture, after which the call can be captured
 *     into a CUDA graph (tested).  `stream` must belong to the current device (else
 *     GVA_ERR_CUDA); while `stream` is capturing, its device is taken to be that of `out`.
 *   - Every call on a device shares the one array, and its contents persist from the
 *     previous call.  The call takes the automatic path, which writes every scratch
 *     value before it reads it, so nothing in the array has to start at any value.
 *     Calls that may overlap on the GPU (different streams, or work not ordered by the
 *     caller) race on the array; order them.
 * Arguments, outputs and errors otherwise as gva_decode_attention. */
int gva_decode_attention_static(void *stream, const gva_dims *dims, const void *q_nope,
                                const void *q_rope, const float *M, const int *seq_len,
                                const gva_cache *cache, const float *rope_tab,
                                int rope_max_pos, float scale, float *out, float *lse);

/* One layer of a decode step (gva_decode_step): its new token's value and positional key
 * (v_new device fp32 [B][G][d_h], k_rope_new device fp32 [B][d_r] unrotated; v_new NULL:
 * no append for this layer), its queries and map as in gva_decode_attention, its cache,
 * and its outputs out (device fp32 [B][H][d_h]) and lse (device fp32 [B][H] or NULL). */
typedef struct {
    const float *v_new;
    const float *k_rope_new;
    const void *q_nope;
    const void *q_rope;
    const float *M;
    gva_cache cache;
    float *out;
    float *lse;
} gva_layer_args;

/* One decode step through n_layers layers of the same shape, issued from one host call
 * (a native executor for the per-step loop of a model's layers).  For l = 0 .. n_layers-1
 * in order on `stream`: gva_append_cache(v_new, k_rope_new, pos, NULL) when layers[l].v_new
 * is not NULL, then gva_decode_attention_ex(q_nope, q_rope, M, seq_len, layers[l].cache,
 * rope_tab, rope_max_pos, scale, out, lse, workspace, ws_bytes, opts).  The layers share
 * the positions, lengths, table, scale, options and one workspace (>= 
 * gva_decode_workspace_size(dims)): every kernel of a layer waits for the layer before it,
 * so the scratch is reused in order.  The result is that of the per-layer calls, bit for
 * bit.  The append and the absorption read and write disjoint buffers, so on the
 * tensor-core path with a bf16 cache and d_n = 64 or 128 they run as one grid (a layer is
 * then three launches).  The decode streams the cache while that grid runs and copies the
 * 16-row slab that holds sequence b's position pos[b] only once the grid has completed, so
 * a new row must be read by its own sequence only (no other sequence's rows or pages may
 * hold it), and the layer's cache must not overlap its queries, map, lengths or positions.  A layer's append and decode
 * arguments are both checked before its first launch.  Returns GVA_OK, GVA_ERR_ARG for
 * n_layers < 0 or a NULL `layers` with n_layers > 0, or the first error of a layer's call
 * (the layers before it are launched, the rest are not). */
int gva_decode_step(void *stream, const gva_dims *dims, int n_layers,
                    const gva_layer_args *layers, const int *pos, const int *seq_len,
                    const float *rope_tab, int rope_max_pos, float scale, void *workspace,
                    size_t ws_bytes, const gva_decode_opts *opts);

/* A decode step recorded once and replayed: a native executor over CUDA graphs.
 * gva_step_plan_create records one gva_decode_step with these arguments (on a private
 * stream of the current device, in stream capture) into an instantiated CUDA graph;
 * gva_step_plan_launch replays the whole step on `stream` with one launch.  The plan keeps
 * the addresses, not the contents: the caller refreshes the inputs in place between
 * launches (new tokens, queries, lengths, positions), keeps every buffer alive and in
 * place while the plan exists, and orders launches that share buffers.  A replay computes
 * what gva_decode_step computes on the buffers' current contents, bit for bit.
 * Creating a plan performs the library's one-time device set-up first and allocates
 * driver resources (a stream and an instantiated graph), no device buffers.
 * create: GVA_ERR_ARG for plan_out NULL, n_layers < 1 or layers NULL; any error of the
 * recorded calls (then *plan_out is NULL); GVA_ERR_CUDA when recording or instantiation
 * fails.  launch: GVA_ERR_ARG for a NULL plan, GVA_ERR_CUDA when the stream belongs to
 * another device than the plan's or the launch fails.  destroy: releases the plan (NULL
 * is accepted); the caller orders it after the plan's last launch has completed. */
typedef struct gva_step_plan gva_step_plan;
int gva_step_plan_create(const gva_dims *dims, int n_layers, const gva_layer_args *layers,
                         const int *pos, const int *seq_len, const float *rope_tab,
                         int rope_max_pos, float scale, void *workspace, size_t ws_bytes,
                         const gva_decode_opts *opts, gva_step_plan **plan_out);
int gva_step_plan_launch(gva_step_plan *plan, void *stream);

/* One layer of a recorded prefill: its chunk's queries, map, new values and positional
 * keys, cache and outputs, as in gva_prefill_attention. */
typedef struct {
    const void *q_nope;
    const void *q_rope;
    const float *M;
    const float *v_new;
    const float *k_rope_new;
    gva_cache cache;
    float *out;
    float *lse;
} gva_prefill_layer_args;

/* A chunked prefill through n_layers layers recorded as a plan: one gva_prefill_attention
 * per layer, in order, sharing L0, the table, scale, options and one workspace
 * (>= gva_prefill_workspace_size(dims, n, &layers[0].cache.rows); every layer's rows
 * must have that layout and size).  Launched and destroyed like a step plan, with the
 * same rules on buffers, and the same errors (GVA_ERR_ARG also for n < 1). */
int gva_prefill_plan_create(const gva_dims *dims, int n, int n_layers,
                            const gva_prefill_layer_args *layers, const int *L0,
                            const float *rope_tab, int rope_max_pos, float scale,
                            void *workspace, size_t ws_bytes, const gva_decode_opts *opts,
                            gva_step_plan **plan_out);
int gva_step_plan_destroy(gva_step_plan *plan);

/* Read and clear the current device's status word (synchronous: it waits for all
 * work on the device).  *code_out receives a gva_device_check value.  Returns
 * GVA_OK when no check tripped, GVA_ERR_DEVICE_CHECK when one did, GVA_ERR_CUDA on
 * a CUDA failure. */
int gva_get_device_status(int *code_out);

/* Measurement helper (not on the decode path): read `bytes` of device memory at `buf`
 * once, as a pure read stream (16-byte non-allocating loads, about 16 loads in flight
 * per thread, 2048 threads per SM), and fold the words into *sink (device unsigned,
 * XOR of every 32-bit word of the buffer, overwritten) so that no load is dead.  Its
 * throughput is the read-only ceiling the decode kernels are compared with.  `buf`
 * 16-byte aligned, `bytes` a positive multiple of 16; otherwise GVA_ERR_ARG. */
int gva_read_probe(void *stream, const void *buf, size_t bytes, unsigned *sink);

/* Self-test of the kernels' bounded waits (not on the decode path).  Every in-kernel wait
 * on an mbarrier gives up after a limit, records GVA_DEV_TIMEOUT and lets its kernel
 * return, so a lost producer never hangs the GPU.  This launches one warp that waits on
 * an mbarrier nothing arrives on, with a limit of `limit_us` microseconds (1 .. 10^6):
 * after it the device status (gva_get_device_status) reads GVA_DEV_TIMEOUT and the
 * context stays usable.  Asynchronous on `stream`; GVA_ERR_ARG for a limit out of range. */
int gva_selftest_bounded_wait(void *stream, unsigned limit_us);

/* Streaming multiprocessors of the current device (the decode grid is sized from it). */
int gva_num_sms(void);

/* cudaError_t code of the most recent CUDA failure seen by a gva_* call on the calling
 * host thread (0 if none); it explains a GVA_ERR_CUDA return. */
int gva_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GVA_H */
