/*
 * csa2.h -- C ABI of the CSA2 (Compressed Sparse Attention 2) attention step
 * for one GB300 GPU (sm_103a).
 *
 * Sources for the operations (page title, section):
 *   [P1] "DeepSeek-V4.1-Flash" research note (vibe-research.pages.dev)
 *   [P2] "DeepSeek-V4.1-Flash 架构详解：CED、CSA2 与 890 字节 KV Cache" (gentlecold.top)
 *   [P3] DeepSeek-V4 report explainer (mlqm.cn)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All data pointers are DEVICE pointers unless a comment says otherwise.
 *   The caller owns every buffer (caches, block tables, inputs, outputs,
 *   workspaces); the library never allocates, frees or keeps a pointer past
 *   the call.
 * - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *   stream).  Host pointers to descriptor structs are read during the call
 *   only.
 * - Every function returns CSA2_OK (0) or a negative csa2 status.  Shapes and
 *   pointers are validated on the host before any launch; nothing is launched
 *   when validation fails.  A launch failure returns CSA2_ERR_CUDA and
 *   csa2_last_cuda_error() gives the cudaError_t.
 * - Data-dependent faults found on the device (a block-table page id outside
 *   the cache, a slot outside the cache) skip the offending access and set
 *   a bit in the cache's optional device status word (csa2_cache.status,
 *   CSA2_DEV_* bits), which the caller may read after synchronising.
 * - bf16 tensors are passed as uint16_t bit patterns.
 *
 * Cache layout (per compressed entry "slot"; one block-table page = 64 slots)
 * ---------------------------------------------------------------------------
 *   kv_codes  [num_slots][256]  FP4 E2M1 codes of the 512-dim main KV entry:
 *                               element 2i in the low nibble of byte i,
 *                               element 2i+1 in the high nibble; nibble bit 3
 *                               is the sign.  [P2] §4 (OCP MXFP4, E2M1).
 *   kv_scales [num_slots][16]   kv_format CSA2_KV_MXFP4: E8M0 scale byte
 *                               (2^(byte-127)) of each 32-element block
 *                               (OCP MX block size), 272 B per entry;
 *             [num_slots][32]   kv_format CSA2_KV_FP4_E4M3: E4M3 scale byte of
 *                               each 16-element block ([P2] §4 and [P4]: 16
 *                               channels share one E4M3 scale), 288 B.
 *   ik_codes  [num_slots][128]  FP8 e4m3 codes of the 128-dim indexer key.
 *   ik_scales [num_slots]       fp32 per-entry scale of the indexer key.
 * Logical entry e of sequence b lives in slot
 *   block_table[b * max_pages + e / 64] * 64 + e % 64.
 * The main KV and the indexer keys of an entry share that slot: both are
 * produced by a Full layer and reused by the layers after it ([P2] §3 mode
 * table).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa2_stream_t; /* same object as cudaStream_t */

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

/* ---- status codes ------------------------------------------------------ */
#define CSA2_OK               0
#define CSA2_ERR_NULL        (-1)  /* a required pointer is NULL            */
#define CSA2_ERR_SHAPE       (-2)  /* a size or count is out of range       */
#define CSA2_ERR_UNSUPPORTED (-3)  /* valid but not implemented (e.g. mode) */
#define CSA2_ERR_RANGE       (-4)  /* index / length beyond a buffer        */
#define CSA2_ERR_WORKSPACE   (-5)  /* workspace missing or too small        */
#define CSA2_ERR_TIMEOUT     (-6)  /* a bounded device wait gave up         */
#define CSA2_ERR_CUDA        (-7)  /* a CUDA call failed (see below)        */
#define CSA2_ERR_ALIGN       (-8)  /* a pointer lacks the required alignment */

/* bits of the device status word */
#define CSA2_DEV_BAD_PAGE     1    /* block-table page id outside the cache */
#define CSA2_DEV_BAD_SLOT     2    /* destination slot outside the cache    */
#define CSA2_DEV_TIMEOUT      4    /* a bounded spin-wait ran out            */
#define CSA2_DEV_BAD_INDEX    8    /* a selected index outside the context   */

/* ---- fixed dimensions ([P2] §1 configuration table) ---------------------- */
#define CSA2_HEADS         64     /* query heads                             */
#define CSA2_HEAD_DIM      512    /* head dim = main KV entry width (MQA)    */
#define CSA2_IDX_HEADS     32     /* lightning-indexer heads                  */
#define CSA2_IDX_DIM       128    /* lightning-indexer dim                    */
#define CSA2_TOPK          512    /* selected entries per query               */
#define CSA2_BLOCK         8      /* positions per candidate block            */
#define CSA2_POOL_BLOCKS   2048   /* blocks kept by a Full layer              */
#define CSA2_POOL_MAX      16384  /* = CSA2_POOL_BLOCKS * CSA2_BLOCK          */
#define CSA2_SWA_WINDOW    128    /* sliding-window tokens                    */
#define CSA2_PAGE          64     /* slots per block-table page               */
#define CSA2_MX_BLOCK      32     /* elements per MX scale                    */

/* layer modes ([P2] §3 mode table) */
#define CSA2_MODE_FULL     0
#define CSA2_MODE_REINDEX  1
#define CSA2_MODE_REUSE    2

/* main-KV formats (csa2_cache.kv_format) */
#define CSA2_KV_MXFP4      0      /* 32-element blocks, E8M0 scale            */
#define CSA2_KV_FP4_E4M3   1      /* 16-element blocks, E4M3 scale            */

/* ---- descriptors -------------------------------------------------------- */

/* The layer-shared global cache of compressed entries. */
typedef struct csa2_cache {
    uint8_t       *kv_codes;     /* [num_slots][256]                         */
    uint8_t       *kv_scales;    /* [num_slots][16]                          */
    uint8_t       *ik_codes;     /* [num_slots][128]                         */
    float         *ik_scales;    /* [num_slots]                              */
    int64_t        num_slots;    /* > 0, multiple of 64                      */
    const int32_t *block_table;  /* [batch][max_pages] page ids              */
    int32_t        max_pages;    /* row stride of block_table, > 0           */
    int32_t        kv_format;    /* CSA2_KV_MXFP4 (0) or CSA2_KV_FP4_E4M3 (1) */
    int32_t       *status;       /* device status word (CSA2_DEV_*), or NULL */
} csa2_cache;

/* A batch of sequences, each with nq query tokens. */
typedef struct csa2_batch {
    int32_t        batch;        /* B >= 1                                   */
    int32_t        nq;           /* queries per sequence Q >= 1              */
    int32_t        m;            /* compression ratio (1 decoder, 2 encoder) */
    int32_t        pad_;
    int64_t        max_entries;  /* host-side bound on n_entries[b]; sizes
                                    grids and score rows                      */
    const int64_t *n_entries;    /* [B] entries held in the cache (device)    */
    const int64_t *q_pos;        /* [B*Q] token position t of each query;
                                    entry j is visible to it iff
                                    (j+1)*m - 1 <= t and j < n_entries[b]
                                    ([P3] §3.3: a query cannot see the rest
                                    of its own unfinished block)              */
} csa2_batch;

/* One layer's FP8 sliding-window KV ([P1] §3.3 / [P2] §4: FP8, per layer).
 * A ring of `rows` token rows per sequence: token t lives in row t % rows.
 * The window of the query at token t is SWAKeys(t) = [max(s, t-127), t]
 * ([P2] §5 bounded-replay equation), s = start[b] (0 when start is NULL).
 * The caller guarantees that every window token of every query of the call
 * is present in its row (rows >= 128 + spread of query positions). */
typedef struct csa2_swa {
    const uint8_t *codes;        /* [B][rows][512] e4m3                       */
    const float   *scales;       /* [B][rows] fp32 per-token scale            */
    int32_t        rows;         /* ring capacity, >= 128                     */
    int32_t        flags;        /* CSA2_ATTN_* option bits                   */
    const int64_t *start;        /* [B] replay start s, or NULL               */
    const float   *new_rows;     /* NULL, or fp32 [B][512] (decode, Q = 1):   */
                                 /* the window row of each query's own token, */
                                 /* quantised by the attention call itself    */
                                 /* into ring row q_pos % rows (codes and     */
                                 /* scale written, as csa2_quant_fp8 would)   */
                                 /* before it is attended; 16-byte aligned    */
    const float   *sink;         /* NULL, or fp32 [64]: per-head sink logit z_h
                                    joining the softmax denominator without a
                                    value ([P3] §4.3): o_h = sum e^l k /
                                    (e^z_h + sum e^l), lse_h = log(e^z_h +
                                    sum e^l); -inf is no sink                 */
    float          rope_base;    /* > 0: rotate the output's RoPE dims back by
                                    the query position t ([P3] §4.3 partial
                                    RoPE on the last 64 dims): dims 448+i and
                                    480+i (i < 32) by -t * rope_base^(-i/32);
                                    0: no rotation                             */
    int32_t        pad_;
} csa2_swa;

/* csa2_swa.flags: drop the selected entries whose token is also in the
 * query's window (m = 1; the window row stays) instead of attending to both. */
#define CSA2_ATTN_DEDUP_WINDOW 1
/* csa2_swa.flags, honoured by csa2_layer in REUSE mode (ignored elsewhere):
 * the caller guarantees that the previous call into this library on the same
 * stream was csa2_layer, and that the index array, the main-KV entries it
 * selects, the window rows other than each query's own token and the batch
 * description were all written before that call's attention.  The attention
 * then loads and dequantises those keys while the previous layer's last kernel
 * is still running (q and new_rows are still read only after that kernel has
 * completed).  A decode stack that calls csa2_layer layer after layer, with
 * the window rows of its own tokens passed as new_rows, satisfies it. */
#define CSA2_ATTN_EARLY_INPUTS 2
/* csa2_swa.flags, honoured by csa2_layer in REUSE mode (ignored elsewhere;
 * refused by csa2_layer_noalloc, whose calls share one scratch array): all of
 * CSA2_ATTN_EARLY_INPUTS's guarantees, and further that q and new_rows are in
 * place before this call's kernels can start (written before the previous
 * call into this library on the stream, or ordered before this call by a
 * stream or event dependency), and that this call's workspace does not overlap
 * the previous call's.  The
 * attention then runs its whole computation while the previous layer's last
 * kernel is still running and waits for it only before writing its workspace
 * (which the previous layer's merge may still be reading from its own).  A
 * decode stack whose inputs are in place before the step and whose layer
 * calls alternate between two workspaces satisfies it.  No counterpart in the
 * pages. */
#define CSA2_ATTN_EARLY_ALL 16
/* csa2_swa.flags: the schedule of the attention kernels (the same arithmetic
 * either way up to the order of the softmax rescaling; no counterpart in the
 * pages).  CHUNKS: one two-CTA cluster per (query row, 128-key chunk) and a
 * merge kernel -- the shortest latency for a few rows.  ROWS: persistent
 * two-CTA clusters, each taking whole rows with an online softmax over the
 * row's chunks and writing o and lse directly -- for many rows (prefill,
 * several query tokens per sequence, large decode batches).  Neither bit:
 * CHUNKS below 40 query rows, ROWS from 40.  Both bits: CSA2_ERR_UNSUPPORTED. */
#define CSA2_ATTN_SCHEDULE_CHUNKS 4
#define CSA2_ATTN_SCHEDULE_ROWS 8

/* csa2_layer_io.flags: FULL and REINDEX layers keep the index scores in bf16
 * (each fp32 score rounded to nearest even) and select on them: the block
 * maxima are those of the rounded scores and the Top-512 ranks the rounded
 * scores (ties to the lower position).  The pages report that a BF16 score
 * path doubles Top-K speed at 99.7 % recall ("DeepSeek-V4 report explainer"
 * §10.2); this is that trade, outside the fp32 parity rule: near-ties at the
 * threshold may resolve differently from fp32 scores. */
#define CSA2_LAYER_SCORES_BF16 1
/* csa2_layer_io.flags: a FULL layer's scan takes each indexer query as one
 * e4m3 operand per head (q_h scaled by the power of two that puts its largest
 * element in [128, 256), rounded to e4m3: 4 significant bits) instead of two
 * (hi + lo, about 8, the precision of the bf16 query).  Fewer products per
 * key tile and one tensor-memory column per head to read; a trade outside the
 * fp32 parity rule, the counterpart for the index scan of the FP8 indexer
 * the pages describe ("DeepSeek-V4 report explainer" §3.2, §10.2): each score
 * then carries the query's e4m3 rounding (a relative error of order 2^-5 per
 * element), so near-ties at the Top-K threshold may resolve differently.
 * REINDEX layers and csa2_index_scores keep the two-part query. */
#define CSA2_LAYER_INDEX_E4M3_QUERY 2

/* Per-layer inputs, outputs and carried selection state for csa2_layer. */
typedef struct csa2_layer_io {
    const uint16_t *q;           /* bf16 [B*Q][64][512] attention queries      */
    const uint16_t *qi;          /* bf16 [B*Q][32][128] indexer queries        */
    const float    *w;           /* [B*Q][32] indexer head weights             */
    csa2_swa        swa;         /* this layer's window                        */
    float           sm_scale;    /* multiplies q.k (1 if q is pre-scaled)     */
    int32_t         flags;       /* CSA2_LAYER_* option bits (0: none)        */
    int32_t        *idx;         /* [B*Q][512] selection (written by FULL and
                                    REINDEX, read by every mode)              */
    int32_t        *pool;        /* [B*Q][16384] candidate pool (written by
                                    FULL, read by REINDEX: blocks of 8
                                    consecutive positions from multiples of 8,
                                    the last possibly shorter; a REINDEX pool
                                    not of that form has the offending blocks
                                    scored -inf and flagged CSA2_DEV_BAD_INDEX);
                                    16-byte aligned                           */
    int32_t        *pool_len;    /* [B*Q]                                     */
    float          *o;           /* [B*Q][64][512] attention output           */
    float          *lse;         /* [B*Q][64] natural-log sum of exp          */
    void           *prof_begin;  /* optional cudaEvent_t recorded on the stream
                                    just before the layer's index kernel (the
                                    Full scan / the Reindex pool rescoring and
                                    selection),
                                    as an external node when captured; NULL
                                    for none                                   */
    void           *prof_end;    /* optional cudaEvent_t recorded just after it */
} csa2_layer_io;

/* ---- compressor ----------------------------------------------------------
 * e_j[d] = sum_{i<m} softmax_i(Z[jm+i][d] + bias[i][d]) * C[jm+i][d]
 * [P3] §3.1 (softmax-weighted pooling of m tokens with a learned bias);
 * [P2] §2 (C, Z projected per layer), §3.1-3.2 (m = 2 encoder, m = 1 decoder,
 * no overlap, bias by offset within the group).
 *   C, Z  bf16 [n_tok][512];  bias fp32 [m][512];  out fp32 [n_tok/m][512].
 *   Trailing n_tok % m tokens are not compressed.  1 <= m <= 16.
 *   Computed in double precision and rounded once to fp32. */
CSA2_API int csa2_compress(const uint16_t *C, const uint16_t *Z, const float *bias, int32_t m,
                  int64_t n_tok, float *out, csa2_stream_t stream);

/* ---- MXFP4 quantisation of main-KV entries --------------------------------
 * Per 32-element block: X = floor(log2(amax)) - 2 (0 if amax == 0), clamped
 * to [-127, 127], stored as E8M0 byte X + 127; each element x becomes the
 * E2M1 value nearest to x * 2^-X (ties to even mantissa, saturating at 6),
 * its sign bit copying x's.  [P2] §4; OCP MX block 32 / E8M0.
 *   x      fp32 [n][512] (finite values), n <= 2^31 - 1 (CSA2_ERR_SHAPE beyond)
 *   slots  int64 [n] destination slot of each row, or NULL for row i -> slot i;
 *          a negative slot skips the row; a slot >= num_slots is skipped and
 *          flagged CSA2_DEV_BAD_SLOT in *status (status may be NULL).
 *   codes  [num_slots][256], scales [num_slots][16]  (a csa2_cache's kv_*). */
CSA2_API int csa2_quant_mxfp4(const float *x, int64_t n, const int64_t *slots, uint8_t *codes,
                     uint8_t *scales, int64_t num_slots, int32_t *status, csa2_stream_t stream);

/* FP4 main KV with one E4M3 scale per 16-element block ([P2] §4 and [P4]:
 * "16 channels share one E4M3 scale"; csa2_cache.kv_format CSA2_KV_FP4_E4M3).
 * Per block: s = e4m3(amax / 6) (one fp32 IEEE division, then round to
 * nearest even, saturating at 448); each element x becomes e2m1(x / s) (one
 * fp32 IEEE division, nearest E2M1 value, ties to even, saturating at 6, sign
 * bit copied); a block whose scale rounds to zero keeps only the sign bits.
 *   x, slots, status, errors as csa2_quant_mxfp4;
 *   codes  [num_slots][256] (same nibble order), scales [num_slots][32]. */
CSA2_API int csa2_quant_fp4_e4m3(const float *x, int64_t n, const int64_t *slots, uint8_t *codes,
                        uint8_t *scales, int64_t num_slots, int32_t *status, csa2_stream_t stream);

/* ---- FP8 e4m3 quantisation with a per-row fp32 scale ---------------------
 * s = amax / 448 (IEEE fp32 division; s = 1 when amax == 0); each element
 * code = e4m3(x / s) (IEEE fp32 division, round to nearest even, saturating
 * at 448, sign kept).  Used for the SWA rows ([P1] §3.3, [P2] §4) and the
 * indexer keys.
 *   x fp32 [n][dim], dim in {128, 512}, n <= 2^31 - 1; slots as for csa2_quant_mxfp4;
 *   codes [num_slots][dim], scales [num_slots]. */
CSA2_API int csa2_quant_fp8(const float *x, int64_t n, int32_t dim, const int64_t *slots, uint8_t *codes,
                   float *scales, int64_t num_slots, int32_t *status, csa2_stream_t stream);

/* ---- a step's new entries into the cache, in one launch ------------------
 * The compressor, the main-KV quantiser of cache->kv_format and the FP8
 * quantiser of the indexer keys for the n_tok / m entries that n_tok new
 * tokens make ([P3] §3.1, [P2] §3.2 and §4): the same results, bit for bit,
 * as csa2_compress, then csa2_quant_mxfp4 (or csa2_quant_fp4_e4m3) of its
 * output and csa2_quant_fp8 (dim 128) of ik, each at the entry's slot.
 *   cache    kv_codes, kv_scales, ik_codes, ik_scales, num_slots, kv_format
 *            and status as for csa2_layer (block_table unused but checked)
 *   C, Z     bf16 [n_tok][512];  bias fp32 [m][512];  1 <= m <= 16
 *   ik       fp32 [n_tok / m][128], 16-byte aligned: each entry's indexer key
 *   slots    int64 [n_tok / m]: a negative slot skips the entry; a slot >=
 *            num_slots is skipped and flagged CSA2_DEV_BAD_SLOT; NULL: entry
 *            i -> slot i (CSA2_ERR_RANGE if that overruns the cache)
 *   entries  fp32 [n_tok / m][512] copy of the compressed entries, or NULL */
CSA2_API int csa2_append_entries(const csa2_cache *cache, const uint16_t *C, const uint16_t *Z,
                                 const float *bias, int32_t m, int64_t n_tok, const float *ik,
                                 const int64_t *slots, float *entries, csa2_stream_t stream);

/* ---- RMSNorm and forward partial RoPE of the attention inputs ------------
 * [P3] §4.3: queries and compressed KV are RMS-normalised before the core
 * attention, and RoPE acts on the last 64 of the 512 dims only (the output is
 * rotated back by csa2_swa.rope_base).  For every 512-dim vector x of row r
 * (vecs vectors per row, all at token position pos[r]):
 *   y = x / sqrt(mean_d(x_d^2) + eps) * gamma
 *   then, when rope_base > 0, for i < 32 the pair (y[448+i], y[480+i]) is
 *   rotated by +pos[r] * rope_base^(-i/32):  (a, b) -> (a cos - b sin,
 *   a sin + b cos) -- the inverse of the output rotation of csa2_swa.
 * Queries: rows = B*Q tokens, vecs = 64 heads, bf16 output (csa2_layer_io.q).
 * KV: rows = entries, vecs = 1, fp32 output for the quantisers; the position
 * of a compressed entry is the caller's choice.
 *   x        fp32 [rows][vecs][512], 16-byte aligned; may equal out_f32
 *   gamma    fp32 [512] RMSNorm weight, 16-byte aligned, or NULL for ones
 *   eps      >= 0, finite
 *   pos      int64 [rows] (may be NULL when rope_base == 0)
 *   out_f32  fp32 [rows][vecs][512] (16-byte aligned) or NULL
 *   out_bf16 bf16 [rows][vecs][512] (8-byte aligned) or NULL: exactly one of
 *            the two outputs (CSA2_ERR_NULL otherwise)
 * Computed in fp32 (IEEE square root and division); each angle is reduced
 * modulo 2π exactly as a 64-bit integer count of turns before its sine and
 * cosine are taken in fp32; the bf16 output is rounded to nearest even.
 * CSA2_ERR_SHAPE for rows < 0, vecs < 1, rows * vecs >= 2^34, eps or
 * rope_base negative or not finite. */
CSA2_API int csa2_norm_rope(const float *x, int64_t rows, int32_t vecs, const float *gamma, float eps,
                   const int64_t *pos, float rope_base, float *out_f32, uint16_t *out_bf16,
                   csa2_stream_t stream);

/* ---- lightning-indexer scores over every visible entry -------------------
 * score(p) = sum_h w[h] * ReLU(qi[h] . k_p), k_p = e4m3(code_p) * scale_p,
 * for every entry p visible to each query; block_max[b8] = max over the
 * visible positions of block b8 (positions 8*b8 .. 8*b8+7).
 * [P3] §3.2 (low-dimensional query against compressed index keys);
 * [P1] §3.2 and [P2] §3.2 (block aggregation of index scores, blocks of 8).
 *   qi bf16 [B*Q][32][128]; w fp32 [B*Q][32]
 *   scores     fp32 [B*Q][ld] or NULL (positions >= visible are not written)
 *   block_max  fp32 [B*Q][ld/8] or NULL (at least one of the two non-NULL)
 *   n_visible  int32 [B*Q] visible entries per query, or NULL
 *   ld         row stride, multiple of 8, >= batch->max_entries. */
CSA2_API int csa2_index_scores(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *qi,
                      const float *w, float *scores, float *block_max, int32_t *n_visible,
                      int64_t ld, csa2_stream_t stream);

/* Reindex variant ([P2] §3.2: later layers rescore only the pool): scores of
 * the entries listed in pool[r][0 .. pool_len[r]), by the kernels a Reindex
 * layer uses: the pool's indexer keys are gathered into dense rows of the
 * workspace, then scanned like the cache.
 *   pool int32 [B*Q][ld] positions; pool_len int32 [B*Q] (clamped to [0, ld]);
 *   scores fp32 [B*Q][ld] (slot i of row r = score of pool[r][i]; a position
 *   at or beyond the query's visible entries, or on a page outside the cache,
 *   scores -inf and is flagged CSA2_DEV_BAD_INDEX / CSA2_DEV_BAD_PAGE);
 *   ld a multiple of 64, <= 2^24 (CSA2_ERR_SHAPE otherwise);
 *   workspace >= csa2_index_scores_pool_workspace_size(batch, ld) bytes,
 *   256-byte aligned (CSA2_ERR_WORKSPACE / CSA2_ERR_ALIGN otherwise). */
CSA2_API int csa2_index_scores_pool(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *qi,
                           const float *w, const int32_t *pool, const int32_t *pool_len,
                           int64_t ld, float *scores, void *workspace, size_t workspace_bytes,
                           csa2_stream_t stream);

/* Workspace of csa2_index_scores_pool: B*Q*ld*132 bytes (rounded up to 256-byte
 * sections); 0 for an invalid batch or ld. */
CSA2_API size_t csa2_index_scores_pool_workspace_size(const csa2_batch *batch, int64_t ld);

/* ---- Top-K selection ---------------------------------------------------
 * For each of `rows` rows: the k slots i < len[r] with the largest scores
 * (ties -> lower slot), reported as positions (cand[r][i] when cand is
 * non-NULL, else i) in ascending order, the rest of out[r][0..k) set to -1.
 * With ascending cand rows, "lower slot" is "lower position".  -0.0 and +0.0
 * compare equal.  [P2] §1 table (top-k 512), §3.2 ("its own Top-512").
 *   scores fp32 [rows][ld]; len int32 [rows] (clamped to [0, ld]);
 *   cand int32 [rows][ld] or NULL; out int32 [rows][k]; 1 <= k <= 4096;
 *   ld <= 131072 (CSA2_ERR_SHAPE otherwise). */
CSA2_API int csa2_topk(const float *scores, int64_t ld, const int32_t *len, int32_t rows,
              const int32_t *cand, int32_t k, int32_t *out, csa2_stream_t stream);

/* Block level of the hierarchy ([P1] §3.2, [P2] §3.2): for each row keep the
 * pmax blocks with the largest block_max (ties -> lower block) among the
 * ceil(n_visible[r] / 8) blocks, and write all their visible positions in
 * ascending order to pool[r] (pool_len[r] of them).
 *   block_max fp32 [rows][ld_blocks]; n_visible int32 [rows];
 *   pool int32 [rows][pmax*8]; pool_len int32 [rows]; 1 <= pmax <= 2048;
 *   ld_blocks <= 131072, i.e. at most 1,048,576 visible entries (the pages'
 *   maximum context; CSA2_ERR_SHAPE otherwise). */
CSA2_API int csa2_topk_blocks(const float *block_max, int64_t ld_blocks, const int32_t *n_visible,
                     int32_t rows, int32_t pmax, int32_t *pool, int32_t *pool_len,
                     csa2_stream_t stream);

/* ---- sparse MQA + SWA attention ------------------------------------------
 * For each query (b, i) at token t: key set = the selected entries
 * idx[r][0..k) != -1 (MXFP4 main KV, dequantised exactly) followed by the
 * window rows of tokens [max(s, t-127), t] (FP8, times the row scale); each
 * key is also its value ([P3] §4.3).  For every head h:
 *   l_j = sm_scale * q_h . k_j,  o_h = sum_j softmax(l)_j k_j,
 *   lse_h = log sum_j exp(l_j);  an empty key set gives o_h = 0, lse_h = -inf.
 * One softmax covers both branches ([P2] §1 table, §3; [P3] §3.3).
 *   q bf16 [B*Q][64][512]; idx int32 [B*Q][k], 1 <= k <= 512 (an index at
 *   or beyond the query's visible entries is skipped and flagged
 *   CSA2_DEV_BAD_INDEX); o fp32 [B*Q][64][512]; lse fp32 [B*Q][64]. */
CSA2_API int csa2_sparse_attn(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *q,
                     float sm_scale, const int32_t *idx, int32_t k, const csa2_swa *swa,
                     float *o, float *lse, void *workspace, size_t workspace_bytes,
                     csa2_stream_t stream);

CSA2_API size_t csa2_sparse_attn_workspace_size(int32_t batch, int32_t nq);

/* The schedule csa2_sparse_attn and csa2_layer take for these arguments
 * (CSA2_ATTN_SCHEDULE_CHUNKS: two launches, the attention and its merge;
 * CSA2_ATTN_SCHEDULE_ROWS: one), or a negative CSA2_ERR_* for arguments the
 * calls would refuse (swa->codes and swa->scales must be non-NULL; nothing is
 * dereferenced on the device).  Host only. */
CSA2_API int csa2_sparse_attn_schedule(const csa2_batch *batch, const csa2_swa *swa);

/* ---- a10: one CSA2 layer ---------------------------------------------------
 * mode CSA2_MODE_FULL    : index every visible entry, pool of the best 2,048
 *                          blocks of 8, Top-512 of the pool -> io->idx,
 *                          io->pool, io->pool_len; attention.
 *      CSA2_MODE_REINDEX : rescore io->pool with this layer's (qi, w),
 *                          Top-512 -> io->idx; attention.
 *      CSA2_MODE_REUSE   : attention with io->idx as it is.
 * [P2] §3 mode table and §3.2; [P1] §3.2.  The main KV and the indexer keys
 * are the cache's (the latest Full layer's).  A Full layer takes at most
 * 1,048,576 entries (batch->max_entries).  workspace must hold
 * csa2_layer_workspace_size(mode, batch) bytes, 256-byte aligned. */
CSA2_API int csa2_layer(int32_t mode, const csa2_cache *cache, const csa2_batch *batch,
               const csa2_layer_io *io, void *workspace, size_t workspace_bytes,
               csa2_stream_t stream);

/* The workspace a csa2_layer call of this mode needs; 0 for invalid arguments. */
CSA2_API size_t csa2_layer_workspace_size(int32_t mode, const csa2_batch *batch);

/* ---- allocation-free layer call --------------------------------------------
 * No counterpart in the source pages: a library convenience for callers that
 * cannot allocate device memory per call (a plugin whose host program owns
 * every device allocation, a serving loop that allocates nothing after
 * start-up).  Same computation and arguments as csa2_layer without the
 * workspace: the scratch is one static device array of
 * CSA2_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library, held on
 * every GPU that loads the library until the process exits.
 * - Returns CSA2_ERR_WORKSPACE, before any device work, when the scratch this
 *   call needs exceeds CSA2_NOALLOC_SCRATCH_BYTES (for example a Full layer
 *   over 8 x 1M entries); use csa2_layer there.  A Reuse layer needs only the
 *   attention's scratch (about 5.3 MB at 8 query rows), a Reindex layer that
 *   plus 64 KB per query row for its rescored pool (about 5.8 MB).
 * - Returns CSA2_ERR_UNSUPPORTED, before any device work, for
 *   CSA2_ATTN_EARLY_ALL in io->swa.flags: that option needs a workspace that
 *   differs from the previous call's, and every call here shares one. 
 * - The first call on a device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress); make that first call before any
 *   stream capture.  `stream` must belong to the current device.  The cached
 *   address is good for the life of the device's primary context: after
 *   cudaDeviceReset, do not call this entry point again in the process.
 * - Every call on a device shares the one array, which keeps the previous
 *   call's contents (nothing in it needs to start at zero).  Calls whose
 *   work overlaps on the GPU (other streams, other host threads) race on it
 *   and corrupt each other's results: serialise them. */
#define CSA2_NOALLOC_SCRATCH_BYTES (16u << 20)
CSA2_API int csa2_layer_noalloc(int32_t mode, const csa2_cache *cache, const csa2_batch *batch,
                                const csa2_layer_io *io, csa2_stream_t stream);

/* ---- failure-path test hook ------------------------------------------------
 * No counterpart in the source pages.  Every wait of the tensor-core kernels
 * (the index scan's pipeline, the attention's products) gives up after a
 * bounded number of polls: the kernel then skips the work that depended on
 * it, sets CSA2_DEV_TIMEOUT in the cache's status word and returns normally
 * (its in-flight copies and products are still awaited with a long limit
 * before its shared and tensor memory are released, so the context stays
 * usable; outputs of that call are undefined).  This sets the poll count for
 * launches made after it, process-wide (0 restores the default of 2^24, about
 * a second); a small count makes those waits run out, which is how the tests
 * drive the timeout path without a fault. */
CSA2_API int csa2_debug_set_wait_limit(uint32_t polls);

/* ---- errors -------------------------------------------------------------- */
CSA2_API const char *csa2_status_string(int32_t status);   /* static string, never NULL */
CSA2_API int32_t     csa2_last_cuda_error(void);           /* cudaError_t of the last
                                                     CSA2_ERR_CUDA on this thread */

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
