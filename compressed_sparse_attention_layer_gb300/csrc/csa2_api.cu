// extern "C" entry points of csa2.h: host-side validation, workspace layout,
// kernel launches and the per-layer driver.  No entry point allocates memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "csa2_internal.cuh"

namespace csa2 {

static thread_local int g_last_cuda_error = 0;
void set_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

// ---------------------------------------------------------------- per-device set-up
namespace {
constexpr int kMaxDevices = 64;
struct KernelAttr {
    int dev;
    const void *fn;
    size_t bytes;
};
std::mutex g_dev_mu;
std::vector<KernelAttr> g_kernel_attrs;     // (device, kernel) limits already raised
int g_dev_sms[kMaxDevices] = {};
}  // namespace

int kernel_smem_limit(const void *kernel, size_t bytes, int carveout)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    for (const KernelAttr &a : g_kernel_attrs)
        if (a.dev == dev && a.fn == kernel && a.bytes >= bytes) return CSA2_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && carveout >= 0)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    for (KernelAttr &a : g_kernel_attrs)
        if (a.dev == dev && a.fn == kernel) {
            a.bytes = bytes;
            return CSA2_OK;
        }
    g_kernel_attrs.push_back({dev, kernel, bytes});
    return CSA2_OK;
}

static constexpr uint32_t kDefaultWaitPolls = 1u << 24;
static std::atomic<uint32_t> g_wait_polls{kDefaultWaitPolls};
uint32_t wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

int device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (dev < kMaxDevices && g_dev_sms[dev] > 0) return g_dev_sms[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) g_dev_sms[dev] = n;
    return n;
}

// launchers defined in the kernel files
int launch_compress(const uint16_t *, const uint16_t *, const float *, int, int64_t, float *, cudaStream_t);
int launch_quant_mxfp4(const float *, int64_t, const int64_t *, uint8_t *, uint8_t *, int64_t, int32_t *,
                       cudaStream_t);
int launch_quant_fp8(const float *, int64_t, int, const int64_t *, uint8_t *, float *, int64_t, int32_t *,
                     cudaStream_t);
int launch_quant_fp4_e4m3(const float *, int64_t, const int64_t *, uint8_t *, uint8_t *, int64_t, int32_t *,
                          cudaStream_t);
int launch_append_entries(const uint16_t *, const uint16_t *, const float *, int, int64_t, const float *,
                          const int64_t *, const csa2_cache &, float *, cudaStream_t);
int launch_norm_rope(const float *, int64_t, int, const float *, float, const int64_t *, float, float *, uint16_t *,
                     cudaStream_t);
int launch_index_scan(const csa2_cache &, const csa2_batch &, const uint16_t *, const float *, float *,
                      float *, int32_t *, int64_t, cudaStream_t, bool bf16_scores = false,
                      bool one_part_query = false);
int launch_gather_pool(const csa2_cache &, const csa2_batch &, const int32_t *, const int32_t *, int64_t, uint8_t *,
                       float *, cudaStream_t);
int launch_index_dense(const uint8_t *, const float *, const csa2_batch &, const uint16_t *, const float *,
                       const int32_t *, int64_t, float *, cudaStream_t, bool bf16_scores = false);
int launch_topk(const float *, int64_t, const int32_t *, int32_t, const int32_t *, int32_t, int32_t *,
                cudaStream_t);
int launch_reindex(const csa2_cache &, const csa2_batch &, const uint16_t *, const float *, const int32_t *,
                   const int32_t *, int, int32_t *, bool, void *, cudaStream_t);
size_t reindex_workspace_bytes(int64_t rows);
int launch_topk_blocks(const float *, int64_t, const int32_t *, int32_t, int32_t, int32_t *, int32_t *,
                       cudaStream_t, const PoolKeys * = nullptr, int * = nullptr);
int launch_pool_select(const int32_t *, const int32_t *, const uint32_t *, const uint2 *, int, int, int32_t *, int64_t,
                       cudaStream_t);
int launch_attn(const csa2_cache &, const csa2_batch &, const uint16_t *, float, const int32_t *, int,
                const csa2_swa &, float *, float *, void *, size_t, cudaStream_t, int);
size_t attn_workspace_bytes(int64_t rows);
bool attn_by_rows(int64_t rows, const csa2_swa &swa);
int topk_max_k();
int64_t topk_max_len();

// ---------------------------------------------------------------- validation
static constexpr int64_t kMaxRows = 65535;

static int check_cache(const csa2_cache *c, bool need_kv, bool need_ik)
{
    if (!c || !c->block_table) return CSA2_ERR_NULL;
    if (need_kv && (!c->kv_codes || !c->kv_scales)) return CSA2_ERR_NULL;
    if (need_ik && (!c->ik_codes || !c->ik_scales)) return CSA2_ERR_NULL;
    if (c->num_slots <= 0 || c->num_slots % CSA2_PAGE || c->max_pages <= 0) return CSA2_ERR_SHAPE;
    if (c->kv_format != CSA2_KV_MXFP4 && c->kv_format != CSA2_KV_FP4_E4M3) return CSA2_ERR_UNSUPPORTED;
    if (need_kv && (!aligned(c->kv_codes, 16) || !aligned(c->kv_scales, 16))) return CSA2_ERR_ALIGN;
    if (need_ik && (!aligned(c->ik_codes, 16) || !aligned(c->ik_scales, 16))) return CSA2_ERR_ALIGN;
    return CSA2_OK;
}

static int check_batch(const csa2_batch *b, const csa2_cache *c)
{
    if (!b || !b->n_entries || !b->q_pos) return CSA2_ERR_NULL;
    if (b->batch < 1 || b->nq < 1 || b->m < 1 || b->m > 16 || b->max_entries < 0) return CSA2_ERR_SHAPE;
    if ((int64_t)b->batch * b->nq > kMaxRows) return CSA2_ERR_SHAPE;
    if (c && b->max_entries > (int64_t)c->max_pages * CSA2_PAGE) return CSA2_ERR_RANGE;
    if (b->max_entries > (int64_t)INT32_MAX) return CSA2_ERR_RANGE;
    return CSA2_OK;
}

static int check_swa(const csa2_swa *s, const csa2_batch *b)
{
    if (!s || !s->codes || !s->scales) return CSA2_ERR_NULL;
    if (s->rows < CSA2_SWA_WINDOW) return CSA2_ERR_SHAPE;
    if (!aligned(s->codes, 16)) return CSA2_ERR_ALIGN;
    if (s->flags & ~(CSA2_ATTN_DEDUP_WINDOW | CSA2_ATTN_EARLY_INPUTS | CSA2_ATTN_SCHEDULE_CHUNKS |
                     CSA2_ATTN_SCHEDULE_ROWS | CSA2_ATTN_EARLY_ALL))
        return CSA2_ERR_UNSUPPORTED;
    if ((s->flags & CSA2_ATTN_SCHEDULE_CHUNKS) && (s->flags & CSA2_ATTN_SCHEDULE_ROWS)) return CSA2_ERR_UNSUPPORTED;
    if (!(s->rope_base >= 0.0f)) return CSA2_ERR_SHAPE;           // negative or NaN
    if (s->new_rows) {
        // the window of a query in a multi-token chunk holds other new tokens, which
        // must be in the ring before any query attends: quantise them first instead
        if (b->nq != 1) return CSA2_ERR_UNSUPPORTED;
        if (!aligned(s->new_rows, 16)) return CSA2_ERR_ALIGN;
    }
    return CSA2_OK;
}

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static inline int64_t score_ld(const csa2_batch *b)
{
    int64_t ld = (b->max_entries + 7) / 8 * 8;
    return ld > 0 ? ld : 8;
}

// FULL workspace:    scores [rows][ld] | block_max [rows][ld/8] | n_visible [rows]
//                    | the pool's keys [rows][16384] and bounds | attention workspace
// REINDEX workspace: the pool's rescored keys [rows][16384] and group minima
//                    | attention workspace
// REUSE workspace:   attention workspace
struct LayerWs {
    float *scores = nullptr, *block_max = nullptr;
    int32_t *n_visible = nullptr;
    void *rx = nullptr;
    void *attn = nullptr;
    size_t attn_bytes = 0, total = 0;
};

static LayerWs layer_ws(int32_t mode, const csa2_batch *b, void *base)
{
    LayerWs w;
    const int64_t rows = (int64_t)b->batch * b->nq;
    const int64_t ld = score_ld(b);
    size_t off = 0;
    char *p = static_cast<char *>(base);
    auto take = [&](size_t bytes) {
        void *q = p ? p + off : nullptr;
        off += align256(bytes);
        return q;
    };
    if (mode == CSA2_MODE_FULL) {
        w.scores = (float *)take((size_t)rows * ld * 4);
        w.block_max = (float *)take((size_t)rows * (ld / 8) * 4);
        w.n_visible = (int32_t *)take((size_t)rows * 4);
    }
    if (mode != CSA2_MODE_REUSE) w.rx = take(reindex_workspace_bytes(rows));
    w.attn_bytes = attn_workspace_bytes(rows);
    w.attn = take(w.attn_bytes);
    w.total = off;
    return w;
}

// Workspace a csa2_layer call with these arguments needs.
size_t layer_workspace_need(int32_t mode, const csa2_batch *b, const csa2_layer_io *)
{
    if (!b || b->batch < 1 || b->nq < 1 || mode < 0 || mode > 2) return 0;
    return layer_ws(mode, b, nullptr).total;
}

}  // namespace csa2

using namespace csa2;

extern "C" {

const char *csa2_status_string(int32_t s)
{
    switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_NULL: return "a required pointer is NULL";
    case CSA2_ERR_SHAPE: return "a size or count is out of range";
    case CSA2_ERR_UNSUPPORTED: return "unsupported argument";
    case CSA2_ERR_RANGE: return "an index or length exceeds its buffer";
    case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA2_ERR_TIMEOUT: return "a bounded device wait timed out";
    case CSA2_ERR_CUDA: return "a CUDA call failed";
    case CSA2_ERR_ALIGN: return "a pointer is not suitably aligned";
    default: return "unknown status";
    }
}

int32_t csa2_last_cuda_error(void) { return g_last_cuda_error; }

int csa2_debug_set_wait_limit(uint32_t polls)
{
    g_wait_polls.store(polls ? polls : kDefaultWaitPolls, std::memory_order_relaxed);
    return CSA2_OK;
}

int csa2_compress(const uint16_t *C, const uint16_t *Z, const float *bias, int32_t m, int64_t n_tok,
                  float *out, csa2_stream_t stream)
{
    if (m < 1 || m > 16 || n_tok < 0) return CSA2_ERR_SHAPE;
    if (n_tok / m == 0) return CSA2_OK;
    if (!C || !Z || !bias || !out) return CSA2_ERR_NULL;
    return launch_compress(C, Z, bias, m, n_tok, out, (cudaStream_t)stream);
}

int csa2_quant_mxfp4(const float *x, int64_t n, const int64_t *slots, uint8_t *codes, uint8_t *scales,
                     int64_t num_slots, int32_t *status, csa2_stream_t stream)
{
    if (n < 0 || n > INT32_MAX || num_slots < 0) return CSA2_ERR_SHAPE;
    if (n == 0) return CSA2_OK;
    if (!x || !codes || !scales) return CSA2_ERR_NULL;
    if (!slots && n > num_slots) return CSA2_ERR_RANGE;
    if (!aligned(x, 16) || !aligned(codes, 16)) return CSA2_ERR_ALIGN;
    return launch_quant_mxfp4(x, n, slots, codes, scales, num_slots, status, (cudaStream_t)stream);
}

int csa2_quant_fp4_e4m3(const float *x, int64_t n, const int64_t *slots, uint8_t *codes, uint8_t *scales,
                        int64_t num_slots, int32_t *status, csa2_stream_t stream)
{
    if (n < 0 || n > INT32_MAX || num_slots < 0) return CSA2_ERR_SHAPE;
    if (n == 0) return CSA2_OK;
    if (!x || !codes || !scales) return CSA2_ERR_NULL;
    if (!slots && n > num_slots) return CSA2_ERR_RANGE;
    if (!aligned(x, 16) || !aligned(codes, 16)) return CSA2_ERR_ALIGN;
    return launch_quant_fp4_e4m3(x, n, slots, codes, scales, num_slots, status, (cudaStream_t)stream);
}

int csa2_quant_fp8(const float *x, int64_t n, int32_t dim, const int64_t *slots, uint8_t *codes,
                   float *scales, int64_t num_slots, int32_t *status, csa2_stream_t stream)
{
    if (n < 0 || n > INT32_MAX || num_slots < 0 || (dim != 128 && dim != 512)) return CSA2_ERR_SHAPE;
    if (n == 0) return CSA2_OK;
    if (!x || !codes || !scales) return CSA2_ERR_NULL;
    if (!slots && n > num_slots) return CSA2_ERR_RANGE;
    if (!aligned(x, 16) || !aligned(codes, 4)) return CSA2_ERR_ALIGN;
    return launch_quant_fp8(x, n, dim, slots, codes, scales, num_slots, status, (cudaStream_t)stream);
}

int csa2_append_entries(const csa2_cache *cache, const uint16_t *C, const uint16_t *Z, const float *bias, int32_t m,
                        int64_t n_tok, const float *ik, const int64_t *slots, float *entries, csa2_stream_t stream)
{
    if (m < 1 || m > 16 || n_tok < 0) return CSA2_ERR_SHAPE;
    const int64_t n_ent = n_tok / m;
    if (n_ent > INT32_MAX) return CSA2_ERR_SHAPE;
    if (n_ent == 0) return CSA2_OK;
    int s = check_cache(cache, true, true);
    if (s) return s;
    if (!C || !Z || !bias || !ik) return CSA2_ERR_NULL;
    if (!slots && n_ent > cache->num_slots) return CSA2_ERR_RANGE;
    if (!aligned(ik, 16) || (entries && !aligned(entries, 4))) return CSA2_ERR_ALIGN;
    return launch_append_entries(C, Z, bias, m, n_tok, ik, slots, *cache, entries, (cudaStream_t)stream);
}

int csa2_norm_rope(const float *x, int64_t rows, int32_t vecs, const float *gamma, float eps, const int64_t *pos,
                   float rope_base, float *out_f32, uint16_t *out_bf16, csa2_stream_t stream)
{
    if (rows < 0 || vecs < 1 || !(eps >= 0.0f) || !std::isfinite(eps) || !(rope_base >= 0.0f) ||
        !std::isfinite(rope_base) || rows > ((((int64_t)1 << 34) - 1) / vecs))   // rows * vecs < 2^34
        return CSA2_ERR_SHAPE;
    if (rows == 0) return CSA2_OK;
    if (!x || (!out_f32) == (!out_bf16) || (rope_base > 0.0f && !pos)) return CSA2_ERR_NULL;
    if (!aligned(x, 16) || (gamma && !aligned(gamma, 16)) || (out_f32 && !aligned(out_f32, 16)) ||
        (out_bf16 && !aligned(out_bf16, 8)))
        return CSA2_ERR_ALIGN;
    return launch_norm_rope(x, rows, vecs, gamma, eps, pos, rope_base, out_f32, out_bf16, (cudaStream_t)stream);
}

int csa2_index_scores(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *qi, const float *w,
                      float *scores, float *block_max, int32_t *n_visible, int64_t ld, csa2_stream_t stream)
{
    int s = check_cache(cache, false, true);
    if (s) return s;
    if ((s = check_batch(batch, cache))) return s;
    if (!qi || !w || (!scores && !block_max)) return CSA2_ERR_NULL;
    if (ld < batch->max_entries || ld % 8 || ld <= 0) return CSA2_ERR_SHAPE;
    return launch_index_scan(*cache, *batch, qi, w, scores, block_max, n_visible, ld, (cudaStream_t)stream);
}

// The pool's indexer keys gathered into dense rows of ld slots (codes, then
// scales), the layout the Reindex layers scan.
static size_t pool_keys_bytes(int64_t rows, int64_t ld)
{
    return align256((size_t)rows * ld * 128) + align256((size_t)rows * ld * 4);
}

size_t csa2_index_scores_pool_workspace_size(const csa2_batch *batch, int64_t ld)
{
    if (!batch || batch->batch < 1 || batch->nq < 1 || ld <= 0 || ld % CSA2_PAGE || ld > (int64_t)1 << 24) return 0;
    return pool_keys_bytes((int64_t)batch->batch * batch->nq, ld);
}

int csa2_index_scores_pool(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *qi,
                           const float *w, const int32_t *pool, const int32_t *pool_len, int64_t ld,
                           float *scores, void *workspace, size_t workspace_bytes, csa2_stream_t stream)
{
    int s = check_cache(cache, false, true);
    if (s) return s;
    if ((s = check_batch(batch, cache))) return s;
    if (!qi || !w || !pool || !pool_len || !scores) return CSA2_ERR_NULL;
    if (ld <= 0 || ld % CSA2_PAGE || ld > (int64_t)1 << 24) return CSA2_ERR_SHAPE;
    const int64_t rows = (int64_t)batch->batch * batch->nq;
    if (!workspace || workspace_bytes < pool_keys_bytes(rows, ld)) return CSA2_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return CSA2_ERR_ALIGN;
    const cudaStream_t st = (cudaStream_t)stream;
    uint8_t *codes = static_cast<uint8_t *>(workspace);
    float *kscales = reinterpret_cast<float *>(codes + align256((size_t)rows * ld * 128));
    // the same two kernels as a Reindex layer: gather the pool's keys, scan them densely
    if ((s = launch_gather_pool(*cache, *batch, pool, pool_len, ld, codes, kscales, st))) return s;
    return launch_index_dense(codes, kscales, *batch, qi, w, pool_len, ld, scores, st);
}

int csa2_topk(const float *scores, int64_t ld, const int32_t *len, int32_t rows, const int32_t *cand,
              int32_t k, int32_t *out, csa2_stream_t stream)
{
    if (rows < 0 || rows > kMaxRows * 16 || k < 1 || k > topk_max_k() || ld < 0) return CSA2_ERR_SHAPE;
    if (rows == 0) return CSA2_OK;
    if (!scores || !len || !out) return CSA2_ERR_NULL;
    if (ld > topk_max_len()) return CSA2_ERR_SHAPE;
    return launch_topk(scores, ld, len, rows, cand, k, out, (cudaStream_t)stream);
}

int csa2_topk_blocks(const float *block_max, int64_t ld_blocks, const int32_t *n_visible, int32_t rows,
                     int32_t pmax, int32_t *pool, int32_t *pool_len, csa2_stream_t stream)
{
    if (rows < 0 || rows > kMaxRows * 16 || pmax < 1 || pmax > CSA2_POOL_BLOCKS || ld_blocks < 0)
        return CSA2_ERR_SHAPE;
    if (rows == 0) return CSA2_OK;
    if (!block_max || !n_visible || !pool || !pool_len) return CSA2_ERR_NULL;
    if (ld_blocks > topk_max_len()) return CSA2_ERR_SHAPE;
    return launch_topk_blocks(block_max, ld_blocks, n_visible, rows, pmax, pool, pool_len,
                              (cudaStream_t)stream);
}

int csa2_sparse_attn_schedule(const csa2_batch *batch, const csa2_swa *swa)
{
    if (!batch || !swa) return CSA2_ERR_NULL;
    if (batch->batch < 1 || batch->nq < 1) return CSA2_ERR_SHAPE;
    if (const int s = check_swa(swa, batch)) return s;
    return attn_by_rows((int64_t)batch->batch * batch->nq, *swa) ? CSA2_ATTN_SCHEDULE_ROWS : CSA2_ATTN_SCHEDULE_CHUNKS;
}

size_t csa2_sparse_attn_workspace_size(int32_t batch, int32_t nq)
{
    if (batch < 1 || nq < 1) return 0;
    return attn_workspace_bytes((int64_t)batch * nq);
}

int csa2_sparse_attn(const csa2_cache *cache, const csa2_batch *batch, const uint16_t *q, float sm_scale,
                     const int32_t *idx, int32_t k, const csa2_swa *swa, float *o, float *lse,
                     void *workspace, size_t workspace_bytes, csa2_stream_t stream)
{
    int s = check_cache(cache, true, false);
    if (s) return s;
    if ((s = check_batch(batch, cache))) return s;
    if ((s = check_swa(swa, batch))) return s;
    if (!q || !idx || !o || !lse) return CSA2_ERR_NULL;
    if (k < 1 || k > CSA2_TOPK) return CSA2_ERR_SHAPE;
    const size_t need = attn_workspace_bytes((int64_t)batch->batch * batch->nq);
    if (need && (!workspace || workspace_bytes < need)) return CSA2_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 256)) return CSA2_ERR_ALIGN;
    if (!aligned(q, 16) || !aligned(o, 16)) return CSA2_ERR_ALIGN;
    return launch_attn(*cache, *batch, q, sm_scale, idx, k, *swa, o, lse, workspace, workspace_bytes,
                       (cudaStream_t)stream, 0);
}

size_t csa2_layer_workspace_size(int32_t mode, const csa2_batch *batch)
{
    return layer_workspace_need(mode, batch, nullptr);
}

int csa2_layer(int32_t mode, const csa2_cache *cache, const csa2_batch *batch, const csa2_layer_io *io,
               void *workspace, size_t workspace_bytes, csa2_stream_t stream)
{
    if (mode < CSA2_MODE_FULL || mode > CSA2_MODE_REUSE) return CSA2_ERR_UNSUPPORTED;
    int s = check_cache(cache, true, mode != CSA2_MODE_REUSE);
    if (s) return s;
    if ((s = check_batch(batch, cache))) return s;
    if (!io) return CSA2_ERR_NULL;
    if ((s = check_swa(&io->swa, batch))) return s;
    if (!io->q || !io->idx || !io->o || !io->lse) return CSA2_ERR_NULL;
    if (mode != CSA2_MODE_REUSE && (!io->qi || !io->w || !io->pool || !io->pool_len)) return CSA2_ERR_NULL;
    if (io->flags & ~(CSA2_LAYER_SCORES_BF16 | CSA2_LAYER_INDEX_E4M3_QUERY)) return CSA2_ERR_UNSUPPORTED;
    const bool bf16 = (io->flags & CSA2_LAYER_SCORES_BF16) != 0;
    if (mode == CSA2_MODE_FULL && score_ld(batch) / 8 > topk_max_len()) return CSA2_ERR_SHAPE;
    if (mode != CSA2_MODE_REUSE && !aligned(io->pool, 16)) return CSA2_ERR_ALIGN;
    if (!aligned(io->q, 16) || !aligned(io->o, 16)) return CSA2_ERR_ALIGN;
    LayerWs ws = layer_ws(mode, batch, workspace);
    if (ws.total && (!workspace || workspace_bytes < ws.total)) return CSA2_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 256)) return CSA2_ERR_ALIGN;

    const cudaStream_t st = (cudaStream_t)stream;
    const int32_t rows = batch->batch * batch->nq;
    const int64_t ld = score_ld(batch);
    auto prof = [&](void *ev) {
        if (!ev) return CSA2_OK;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(st, &cs);
        if (e == cudaSuccess)
            e = cs == cudaStreamCaptureStatusActive
                    ? cudaEventRecordWithFlags((cudaEvent_t)ev, st, cudaEventRecordExternal)
                    : cudaEventRecord((cudaEvent_t)ev, st);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return CSA2_ERR_CUDA;
        }
        return CSA2_OK;
    };
    if (mode == CSA2_MODE_FULL) {
        // scores of every visible entry and the per-block maxima
        if ((s = prof(io->prof_begin))) return s;
        if ((s = launch_index_scan(*cache, *batch, io->qi, io->w, ws.scores, ws.block_max, ws.n_visible, ld, st,
                                   bf16, (io->flags & CSA2_LAYER_INDEX_E4M3_QUERY) != 0)))
            return s;
        if ((s = prof(io->prof_end))) return s;
        // the best 2,048 blocks of 8 -> candidate pool, with the pool's scores as
        // order keys and a lower bound of its 512th largest
        PoolKeys pk;
        pk.scores = ws.scores;
        pk.ld_scores = ld;
        pk.bf16 = bf16;
        pk.k = CSA2_TOPK;
        pk.keys = static_cast<uint32_t *>(ws.rx);
        pk.bound = reinterpret_cast<uint2 *>(pk.keys + (int64_t)rows * CSA2_POOL_MAX);
        pk.bound_ld = 32;
        int P = 0;
        if ((s = launch_topk_blocks(ws.block_max, ld / 8, ws.n_visible, rows, CSA2_POOL_BLOCKS, io->pool,
                                    io->pool_len, st, &pk, &P)))
            return s;
        // Top-512 of the pool (the Reindex layer's select)
        if ((s = launch_pool_select(io->pool, io->pool_len, pk.keys, pk.bound, P, CSA2_TOPK, io->idx, rows, st)))
            return s;
    } else if (mode == CSA2_MODE_REINDEX) {
        // rescore the pool (its blocks' keys read from the cache) with this
        // layer's indexer query and take its Top-512
        if ((s = prof(io->prof_begin))) return s;
        if ((s = launch_reindex(*cache, *batch, io->qi, io->w, io->pool, io->pool_len, CSA2_TOPK, io->idx, bf16,
                                ws.rx, st)))
            return s;
        if ((s = prof(io->prof_end))) return s;
    }
    // REUSE keeps io->idx as it is; the attention for every mode.
    // CSA2_ATTN_EARLY_INPUTS / _ALL are honoured in REUSE mode, where the indices come from an earlier layer call
    const int early = mode != CSA2_MODE_REUSE ? 0
                      : (io->swa.flags & CSA2_ATTN_EARLY_ALL) ? 2
                      : (io->swa.flags & CSA2_ATTN_EARLY_INPUTS) ? 1 : 0;
    return launch_attn(*cache, *batch, io->q, io->sm_scale, io->idx, CSA2_TOPK, io->swa, io->o, io->lse,
                       ws.attn, ws.attn_bytes, st, early);
}

}  // extern "C"
