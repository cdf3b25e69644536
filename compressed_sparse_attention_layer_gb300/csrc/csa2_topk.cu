// Top-K selection with ties broken toward the lower slot
// ("DeepSeek-V4.1-Flash 架构详解" §1 table: top-k 512; §3.2: the best 2,048
// blocks of 8 form the candidate pool, then the pool's own Top-512; the
// research note §3.2).
//
// Rows of up to 16,384 keys (csa2_topk) run on one CTA per row with the keys in
// registers (k_topk_rows; description below); the layers' pool Top-512 runs the
// Reindex select (csa2_reindex.cu) on keys the block level writes here.  The
// block level and generic rows longer than 16,384 keys use one thread-block
// cluster per row:
// the CL CTAs each stage one contiguous 1/CL of
// the row in shared memory as order-preserving 32-bit keys, read once from
// global memory.  A radix select
// finds the k-th largest key T: the digits are 11-bit fields of (key - kmin)
// from the top bit of the row's actual range (kmax - kmin), so that scores
// crowded into a few exponents still spread over all 2,048 bins; each CTA
// counts its slice, the histograms are summed through distributed shared
// memory, and every CTA takes the same decision.  An ordered compaction then
// writes every key > T and the lowest-slot keys == T: each CTA learns how many selected
// slots lie in the slices before its own from the cluster's counts, so the
// output comes out in ascending slot order without atomics deciding order.
#include "csa2_select.cuh"

namespace csa2 {

// Stage row[0 .. m) as order keys: 16-byte loads, many in flight.
__device__ __forceinline__ void stage_keys(uint32_t *keys, const float *row, int m)
{
    const int tid = threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        const int m4 = m >> 2;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
#pragma unroll 4
        for (int i = tid; i < m4; i += TK_THREADS) {
            const float4 v = __ldg(r4 + i);
            *reinterpret_cast<uint4 *>(keys + 4 * i) =
                make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        }
        for (int i = 4 * m4 + tid; i < m; i += TK_THREADS) keys[i] = order_key(__ldg(row + i));
    } else {
#pragma unroll 8
        for (int i = tid; i < m; i += TK_THREADS) keys[i] = order_key(__ldg(row + i));
    }
}

// Keys of one CTA's slice of a row of ld slots (its staged keys, then as many
// again for the compacted candidates): the dynamic shared memory is twice that.
__host__ __device__ __forceinline__ int64_t slice_cap(int64_t ld, int cl) { return ((ld + cl - 1) / cl + 3) & ~(int64_t)3; }

// Slice of a row of n keys held by cluster rank q: a multiple of 4 keys so
// that slices of 16-byte aligned rows stay aligned.
__device__ __forceinline__ void slice_of(int64_t n, int cl, int q, int64_t &lo, int &m)
{
    const int64_t slice = ((n + cl - 1) / cl + 3) & ~(int64_t)3;
    lo = q * slice < n ? q * slice : n;
    m = (int)((lo + slice < n ? lo + slice : n) - lo);
}

// ---------------------------------------------------------------- kernels
// Top-k slots of each row of scores (reported as cand positions when given).
template <int CL>
__global__ void __launch_bounds__(TK_THREADS) k_topk(const float *__restrict__ scores, int64_t ld,
                                                     const int32_t *__restrict__ len,
                                                     const int32_t *__restrict__ cand, int k,
                                                     int32_t *__restrict__ out)
{
    extern __shared__ uint32_t keys[];
    __shared__ TkShared sh;
    pdl_launch_dependents();
    pdl_wait();
    cg::cluster_group cluster = cg::this_cluster();
    const int64_t r = blockIdx.x / CL;
    const int q = (int)cluster.block_rank();
    int64_t n = len[r];
    n = n < 0 ? 0 : (n > ld ? ld : n);
    int64_t lo;
    int m;
    slice_of(n, CL, q, lo, m);
    stage_keys(keys, scores + r * ld + lo, m);
    __syncthreads();
    int32_t *o = out + r * k;
    const int32_t *cr = cand ? cand + r * ld : nullptr;
    cluster_select<CL>(cluster, keys, keys + slice_cap(ld, CL), lo, m, n, k, sh, [&](int j, int64_t i) {
        if (j < k) o[j] = cr ? cr[i] : (int32_t)i;
    });
    const int64_t nsel = n < k ? n : k;
    if (q == CL - 1)
        for (int64_t j = nsel + threadIdx.x; j < k; j += TK_THREADS) o[j] = -1;
}

// Block level of the hierarchy: the pmax best blocks -> their visible positions.
// With pkeys, also the pool's own selection input: the order keys of its slots'
// scores (pkeys[r][8 j + t] for block rank j; scores rows of ld_scores, fp32 or
// bf16) and, per CTA q of the cluster, (the smallest, the largest) block maximum
// it selected in pbound[r * bound_ld + q].  Every selected block holds a key
// equal to its maximum (the scan's block maximum is one of its scores), so with
// at least kbound selected blocks the smallest of those is a lower bound of the
// pool's kbound-th largest key; with fewer, the bound is 0 (none).
template <int CL>
__global__ void __launch_bounds__(TK_THREADS) k_topk_blocks(const float *__restrict__ block_max, int64_t ld_blocks,
                                                            const int32_t *__restrict__ n_visible, int pmax,
                                                            int32_t *__restrict__ pool,
                                                            int32_t *__restrict__ pool_len,
                                                            const void *__restrict__ scores, int64_t ld_scores,
                                                            int bf16, int kbound, uint32_t *__restrict__ pkeys,
                                                            uint2 *__restrict__ pbound, int bound_ld)
{
    extern __shared__ uint32_t keys[];
    __shared__ TkShared sh;
    pdl_launch_dependents();
    pdl_wait();
    cg::cluster_group cluster = cg::this_cluster();
    const int64_t r = blockIdx.x / CL;
    const int q = (int)cluster.block_rank();
    int64_t nv = n_visible[r];
    nv = nv < 0 ? 0 : (nv > ld_blocks * 8 ? ld_blocks * 8 : nv);
    const int64_t nb = (nv + 7) / 8;
    int64_t lo;
    int m;
    slice_of(nb, CL, q, lo, m);
    stage_keys(keys, block_max + r * ld_blocks + lo, m);
    __syncthreads();
    int32_t *pr = pool + r * (int64_t)pmax * 8;
    const int nsel = (int)(nb < pmax ? nb : pmax);
    uint32_t bmin = 0xFFFFFFFFu, bmax = 0u;          // this thread's selected block maxima
    cluster_select<CL>(cluster, keys, keys + slice_cap(ld_blocks, CL), lo, m, nb, pmax, sh, [&](int j, int64_t blk) {
        if (j >= pmax) return;
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const int64_t p = blk * 8 + t;
            if (p < nv) pr[(int64_t)j * 8 + t] = (int32_t)p;
        }
        if (j == nsel - 1) {                         // the last selected block sets the pool size
            const int64_t tail = nv - blk * 8 < 8 ? nv - blk * 8 : 8;
            pool_len[r] = (nsel - 1) * 8 + (int)tail;
        }
        if (pkeys) {
            uint32_t kv[8];
            if (bf16) {
                const uint4 h = __ldcg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(scores) +
                                                                       r * ld_scores + blk * 8));
                const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int t = 0; t < 8; t++) kv[t] = order_key(__uint_as_float((hw[t >> 1] >> (16 * (t & 1))) << 16));
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(scores) +
                                                                     r * ld_scores + blk * 8);
                const float4 a = __ldcg(src), b = __ldcg(src + 1);
                const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int t = 0; t < 8; t++) kv[t] = order_key(f[t]);
            }
#pragma unroll
            for (int t = 0; t < 8; t++)
                if (blk * 8 + t >= nv) kv[t] = 0u;   // past the visible entries (outside the pool)
            uint4 *dst = reinterpret_cast<uint4 *>(pkeys + (r * pmax + j) * 8);
            dst[0] = make_uint4(kv[0], kv[1], kv[2], kv[3]);
            dst[1] = make_uint4(kv[4], kv[5], kv[6], kv[7]);
            const uint32_t bk = keys[blk - lo];      // the block's maximum, as staged
            bmin = min(bmin, bk);
            bmax = max(bmax, bk);
        }
    });
    if (nsel == 0 && q == 0 && threadIdx.x == 0) pool_len[r] = 0;
    if (pkeys) {
        bmin = __reduce_min_sync(0xffffffffu, bmin);
        bmax = __reduce_max_sync(0xffffffffu, bmax);
        __syncthreads();                             // the select's shared state is no longer read
        if (threadIdx.x == 0) {
            sh.kmin = 0xFFFFFFFFu;
            sh.kmax = 0u;
        }
        __syncthreads();
        if ((threadIdx.x & 31) == 0) {
            atomicMin(&sh.kmin, bmin);
            atomicMax(&sh.kmax, bmax);
        }
        __syncthreads();
        if (threadIdx.x == 0) pbound[r * bound_ld + q] = make_uint2(nsel >= kbound ? sh.kmin : 0u, sh.kmax);
    }
}

// ---------------------------------------------------------------- one CTA per row, keys in registers
// Rows of up to RS_MAX = 16,384 keys: 1,024 threads hold 16 consecutive slots
// each (thread t: slots 16 t .. 16 t + 15) as order keys in registers.
//  1. A lower bound L of the k-th largest key (k <= 512): the 512 groups of
//     32 keys (one register index of one warp) each hold a key >= their
//     maximum, so at least 512 keys are >= L = the smallest group maximum.
//     Only keys >= L are counted below (typically a few percent of the row).
//  2. A radix select on (key - L) over [L, kmax], 11 bits per round from the
//     top, counted in one shared-memory histogram of 2,048 bins; the bin that
//     holds the k-th largest key is found by one block scan of the bin counts.
//     Once that bin holds at most 32 keys, one warp ranks them directly.
//  3. One packed block scan of (count > T, count == T) places every selected
//     slot: rank = slots above T before it + the ties before it, ties taken
//     lowest slot first -- so the output is in ascending slot order and
//     identical on every run.
constexpr int RS_THREADS = 1024;
constexpr int RS_PER = 16;
constexpr int RS_MAX = RS_THREADS * RS_PER;
constexpr int RS_BITS = 11;
constexpr int RS_BINS = 1 << RS_BITS;
constexpr int RS_GROUPS = RS_MAX / 32;         // groups of the lower bound (k <= RS_GROUPS)
constexpr int RS_DIRECT = 32;                  // a bin of at most this many keys is ranked directly

struct __align__(16) RsShared {
    uint32_t hist[RS_BINS];                    // digit counts of the round
    uint32_t warp_u[RS_THREADS / 32];          // block scan partials
    uint32_t wmin[RS_THREADS / 32], wmax[RS_THREADS / 32];
    uint32_t direct[RS_DIRECT];                // the keys of a small bin
    uint32_t ndirect;
    uint32_t digit, bin_count;
    int above;
    uint32_t T;
    int need_eq;
};

// Block-wide exclusive scan of one 32-bit value per thread (1,024 threads).
__device__ __forceinline__ uint32_t rs_exclusive_scan(uint32_t v, RsShared &sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.warp_u[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t s2 = sh.warp_u[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s2, o);
            if (lane >= o) s2 += y;
        }
        sh.warp_u[lane] = s2;                          // inclusive
    }
    __syncthreads();
    const uint32_t base = wid ? sh.warp_u[wid - 1] : 0u;
    __syncthreads();                                   // warp_u free for the next use
    return base + x - v;
}

// Top k (k >= 1) of the n valid keys key[] of this row (bit j of `valid`
// marks slot 16 t + j as valid); calls emit(rank, j) for every selected slot
// 16 t + j, ranks ascending with the slot.  Returns the number selected,
// min(n, k).
template <class Emit>
__device__ int rs_select(const uint32_t (&key)[RS_PER], uint32_t valid, int n, int k, RsShared &sh, Emit emit)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (n <= k) {                                      // everything valid is selected, in slot order
        uint32_t off = rs_exclusive_scan(__popc(valid), sh);
#pragma unroll
        for (int j = 0; j < RS_PER; j++)
            if (valid >> j & 1u) emit((int)off++, j);
        return n;
    }
    // ---- 1. group maxima (an invalid slot counts as key 0): L and kmax
    uint32_t gmin = 0xFFFFFFFFu, gmax = 0u;
#pragma unroll
    for (int j = 0; j < RS_PER; j++) {
        const uint32_t g = __reduce_max_sync(0xffffffffu, (valid >> j & 1u) ? key[j] : 0u);
        gmin = min(gmin, g);
        gmax = max(gmax, g);
    }
    if (lane == 0) {
        sh.wmin[wid] = gmin;
        sh.wmax[wid] = gmax;
    }
    if (tid == 0) sh.ndirect = 0u;
    __syncthreads();
    uint32_t L = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll 8
    for (int w = 0; w < RS_THREADS / 32; w++) {
        L = min(L, sh.wmin[w]);
        kmax = max(kmax, sh.wmax[w]);
    }
    if (k > RS_GROUPS) L = 0u;                         // the bound holds for k <= RS_GROUPS only
    // ---- 2. radix select over rel = key - L of the keys >= L
    uint32_t cand = 0;                                 // this thread's keys >= L
#pragma unroll
    for (int j = 0; j < RS_PER; j++) cand |= (uint32_t)((valid >> j & 1u) && key[j] >= L) << j;
    const uint32_t range = kmax - L;
    int top = range ? 32 - __clz(range) : 0;
    uint32_t prefix = 0, mask = 0;
    int kk = k;
    bool direct = false;
#pragma unroll 1
    while (top > 0) {
        const int width = top < RS_BITS ? top : RS_BITS;
        const int shift = top - width;
        const uint32_t dmask = (1u << width) - 1u;
        sh.hist[tid] = 0u;
        sh.hist[tid + RS_THREADS] = 0u;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < RS_PER; j++) {
            const uint32_t rel = key[j] - L;
            if ((cand >> j & 1u) && (rel & mask) == prefix) atomicAdd(&sh.hist[(rel >> shift) & dmask], 1u);
        }
        __syncthreads();
        // thread t: bins 2047 - 2t (higher) and 2046 - 2t; counts of the higher
        // bins by one exclusive scan in descending bin order
        const uint32_t c_hi = sh.hist[RS_BINS - 1 - 2 * tid], c_lo = sh.hist[RS_BINS - 2 - 2 * tid];
        const uint32_t ex = rs_exclusive_scan(c_hi + c_lo, sh);
        if (ex < (uint32_t)kk && ex + c_hi + c_lo >= (uint32_t)kk) {
            const bool hi = ex + c_hi >= (uint32_t)kk;
            sh.digit = (uint32_t)(RS_BINS - 1 - 2 * tid - (hi ? 0 : 1));
            sh.above = (int)(hi ? ex : ex + c_hi);
            sh.bin_count = hi ? c_hi : c_lo;
        }
        __syncthreads();
        prefix |= sh.digit << shift;
        mask |= dmask << shift;
        kk -= sh.above;
        top = shift;
        if (top > 0 && sh.bin_count <= (uint32_t)RS_DIRECT) {
            direct = true;
            break;
        }
        // digit, above and bin_count are rewritten only after another block barrier
    }
    uint32_t T;
    int need_eq;
    if (direct) {
        // the bin's keys (at most RS_DIRECT) into shared memory; one warp ranks them
#pragma unroll
        for (int j = 0; j < RS_PER; j++) {
            const uint32_t rel = key[j] - L;
            if ((cand >> j & 1u) && (rel & mask) == prefix) sh.direct[atomicAdd(&sh.ndirect, 1u)] = key[j];
        }
        __syncthreads();
        if (wid == 0) {
            const int nd = (int)sh.ndirect;
            const uint32_t v = lane < nd ? sh.direct[lane] : 0u;
            int gt = 0, ge = 0;
            for (int i = 0; i < nd; i++) {
                const uint32_t u = sh.direct[i];
                gt += u > v;
                ge += u >= v;
            }
            // the kk-th largest of the bin: fewer than kk above it, at least kk from it up
            if (lane < nd && gt < kk && ge >= kk) {
                sh.T = v;                              // every lane that matches holds the same value
                sh.need_eq = kk - gt;
            }
        }
        __syncthreads();
        T = sh.T;
        need_eq = sh.need_eq;
    } else {
        T = prefix + L;
        need_eq = kk;                                  // ties with T that are selected, lowest slots first
    }
    // ---- 3. placement
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < RS_PER; j++)
        if (valid >> j & 1u) {
            gt += key[j] > T;
            eq += key[j] == T;
        }
    const uint32_t pre = rs_exclusive_scan((gt << 16) | eq, sh);   // both sums <= 16,384
    const int gt_prior = (int)(pre >> 16), eq_prior = (int)(pre & 0xFFFFu);
    int take = need_eq - eq_prior;
    take = take < 0 ? 0 : (take > (int)eq ? (int)eq : take);
    int off = gt_prior + (eq_prior < need_eq ? eq_prior : need_eq);
#pragma unroll
    for (int j = 0; j < RS_PER; j++) {
        if (!(valid >> j & 1u)) continue;
        if (key[j] > T) {
            emit(off++, j);
        } else if (key[j] == T && take > 0) {
            emit(off++, j);
            take--;
        }
    }
    return k;
}

// Slots 16 t .. 16 t + 15 of a row of n scores as order keys.  Returns the
// valid mask (slots < n).
__device__ __forceinline__ uint32_t rs_load(const float *__restrict__ row, int n, uint32_t (&key)[RS_PER])
{
    const int s0 = RS_PER * threadIdx.x;
    if (s0 + RS_PER <= n && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
#pragma unroll
        for (int q = 0; q < RS_PER / 4; q++) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(row + s0) + q);
            key[4 * q] = order_key(v.x);
            key[4 * q + 1] = order_key(v.y);
            key[4 * q + 2] = order_key(v.z);
            key[4 * q + 3] = order_key(v.w);
        }
        return 0xFFFFu;
    }
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < RS_PER; j++) {
        key[j] = 0u;
        if (s0 + j < n) {
            key[j] = order_key(__ldg(row + s0 + j));
            valid |= 1u << j;
        }
    }
    return valid;
}

// Top k of each row (one CTA per row, len[r] <= RS_MAX slots of scores[r]),
// reported as cand[r][i] (or i) ascending, -1 after.
__global__ void __launch_bounds__(RS_THREADS, 1) k_topk_rows(const float *__restrict__ scores, int64_t ld,
                                                              const int32_t *__restrict__ len,
                                                              const int32_t *__restrict__ cand, int k,
                                                              int32_t *__restrict__ out)
{
    __shared__ RsShared sh;
    pdl_launch_dependents();
    pdl_wait();
    const int64_t r = blockIdx.x;
    int64_t n64 = len[r];
    n64 = n64 < 0 ? 0 : (n64 > ld ? ld : n64);
    const int n = (int)n64;
    uint32_t key[RS_PER];
    const uint32_t valid = rs_load(scores + r * ld, n, key);
    int32_t *o = out + r * k;
    const int32_t *cr = cand ? cand + r * ld : nullptr;
    const int s0 = RS_PER * threadIdx.x;
    const int nsel = rs_select(key, valid, n, k, sh, [&](int j, int jj) {
        o[j] = cr ? __ldg(cr + s0 + jj) : s0 + jj;
    });
    for (int j = nsel + (int)threadIdx.x; j < k; j += RS_THREADS) o[j] = -1;
}

// Cluster size for rows of up to n keys (slices <= TK_SLICE keys): the block
// level of long rows and generic rows longer than RS_MAX keys.
static int topk_cluster_for(int64_t n)
{
    return n > 32768 ? 8 : (n > 8192 ? 4 : (n > 2048 ? 2 : 1));
}

template <class K, class... Args>
static int launch_cluster(K kernel, int cl, int64_t ld, int32_t rows, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows * (unsigned)cl);
    cfg.blockDim = dim3(TK_THREADS);
    cfg.dynamicSmemBytes = (size_t)(2 * slice_cap(ld, cl) * 4);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // a programmatic dependent
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

template <int CL>
static int topk_cl(const float *scores, int64_t ld, const int32_t *len, int32_t rows, const int32_t *cand,
                   int32_t k, int32_t *out, cudaStream_t st)
{
    if (const int s = kernel_smem_limit((const void *)k_topk<CL>, 2 * TK_SLICE * 4)) return s;
    return launch_cluster(k_topk<CL>, CL, ld, rows, st, scores, ld, len, cand, (int)k, out);
}

template <int CL>
static int blocks_cl(const float *block_max, int64_t ld_blocks, const int32_t *n_visible, int32_t rows,
                     int32_t pmax, int32_t *pool, int32_t *pool_len, const PoolKeys &pk, cudaStream_t st)
{
    if (const int s = kernel_smem_limit((const void *)k_topk_blocks<CL>, 2 * TK_SLICE * 4)) return s;
    return launch_cluster(k_topk_blocks<CL>, CL, ld_blocks, rows, st, block_max, ld_blocks, n_visible, (int)pmax,
                          pool, pool_len, pk.scores, pk.ld_scores, (int)pk.bf16, pk.k, pk.keys, pk.bound, pk.bound_ld);
}

int launch_topk(const float *scores, int64_t ld, const int32_t *len, int32_t rows, const int32_t *cand,
                int32_t k, int32_t *out, cudaStream_t st)
{
    if (rows == 0) return CSA2_OK;
    if (ld <= RS_MAX)
        return launch_pdl(k_topk_rows, dim3((unsigned)rows), dim3(RS_THREADS), 0, st, scores, ld, len, cand, (int)k,
                          out);
    switch (topk_cluster_for(ld)) {
    case 1: return topk_cl<1>(scores, ld, len, rows, cand, k, out, st);
    case 2: return topk_cl<2>(scores, ld, len, rows, cand, k, out, st);
    case 4: return topk_cl<4>(scores, ld, len, rows, cand, k, out, st);
    default: return topk_cl<8>(scores, ld, len, rows, cand, k, out, st);
    }
}

int launch_topk_blocks(const float *block_max, int64_t ld_blocks, const int32_t *n_visible, int32_t rows,
                       int32_t pmax, int32_t *pool, int32_t *pool_len, cudaStream_t st, const PoolKeys *pool_keys,
                       int *bounds_per_row)
{
    if (rows == 0) return CSA2_OK;
    const PoolKeys pk = pool_keys ? *pool_keys : PoolKeys{};
    int cl = topk_cluster_for(ld_blocks);
    // many rows fill the GPU by themselves: fewer CTAs per row (fewer cluster
    // rounds per row), as long as one CTA's slice still fits its shared memory
    const int sms = device_sms();
    while (cl > 1 && (int64_t)rows * cl > 2 * (int64_t)(sms > 0 ? sms : 1) && slice_cap(ld_blocks, cl / 2) <= TK_SLICE)
        cl /= 2;
    if (bounds_per_row) *bounds_per_row = cl;
    if (pk.keys && (cl > pk.bound_ld || !aligned(pk.scores, 16) || !aligned(pk.keys, 16) ||
                    (pk.ld_scores & 7) != 0))
        return CSA2_ERR_ALIGN;
    switch (cl) {
    case 1: return blocks_cl<1>(block_max, ld_blocks, n_visible, rows, pmax, pool, pool_len, pk, st);
    case 2: return blocks_cl<2>(block_max, ld_blocks, n_visible, rows, pmax, pool, pool_len, pk, st);
    case 4: return blocks_cl<4>(block_max, ld_blocks, n_visible, rows, pmax, pool, pool_len, pk, st);
    default: return blocks_cl<8>(block_max, ld_blocks, n_visible, rows, pmax, pool, pool_len, pk, st);
    }
}

int topk_max_k() { return TK_MAX_K; }

// Longest row a Top-K call accepts: 8 slices of TK_SLICE keys.
int64_t topk_max_len() { return 8 * (int64_t)TK_SLICE; }

}  // namespace csa2
