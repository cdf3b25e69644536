// a5/a6: Top-K selection with ties broken toward the lower slot.
//
// One 1024-thread CTA per row.  Radix select on order-preserving 32-bit keys
// (11 + 11 + 10 bit digits, shared-memory histograms) finds the k-th largest
// key T and how many keys equal to T must be taken; an ordered compaction
// (block-wide prefix sums over contiguous per-thread chunks) then writes the
// chosen positions in ascending slot order, taking the lowest-slot ties.
// Rows of up to TK_STAGE elements are staged in shared memory once; longer
// rows are re-read from global memory (L2) on each pass.
// "DeepSeek-V4.1-Flash 架构详解" §1 table (top-k 512), §3.2 (block pool of
// 2,048 blocks of 8, then its own Top-512); the research note §3.2.
#include "csa2_internal.cuh"

namespace csa2 {

constexpr int TK_THREADS = 1024;
constexpr int TK_STAGE = 40960;            // staged keys (160 KB of shared memory)
constexpr int TK_MAX_K = 4096;

struct SmemKeys {
    const uint32_t *k;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const { return k[i]; }
};
struct GmemKeys {
    const float *s;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const { return order_key(__ldg(s + i)); }
};

struct TkShared {
    uint32_t hist[2048];
    int warp_sums[32];
    int total;
    uint32_t digit;
    int above;
};

// k-th largest key T among n keys (n > k) and the number of keys equal to T
// that belong to the top k.
template <class Src>
__device__ void find_threshold(const Src &src, int64_t n, int k, TkShared &sh, uint32_t &T,
                               int &need_eq)
{
    const int tid = threadIdx.x;
    uint32_t prefix = 0, mask = 0;
    int kk = k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
#pragma unroll 1
    for (int pass = 0; pass < 3; pass++) {
        const int shift = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int b = tid; b < 2048; b += TK_THREADS) sh.hist[b] = 0;
        __syncthreads();
        // every lane of a warp runs the same trip count; lanes with the same digit
        // combine their counts before one shared-memory atomic
        const int lane = tid & 31;
        for (int64_t base = tid - lane; base < n; base += TK_THREADS) {
            const int64_t i = base + lane;
            uint32_t u = 0;
            bool on = false;
            if (i < n) {
                u = src(i);
                on = (u & mask) == prefix;
            }
            const uint32_t act = __ballot_sync(0xffffffffu, on);
            if (on) {
                const uint32_t bin = (u >> shift) & dmask;
                const uint32_t peers = __match_any_sync(act, bin);
                if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        // bins in descending order: thread t owns bins 2047-2t and 2046-2t
        const int c0 = (int)sh.hist[2047 - 2 * tid], c1 = (int)sh.hist[2046 - 2 * tid];
        const int excl = block_exclusive_scan<TK_THREADS>(c0 + c1, sh.warp_sums, nullptr);
        if (excl < kk && excl + c0 + c1 >= kk) {
            if (excl + c0 >= kk) {
                sh.digit = 2047 - 2 * tid;
                sh.above = excl;
            } else {
                sh.digit = 2046 - 2 * tid;
                sh.above = excl + c0;
            }
        }
        __syncthreads();
        prefix |= sh.digit << shift;
        mask |= dmask << shift;
        kk -= sh.above;
        __syncthreads();
    }
    T = prefix;
    need_eq = kk;
}

// Emit, in ascending slot order, every slot with key > T and the first
// need_eq slots with key == T: emit(j, i) for output rank j and slot i.
template <class Src, class Emit>
__device__ void ordered_compact(const Src &src, int64_t n, uint32_t T, int need_eq, TkShared &sh,
                                Emit emit)
{
    const int tid = threadIdx.x;
    const int64_t chunk = ((n + TK_THREADS - 1) / TK_THREADS) | 1;   // odd: no bank conflicts
    const int64_t lo = tid * chunk < n ? tid * chunk : n;
    const int64_t hi = lo + chunk < n ? lo + chunk : n;
    int gt = 0, eq = 0;
    for (int64_t i = lo; i < hi; i++) {
        const uint32_t u = src(i);
        gt += u > T;
        eq += u == T;
    }
    const int eq_before = block_exclusive_scan<TK_THREADS>(eq, sh.warp_sums, nullptr);
    int take = need_eq - eq_before;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    int off = block_exclusive_scan<TK_THREADS>(gt + take, sh.warp_sums, nullptr);
    int seen = 0;
    for (int64_t i = lo; i < hi; i++) {
        const uint32_t u = src(i);
        if (u > T) {
            emit(off++, i);
        } else if (u == T && seen < take) {
            emit(off++, i);
            seen++;
        }
    }
}

// Select the top k of row (src, n); emit(j, slot) for j < min(n, k).
template <class Emit>
__device__ void select_row(const float *row, int64_t n, int k, uint32_t *stage, TkShared &sh,
                           Emit emit)
{
    if (n <= k) {
        for (int64_t i = threadIdx.x; i < n; i += TK_THREADS) emit((int)i, i);
        return;
    }
    uint32_t T;
    int need_eq;
    if (n <= TK_STAGE) {
        for (int64_t i = threadIdx.x; i < n; i += TK_THREADS) stage[i] = order_key(__ldg(row + i));
        __syncthreads();
        SmemKeys src{stage};
        find_threshold(src, n, k, sh, T, need_eq);
        ordered_compact(src, n, T, need_eq, sh, emit);
    } else {
        GmemKeys src{row};
        find_threshold(src, n, k, sh, T, need_eq);
        ordered_compact(src, n, T, need_eq, sh, emit);
    }
}

__global__ void __launch_bounds__(TK_THREADS) k_topk(const float *__restrict__ scores, int64_t ld,
                                                     const int32_t *__restrict__ len,
                                                     const int32_t *__restrict__ cand, int k,
                                                     int32_t *__restrict__ out)
{
    extern __shared__ uint32_t stage[];
    __shared__ TkShared sh;
    const int64_t r = blockIdx.x;
    int64_t n = len[r];
    n = n < 0 ? 0 : (n > ld ? ld : n);
    int32_t *o = out + r * k;
    const int32_t *cr = cand ? cand + r * ld : nullptr;
    select_row(scores + r * ld, n, k, stage, sh, [&](int j, int64_t i) {
        if (j < k) o[j] = cr ? cr[i] : (int32_t)i;
    });
    const int64_t nsel = n < k ? n : k;
    for (int64_t j = nsel + threadIdx.x; j < k; j += TK_THREADS) o[j] = -1;
}

__global__ void __launch_bounds__(TK_THREADS) k_topk_blocks(const float *__restrict__ block_max,
                                                            int64_t ld_blocks,
                                                            const int32_t *__restrict__ n_visible,
                                                            int pmax, int32_t *__restrict__ pool,
                                                            int32_t *__restrict__ pool_len)
{
    extern __shared__ uint32_t stage[];
    __shared__ TkShared sh;
    __shared__ int32_t sel[CSA2_POOL_BLOCKS];
    const int64_t r = blockIdx.x;
    int64_t nv = n_visible[r];
    nv = nv < 0 ? 0 : (nv > ld_blocks * 8 ? ld_blocks * 8 : nv);
    const int64_t nb = (nv + 7) / 8;
    select_row(block_max + r * ld_blocks, nb, pmax, stage, sh, [&](int j, int64_t i) {
        if (j < pmax) sel[j] = (int32_t)i;
    });
    __syncthreads();
    const int nsel = (int)(nb < pmax ? nb : pmax);
    int32_t *pr = pool + r * (int64_t)pmax * 8;
    for (int j = threadIdx.x; j < nsel * 8; j += TK_THREADS) {
        const int64_t p = (int64_t)sel[j >> 3] * 8 + (j & 7);
        if (p < nv) pr[j] = (int32_t)p;
    }
    if (threadIdx.x == 0) {
        int total = 0;
        if (nsel > 0) {
            const int64_t last = (int64_t)sel[nsel - 1] * 8;
            const int64_t tail = nv - last < 8 ? nv - last : 8;
            total = (nsel - 1) * 8 + (int)tail;
        }
        pool_len[r] = total;
    }
}

static int topk_smem_bytes(int64_t n_max)
{
    const int64_t n = n_max < TK_STAGE ? n_max : TK_STAGE;
    return (int)(n * 4);
}

int launch_topk(const float *scores, int64_t ld, const int32_t *len, int32_t rows, const int32_t *cand,
                int32_t k, int32_t *out, cudaStream_t st)
{
    if (rows == 0) return CSA2_OK;
    const int smem = topk_smem_bytes(ld);
    static bool attr = false;                   // raise the limit once, before any graph capture
    if (!attr) {
        cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, TK_STAGE * 4);
        attr = true;
    }
    k_topk<<<rows, TK_THREADS, smem, st>>>(scores, ld, len, cand, k, out);
    return launch_status();
}

int launch_topk_blocks(const float *block_max, int64_t ld_blocks, const int32_t *n_visible,
                       int32_t rows, int32_t pmax, int32_t *pool, int32_t *pool_len, cudaStream_t st)
{
    if (rows == 0) return CSA2_OK;
    const int smem = topk_smem_bytes(ld_blocks);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_topk_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize, TK_STAGE * 4);
        attr = true;
    }
    k_topk_blocks<<<rows, TK_THREADS, smem, st>>>(block_max, ld_blocks, n_visible, pmax, pool, pool_len);
    return launch_status();
}

int topk_max_k() { return TK_MAX_K; }

}  // namespace csa2
