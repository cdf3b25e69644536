// A Reindex layer's selection: rescore the candidate pool with the layer's own
// indexer query, then take its Top-512 ("DeepSeek-V4.1-Flash 架构详解" §3 mode
// table and §3.2: later layers re-rank only the pool the Full layer kept;
// "DeepSeek-V4 report explainer" §3.2 for the weighted-ReLU score).
//
// The pool a Full layer writes is a list of blocks of 8 consecutive positions,
// each inside one 64-entry page, so a block's indexer keys are 8 consecutive
// cache slots: 8 rows of 128 e4m3 codes, exactly one 128-byte-swizzle atom of
// the tensor core's K-major operand.  Two launches:
//   1. k_rx_score: P CTAs per query row (P about SMs / rows, so a decode batch
//      still streams its pools' keys through every SM), each taking a run of
//      128-entry tiles of the pool.  Warp-specialised: four warps copy each
//      block's codes with 16-byte cp.async straight into the swizzled operand
//      layout, plus its 8 fp32 scales, eight stages in flight; two threads
//      issue the kind::f8f6f4 MMAs of alternate tiles against the query
//      operand (two e4m3 parts per head, hi | lo stacked as N = 64, as in the
//      Full layer's scan) into four tensor-memory slots; eight warps first
//      write the query operand (one 16-dim chunk of one head per thread), then
//      read the slots out (two warps per lane quarter, alternate tiles):
//      score = s_e * sum_h w_h ReLU(hi_h . k + lo_h . k), written as an order
//      key, and the CTA's smallest maximum over groups of G consecutive slots;
//   2. k_rx_select: one CTA per row, thread t holding the keys of slots
//      16 t .. 16 t + 15 in registers.  The smallest group
//      maximum over the row is a lower bound L with at least k keys >= L (G is
//      chosen so that there are at least k groups, and each group holds a key
//      equal to its maximum); an exact radix select over the keys >= L
//      (typically a few percent), from the top bit of the row's largest key
//      down, gives the k-th largest, and one block scan places every thread's
//      selected slots in ascending order (ties to the lower slot).
// No copy of the pool's keys is made; the scores cross HBM once as 4-byte keys.
#include "csa2_index_common.cuh"

namespace csa2 {

constexpr int RX_BLK = CSA2_BLOCK;                 // slots per pool block
constexpr int RX_TILE = 128;                       // entries per tile (MMA M)
constexpr int RX_BPT = RX_TILE / RX_BLK;           // blocks per tile
constexpr int RX_ROW_TILES = CSA2_POOL_MAX / RX_TILE;
constexpr int RX_PMAX = 32;                        // scoring CTAs per row at most
constexpr int RX_STAGES = 8;
constexpr int RX_SLOTS = 4;                        // tensor-memory accumulators of 64 columns
constexpr int RX_THREADS = 512;
constexpr int RX_PROD = 128;                       // warps 0-3 copy the tiles
constexpr int RX_MMA_WARP = 4;                     // warps 4 and 5: one MMA thread each
constexpr int RX_EPI_WARP = 8;                     // warps 8-15 write the query, read the accumulators out
constexpr int RX_EPI = 8;
constexpr uint32_t RX_TMEM_COLS = 64 * RX_SLOTS;
constexpr uint32_t RX_IDESC = tc::idesc_e4m3(128, 64);
constexpr int RX_DIGIT = 12;                       // radix digit of the select
constexpr int RX_BINS = 1 << RX_DIGIT;
constexpr int RX_SEL_THREADS = 1024;               // select threads per row
constexpr int RX_KPT = CSA2_POOL_MAX / RX_SEL_THREADS;   // keys a select thread holds
static_assert(RX_SLOTS % 2 == 0, "each MMA thread owns its own accumulator slots");
static_assert(RX_BINS % RX_SEL_THREADS == 0, "whole bins per thread");
static_assert(RX_KPT <= 16 && RX_KPT % 4 == 0, "a thread's counts packed in 16 bits, keys in 16-byte loads");

struct RxSmem {
    uint8_t a[RX_STAGES][RX_TILE * 128];           // e4m3 key codes, swizzled
    uint8_t b[64 * 128];                           // query: hi rows 0-31, lo rows 32-63
    float sc[RX_STAGES][RX_TILE];                  // the tile's key scales
    float wq[32];                                  // w_h * 2^e_h
    int64_t bslot[CSA2_POOL_MAX / RX_BLK];         // first cache slot of each block, -1: none
    uint2 gred[RX_THREADS / 32];                   // per warp: smallest group maximum, largest key
    uint64_t full[RX_STAGES], empty[RX_STAGES], tfull[RX_SLOTS], tempty[RX_SLOTS], bready;
    uint32_t tmem;
    int abort;
    int cslot[RX_SLOTS];                           // per accumulator slot: 1 + last tile committed
};

struct RsSmem {
    uint32_t hist[2][RX_BINS];                     // radix histograms of alternate rounds
    int warp_sums[RX_SEL_THREADS / 32];
    uint32_t digit;
    int above;
    int bincnt;                                    // candidates in the crossing bin
    int ncand;                                     // of them gathered into cand (at most 32)
    uint32_t cand[32];
    uint32_t tval;                                 // the k-th largest offset, once ranked by one warp
    int tneed;
};

// Scales copied for the entries of a block that is not read: they score -inf
// (copied like the real scales, so the stage's barrier covers them).
__device__ __align__(16) float g_rx_neg_inf[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};

// Groups of G consecutive slots for the lower bound: the largest power of two
// <= 32 leaving at least k groups among the pool's n slots.
__device__ __forceinline__ int rx_group(int64_t n, int k)
{
    int G = 1;
    while (G < 32 && (int64_t)(G * 2) * k <= n) G *= 2;
    return G;
}

// Grid P x rows (CTA p of row r at r P + p); 512 threads.  keys [rows][16384]
// order keys of the pool's slots (slots < pool_len), gmm [rows][RX_PMAX]: each
// CTA's smallest group maximum (all ones when it has no group) and largest key.
__global__ void __launch_bounds__(RX_THREADS, 1)
    k_rx_score(csa2_cache c, csa2_batch bt, const uint16_t *__restrict__ qi, const float *__restrict__ w,
               const int32_t *__restrict__ pool, const int32_t *__restrict__ pool_len, int k, int P, int tpc,
               uint32_t *__restrict__ keys, uint2 *__restrict__ gmm, int bf16_scores, uint32_t polls)
{
    extern __shared__ uint8_t smem_raw[];
    RxSmem &S = *reinterpret_cast<RxSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t r = blockIdx.x / P;
    const int p = (int)(blockIdx.x - r * P);
    const int b = (int)(r / bt.nq);
    volatile int *abort = &S.abort;
    const int32_t *prow = pool + r * CSA2_POOL_MAX;
    const int64_t b0 = (int64_t)p * tpc * RX_BPT;  // first block of this CTA's run

    if (tid == 0) {
        for (int i = 0; i < RX_STAGES; i++) {
            tc::mbar_init(&S.full[i], RX_PROD);    // every copying thread, once its copies landed
            tc::mbar_init(&S.empty[i], RX_EPI / 2);   // the tile's four read-out warps
        }
        for (int i = 0; i < RX_SLOTS; i++) {
            tc::mbar_init(&S.tfull[i], 1);
            tc::mbar_init(&S.tempty[i], RX_EPI / 2);
            S.cslot[i] = 0;
        }
        tc::mbar_init(&S.bready, RX_EPI);
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == RX_MMA_WARP) tc::tmem_alloc(&S.tmem, RX_TMEM_COLS);
    // the inputs into L2 while the previous kernel finishes (nothing is read yet)
    if (warp < RX_PROD / 32) {
        const int64_t s_first = b0 * RX_BLK, s_end = min((int64_t)CSA2_POOL_MAX, s_first + (int64_t)tpc * RX_TILE);
        const uint8_t *pr = reinterpret_cast<const uint8_t *>(prow);
        for (int64_t s = s_first + 32 * tid; s < s_end; s += 32 * RX_PROD) prefetch_l2(pr + 4 * s);
        const int64_t bt_lines = ((int64_t)c.max_pages * 4 + 127) / 128;
        const uint8_t *btr = reinterpret_cast<const uint8_t *>(c.block_table + (int64_t)b * c.max_pages);
        for (int64_t j = p + (int64_t)P * tid; j < bt_lines; j += (int64_t)P * RX_PROD) prefetch_l2(btr + 128 * j);
    } else if (warp >= RX_EPI_WARP) {
        const int et = tid - RX_EPI_WARP * 32;
        if (et < CSA2_IDX_HEADS * CSA2_IDX_DIM * 2 / 128)
            prefetch_l2(reinterpret_cast<const uint8_t *>(qi + r * (CSA2_IDX_HEADS * CSA2_IDX_DIM)) + 128 * et);
        if (et == RX_EPI * 32 - 1) prefetch_l2(w + r * CSA2_IDX_HEADS);
    }
    pdl_launch_dependents();
    pdl_wait();                                    // the pool and the queries are inputs

    int64_t n = pool_len[r];
    n = n < 0 ? 0 : (n > CSA2_POOL_MAX ? CSA2_POOL_MAX : n);
    const int64_t nblk_row = (n + RX_BLK - 1) / RX_BLK;
    int64_t nb = nblk_row - b0;                    // this CTA's blocks (none when n <= k:
    nb = n <= k ? 0 : (nb < 0 ? 0 : (nb > (int64_t)tpc * RX_BPT ? (int64_t)tpc * RX_BPT : nb));   // all selected)
    const int nblocks = (int)nb;
    const int ntiles = (nblocks + RX_BPT - 1) / RX_BPT;
    const int64_t nvis = visible_entries(bt, r);
    const int G = rx_group(n, k);

    // ---- the first cache slot of every block of the run (all lookups in flight
    //      at once).  A block is its positions p0 .. p0 + cnt - 1 (cnt = 8, fewer
    //      for the pool's last), p0 a multiple of 8 below the visible entries;
    //      anything else (a pool not written by a Full layer), or a page outside
    //      the cache, is flagged and scores -inf
    for (int j = tid; j < nblocks; j += RX_THREADS) {
        const int64_t s0 = (b0 + j) * RX_BLK;
        const int cnt = (int)(n - s0 < RX_BLK ? n - s0 : RX_BLK);
        const int4 v0 = __ldg(reinterpret_cast<const int4 *>(prow + s0));
        const int4 v1 = __ldg(reinterpret_cast<const int4 *>(prow + s0) + 1);
        const int32_t pv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        const int32_t p0 = pv[0];
        bool ok = p0 >= 0 && (p0 & (RX_BLK - 1)) == 0 && p0 + cnt <= nvis;
#pragma unroll
        for (int t = 1; t < RX_BLK; t++) ok = ok && (t >= cnt || pv[t] == p0 + t);
        int64_t slot = -1;
        if (ok) {
            const int32_t pg = __ldg(c.block_table + (int64_t)b * c.max_pages + (p0 >> 6));
            if (pg >= 0 && ((int64_t)pg + 1) * CSA2_PAGE <= c.num_slots) slot = (int64_t)pg * CSA2_PAGE + (p0 & 63);
            else flag(c.status, CSA2_DEV_BAD_PAGE);
        } else {
            flag(c.status, CSA2_DEV_BAD_INDEX);
        }
        S.bslot[j] = slot;
    }
    __syncthreads();

    const uint32_t tmem = S.tmem;
    uint32_t gmin = 0xFFFFFFFFu, gmax = 0u;
    if (warp < RX_PROD / 32) {
        // ---------------- producers: tile i's blocks into stage i % RX_STAGES; thread t
        //                  copies chunks t + 128 u (block u, row t / 8 % 8, 16-byte chunk
        //                  t % 8 of it: into the swizzled position of row 8 u + row)
        for (int i = 0; i < ntiles; i++) {
            const int s = i % RX_STAGES;
            const bool ok = i < RX_STAGES ||
                            tc::mbar_wait_or_abort(&S.empty[s], (uint32_t)(((i / RX_STAGES) - 1) & 1), abort, polls);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) *abort = 1;
                break;
            }
            const uint32_t a0 = tc::smem_u32(S.a[s]);
#pragma unroll
            for (int u = 0; u < RX_BPT * 64 / RX_PROD; u++) {
                const int cidx = tid + RX_PROD * u;             // chunk of the tile
                const int jj = cidx >> 6, row = (cidx >> 3) & 7, ch = cidx & 7;
                const int j = i * RX_BPT + jj;
                const int64_t slot = j < nblocks ? S.bslot[j] : -1;
                if (slot >= 0)
                    cp_async16(a0 + (uint32_t)(jj * 8 + row) * 128u + ((uint32_t)(ch ^ row) << 4),
                               c.ik_codes + (slot + row) * 128 + ch * 16);
            }
            if (tid < 2 * RX_BPT) {                             // the scales: two 16-byte halves per block
                const int jj = tid >> 1, j = i * RX_BPT + jj;
                const int64_t slot = j < nblocks ? S.bslot[j] : -1;
                cp_async16(tc::smem_u32(&S.sc[s][RX_BLK * jj + 4 * (tid & 1)]),
                           slot >= 0 ? c.ik_scales + slot + 4 * (tid & 1) : g_rx_neg_inf);
            }
            cp_async_arrive(&S.full[s]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // nothing of ours lands after we leave
    } else if (warp == RX_MMA_WARP || warp == RX_MMA_WARP + 1) {
        // ---------------- MMA issue (lane 0 of each warp, alternate tiles): tile i into
        //                  accumulator slot i % RX_SLOTS
        if (lane == 0) {
            bool ok = tc::mbar_wait_or_abort(&S.bready, 0, abort, polls);
            for (int i = warp - RX_MMA_WARP; i < ntiles && ok; i += 2) {
                const int s = i % RX_STAGES, sl = i % RX_SLOTS;
                ok = tc::mbar_wait_or_abort(&S.full[s], (uint32_t)((i / RX_STAGES) & 1), abort, polls) &&
                     (i < RX_SLOTS ||
                      tc::mbar_wait_or_abort(&S.tempty[sl], (uint32_t)(((i / RX_SLOTS) - 1) & 1), abort, polls));
                if (!ok) break;
                // the producers' cp.async writes, acquired through the barrier, made
                // visible to the tensor core's (async-proxy) operand reads
                tc::fence_proxy_async_smem();
                tc::tc_fence_after();
                const uint32_t a0 = tc::smem_u32(S.a[s]), bq = tc::smem_u32(S.b);
#pragma unroll
                for (int kk = 0; kk < 4; kk++)     // K = 128 codes in steps of 32
                    tc::mma_f8(tmem + 64u * (uint32_t)sl, tc::smem_desc(a0 + kk * 32, 16, 1024, tc::kSwizzle128B),
                               tc::smem_desc(bq + kk * 32, 16, 1024, tc::kSwizzle128B), RX_IDESC, kk > 0);
                tc::mma_commit(&S.tfull[sl]);
                S.cslot[sl] = i + 1;               // slot sl is this thread's alone
            }
            if (!ok) *abort = 1;
        }
    } else if (warp >= RX_EPI_WARP) {
        // ---------------- the query operand: thread (head h, 16-dim chunk c)
        {
            const int ew = warp - RX_EPI_WARP;
            write_query_chunk(S.b, S.b + 32 * 128, S.wq, qi + r * (CSA2_IDX_HEADS * CSA2_IDX_DIM),
                              w + r * CSA2_IDX_HEADS, 4 * ew + (lane >> 3), lane & 7);
            tc::fence_proxy_async_smem();
            tc::named_bar_sync(1, RX_EPI * 32);    // every w_h * 2^e_h written before the read-out
            if (lane == 0) tc::mbar_arrive(&S.bready);
        }
        // ---------------- read-out: warp w takes lane quarter w % 4 (one entry per lane)
        //                  of the tiles of parity (w - 8) / 4, all 32 heads (hi columns
        //                  0-31, lo 32-63)
        const int qd = warp & 3, par = (warp - RX_EPI_WARP) >> 2;
        for (int i = par; i < ntiles; i += 2) {
            const int s = i % RX_STAGES, sl = i % RX_SLOTS;
            const bool ok = tc::mbar_wait_or_abort(&S.tfull[sl], (uint32_t)((i / RX_SLOTS) & 1), abort, polls) &&
                            tc::mbar_wait_or_abort(&S.full[s], (uint32_t)((i / RX_STAGES) & 1), abort, polls);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) *abort = 1;
                break;
            }
            tc::tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(qd * 32) << 16) + 64u * (uint32_t)sl;
            float half[2];
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {       // heads 16 hh .. 16 hh + 15
                uint32_t dh[16], dl[16];
                tc::tmem_ld16(ta + 16u * (uint32_t)hh, dh);
                tc::tmem_ld16(ta + 32u + 16u * (uint32_t)hh, dl);
                tc::tmem_ld_wait();
                float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const float x = __uint_as_float(dh[j]) + __uint_as_float(dl[j]);
                    p4[j & 3] = fmaf(S.wq[16 * hh + j], fmaxf(x, 0.0f), p4[j & 3]);
                }
                half[hh] = (p4[0] + p4[1]) + (p4[2] + p4[3]);
            }
            const float s_e = S.sc[s][qd * 32 + lane];
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&S.tempty[sl]);
                tc::mbar_arrive(&S.empty[s]);
            }
            float sc = -INFINITY;
            if (s_e != -INFINITY) sc = (half[0] + half[1]) * s_e;
            if (bf16_scores) sc = __bfloat162float(__float2bfloat16_rn(sc));
            const int64_t e = (b0 + (int64_t)i * RX_BPT) * RX_BLK + qd * 32 + lane;   // slot of the pool
            const uint32_t key = order_key(sc);
            if (e < n) {
                keys[r * CSA2_POOL_MAX + e] = key;
                gmax = max(gmax, key);
            }
            uint32_t gm = e < n ? key : 0u;                // past the pool: below every score
            for (int o = 1; o < G; o <<= 1) gm = max(gm, __shfl_xor_sync(0xffffffffu, gm, o));
            if ((e & (G - 1)) == 0 && e < n) gmin = min(gmin, gm);
        }
    }
    gmin = __reduce_min_sync(0xffffffffu, gmin);
    gmax = __reduce_max_sync(0xffffffffu, gmax);
    if (lane == 0) S.gred[warp] = make_uint2(gmin, gmax);
    __syncthreads();
    const bool failed = *abort != 0;
    if (tid == 0) {
        uint2 v = make_uint2(0xFFFFFFFFu, 0u);
#pragma unroll
        for (int u = 0; u < RX_THREADS / 32; u++) v = make_uint2(min(v.x, S.gred[u].x), max(v.y, S.gred[u].y));
        gmm[r * RX_PMAX + p] = v;
        if (failed) flag(c.status, CSA2_DEV_TIMEOUT);
    }
    // ---- teardown of the pipeline: after a timeout, the products in flight are
    //      awaited (long limit) before the tensor memory is released (the
    //      producers waited for their own copies); only a slot's last product
    //      can still be running
    if (failed && tid == 0) {
        for (int sl = 0; sl < RX_SLOTS; sl++)
            if (S.cslot[sl] > 0)
                tc::mbar_wait(&S.tfull[sl], (uint32_t)(((S.cslot[sl] - 1) / RX_SLOTS) & 1), 1u << 22);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == RX_MMA_WARP) tc::tmem_dealloc(tmem, RX_TMEM_COLS);
}

// Grid rows; 1024 threads.  out [rows][k]: the k best pool positions of each
// row in ascending slot order, -1 after the pool's end.
__global__ void __launch_bounds__(RX_SEL_THREADS, 1)
    k_rx_select(const int32_t *__restrict__ pool, const int32_t *__restrict__ pool_len,
                const uint32_t *__restrict__ keys, const uint2 *__restrict__ gmm, int P, int k,
                int32_t *__restrict__ out)
{
    __shared__ RsSmem S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const int32_t *prow = pool + r * CSA2_POOL_MAX;
    const uint32_t *krow = keys + r * CSA2_POOL_MAX;
    static_assert(RX_PMAX <= 32, "one lane per scoring CTA");
    constexpr int BPT = RX_BINS / RX_SEL_THREADS;  // bins per thread in the digit search
#pragma unroll
    for (int j = 0; j < BPT; j++) S.hist[0][tid + RX_SEL_THREADS * j] = 0u;
    pdl_launch_dependents();
    pdl_wait();                                    // the keys and bounds of the scoring launch

    // every load at once: the pool's length, this thread's keys (slots past the
    // pool hold stale values, masked below) and the scoring CTAs' bounds (lane u:
    // CTA u)
    int64_t n = pool_len[r];
    uint4 kq[RX_KPT / 4];
#pragma unroll
    for (int j = 0; j < RX_KPT / 4; j++) kq[j] = __ldcg(reinterpret_cast<const uint4 *>(krow + RX_KPT * tid) + j);
    const uint2 mm = lane < P ? __ldcg(gmm + r * RX_PMAX + lane) : make_uint2(0xFFFFFFFFu, 0u);
    const uint32_t L = __reduce_min_sync(0xffffffffu, mm.x), kmax = __reduce_max_sync(0xffffffffu, mm.y);
    n = n < 0 ? 0 : (n > CSA2_POOL_MAX ? CSA2_POOL_MAX : n);
    int32_t *o = out + r * k;
    if (n <= k) {                                  // every slot is selected, in slot order
        for (int64_t e = tid; e < k; e += RX_SEL_THREADS) o[e] = e < n ? __ldg(prow + e) : -1;
        return;
    }
    // candidates: offsets rel = key - L of this thread's keys >= L
    uint32_t rk[RX_KPT], valid = 0u;
#pragma unroll
    for (int j = 0; j < RX_KPT / 4; j++) {
        const uint32_t kv[4] = {kq[j].x, kq[j].y, kq[j].z, kq[j].w};
#pragma unroll
        for (int cc = 0; cc < 4; cc++) {
            const int i = 4 * j + cc;
            rk[i] = kv[cc] - L;
            valid |= (uint32_t)((int64_t)RX_KPT * tid + i < n && kv[cc] >= L) << i;
        }
    }
    // ---- the k-th largest offset: radix select from the top bit of the largest
    //      key's offset down, RX_DIGIT bits a round, three barriers a round
    const uint32_t range = kmax - L;
    int top = range ? 32 - __clz(range) : 0;
    uint32_t prefix = 0, mask = 0;
    int kk = k, cur = 0;
    __syncthreads();                               // histogram 0 zeroed
#pragma unroll 1
    while (top > 0) {
        const int width = top < RX_DIGIT ? top : RX_DIGIT;
        const int shift = top - width;
        const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
        for (int j = 0; j < RX_KPT; j++)
            if (((valid >> j) & 1u) && (rk[j] & mask) == prefix) atomicAdd(&S.hist[cur][(rk[j] >> shift) & dmask], 1u);
        __syncthreads();
        // thread t: bins RX_BINS - 1 - BPT t downwards; the warp's inclusive scan of
        // their sums; the other histogram zeroed for the next round
        uint32_t cb[BPT];
        int cs = 0;
#pragma unroll
        for (int j = 0; j < BPT; j++) {
            cb[j] = S.hist[cur][RX_BINS - 1 - (BPT * tid + j)];
            cs += (int)cb[j];
        }
        int x = cs;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o2);
            if (lane >= o2) x += y;
        }
        if (lane == 31) S.warp_sums[warp] = x;
#pragma unroll
        for (int j = 0; j < BPT; j++) S.hist[cur ^ 1][tid + RX_SEL_THREADS * j] = 0u;
        __syncthreads();
        int ex = x - cs;
        for (int u = 0; u < warp; u++) ex += S.warp_sums[u];
        if (ex < kk && ex + cs >= kk) {            // the thread whose bins hold the k-th
            int acc = ex;
#pragma unroll
            for (int j = 0; j < BPT; j++) {
                if (acc + (int)cb[j] >= kk) {
                    S.digit = (uint32_t)(RX_BINS - 1 - (BPT * tid + j));
                    S.above = acc;
                    S.bincnt = (int)cb[j];
                    S.ncand = 0;
                    break;
                }
                acc += (int)cb[j];
            }
        }
        __syncthreads();
        prefix |= S.digit << shift;
        mask |= dmask << shift;
        kk -= S.above;
        top = shift;
        cur ^= 1;
        if (top > 0 && S.bincnt <= 32) {
            // a crossing bin of at most 32 keys: one warp ranks them instead of
            // further rounds (the kk-th largest of the bin, and how many equal
            // to it are taken)
#pragma unroll
            for (int j = 0; j < RX_KPT; j++)
                if (((valid >> j) & 1u) && (rk[j] & mask) == prefix) S.cand[atomicAdd(&S.ncand, 1)] = rk[j];
            __syncthreads();
            if (warp == 0) {
                const int nc = S.ncand;
                const uint32_t v = lane < nc ? S.cand[lane] : 0u;
                int gt = 0, eq = 0;
                for (int u = 0; u < nc; u++) {
                    const uint32_t w2 = __shfl_sync(0xffffffffu, v, u);
                    gt += w2 > v;
                    eq += w2 == v;
                }
                if (lane < nc && gt < kk && gt + eq >= kk) {   // lanes holding the same value agree
                    S.tval = v;
                    S.tneed = kk - gt;
                }
            }
            __syncthreads();
            prefix = S.tval;
            kk = S.tneed;
            break;
        }
    }
    const uint32_t T = prefix;                     // the k-th largest offset
    const int need_eq = kk;                        // of the offsets equal to T, the first need_eq
    // ---- this thread's selected (> T) and tied (== T) slots; one scan gives the
    //      ties and the selected slots before it
    uint32_t sel = 0u, teq = 0u;
#pragma unroll
    for (int j = 0; j < RX_KPT; j++) {
        const bool v = (valid >> j) & 1u;
        sel |= (uint32_t)(v && rk[j] > T) << j;
        teq |= (uint32_t)(v && rk[j] == T) << j;
    }
    const int pk = block_exclusive_scan<RX_SEL_THREADS>((__popc(teq) << 16) | __popc(sel), S.warp_sums, nullptr);
    const int tie_before = pk >> 16;
    int take = need_eq - tie_before;
    take = take < 0 ? 0 : (take > __popc(teq) ? __popc(teq) : take);
    uint32_t word = sel, rest = teq;
    for (int u = 0; u < take; u++) {
        const uint32_t bit = rest & (~rest + 1u);  // lowest remaining tie
        word |= bit;
        rest ^= bit;
    }
    // the selected slots' pool positions: every load issued before the first store
    int32_t pv[RX_KPT];
#pragma unroll
    for (int j = 0; j < RX_KPT; j++)
        if ((word >> j) & 1u) pv[j] = __ldg(prow + RX_KPT * tid + j);
    int off = (pk & 0xFFFF) + (tie_before < need_eq ? tie_before : need_eq);
#pragma unroll
    for (int j = 0; j < RX_KPT; j++)
        if ((word >> j) & 1u) {
            if (off < k) o[off] = pv[j];
            off++;
        }
}

// ---------------------------------------------------------------- host side
size_t reindex_workspace_bytes(int64_t rows) { return (size_t)rows * (CSA2_POOL_MAX * 4 + RX_PMAX * 8); }

// The Reindex layer's selection: each row's pool (as a Full layer writes it)
// rescored with (qi, w) against the cache's indexer keys and reduced to its
// best k pool positions (out [rows][k], ascending, -1 after).  ws: at least
// reindex_workspace_bytes(rows), 16-byte aligned.
int launch_reindex(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w, const int32_t *pool,
                   const int32_t *pool_len, int k, int32_t *out, bool bf16, void *ws, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    if (k < 1 || k > CSA2_POOL_MAX / 32) return CSA2_ERR_SHAPE;   // the lower bound's groups of <= 32 slots
    if (!aligned(pool, 16) || !aligned(ws, 16)) return CSA2_ERR_ALIGN;
    const int sms = device_sms();
    int P = (int)((sms > 0 ? sms : 1) / rows);
    P = P < 1 ? 1 : (P > RX_PMAX ? RX_PMAX : P);
    const int tpc = (RX_ROW_TILES + P - 1) / P;
    P = (RX_ROW_TILES + tpc - 1) / tpc;            // no CTA without tiles
    if (rows * P > INT32_MAX) return CSA2_ERR_SHAPE;
    uint32_t *keys = static_cast<uint32_t *>(ws);
    uint2 *gmm = reinterpret_cast<uint2 *>(keys + rows * CSA2_POOL_MAX);
    const size_t smem = sizeof(RxSmem) + 1024;
    if (const int s = kernel_smem_limit((const void *)k_rx_score, smem)) return s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * P));
    cfg.blockDim = dim3(RX_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_rx_score, c, bt, qi, w, pool, pool_len, k, P, tpc, keys, gmm,
                                       (int)bf16, wait_polls());
    if (e == cudaSuccess) {
        cfg.gridDim = dim3((unsigned)rows);
        cfg.blockDim = dim3(RX_SEL_THREADS);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, k_rx_select, (const int32_t *)pool, pool_len, (const uint32_t *)keys,
                               (const uint2 *)gmm, P, k, out);
    }
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

// The Full layer's pool Top-k with the select above: keys and per-CTA bounds as
// the block-level Top-K wrote them (P bounds per row, at most RX_PMAX), out
// [rows][k] ascending, -1 after.
int launch_pool_select(const int32_t *pool, const int32_t *pool_len, const uint32_t *keys, const uint2 *bound,
                       int P, int k, int32_t *out, int64_t rows, cudaStream_t st)
{
    if (rows == 0) return CSA2_OK;
    if (k < 1 || k > CSA2_POOL_MAX / 32 || P < 1 || P > RX_PMAX) return CSA2_ERR_SHAPE;
    if (!aligned(keys, 16)) return CSA2_ERR_ALIGN;
    return launch_pdl(k_rx_select, dim3((unsigned)rows), dim3(RX_SEL_THREADS), 0, st, pool, pool_len, keys, bound,
                      P, k, out);
}

}  // namespace csa2
