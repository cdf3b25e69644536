// The Full layer's lightning-indexer scan, e4m3 keys streamed into shared
// memory by cp.async and multiplied on the kind::f8f6f4 tensor cores.
//
// score(p) = s_p * sum_h w_h ReLU(qi_h . code_p) and the maximum of each
// aligned block of 8 positions ("DeepSeek-V4 report explainer" §3.2;
// "DeepSeek-V4.1-Flash" research note §3.2; "DeepSeek-V4.1-Flash 架构详解"
// §3.2).
//
// The keys stay e4m3 end to end: the 16-byte chunks of each 64-entry page of
// codes (8 KB) are copied by cp.async into a 128-byte-swizzled shared-memory
// tile, which is directly the K-major A operand (M = 128 entries, K = 128
// codes).  cp.async rather than the tensor-map TMA: on this gather of random
// 8 KB pages the TMA stream saturates near 5.3 TB/s while the load-store
// path sustains above 6 TB/s with fewer bytes in flight.  The indexer query is
// the B operand split into two e4m3 parts per head, hi = e4m3(q'), lo =
// e4m3(q' - hi), q' = q * 2^-e_h with max|q'| in [128, 256).  With one or
// two queries per tile hi and lo are stacked as one operand (rows 64 q .. hi,
// 64 q + 32 .. lo of query q), so each K step is one MMA that reads the key
// tile once and the epilogue adds the hi and lo columns; with four, they are
// two operands whose MMAs accumulate into the same fp32 sums (D = A.hi + A.lo),
// one column per head, which halves the epilogue's tensor-memory reads where
// the epilogue is the bottleneck.  The epilogue applies ReLU, w_h * 2^e_h and
// the entry's scale.
//
// Several queries of one sequence (QG = 2 or 4: draft tokens of a
// multi-token decode step, or the new tokens of a prefill chunk) share each
// key tile: their operands are stacked along N, so a tile is read from
// memory once for all of them, and each query keeps its own visible range
// (a score past it is not written, a block maximum covers visible entries only).
//
// A tile is 256 entries (four pages): two M = 128 halves per K step into a
// tensor-memory accumulator slot of 2N columns (512 columns hold 4, 2 or 2
// slots: tile parity gives every slot one issuer).  Warp
// roles (448 threads): warps 0-3 copy key tiles into a ring of stages (sixteen
// 16-byte chunks per thread per tile), warps 0-1 also the entries' fp32
// scales into the same stage, so that no role waits on a dependent global
// load per tile; warps 4-11 drain the accumulator slots (warp w: half
// (w - 4) / 4, TMEM lane quarter w % 4) and free a stage once they have read
// its scales (its MMAs are complete by then); warps 12 and 13 write the query
// operands of each group, and lane 0 of warps 12 and 13 issue the MMAs of the
// even and odd tiles (one issuing thread that also waits on barriers between
// tiles leaves the tensor pipe idle half the time).  A persistent grid walks
// one global list of (query group, tile) items so ragged batches stay balanced.
#include <cuda_bf16.h>

#include <algorithm>

#include "csa2_index_common.cuh"
#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int F8_TILE = 256;               // entries per tile: 4 pages, two MMA halves of M = 128
constexpr int F8_PROD = 128;               // producer threads (warps 0-3)
constexpr int F8_EPI_WARP = 4;             // epilogue warps 4-11: half (w - 4) / 4, lane quarter w % 4
constexpr int F8_EPI = 8;
constexpr int F8_MMA_WARP = 12;            // operand writers and MMA issuers: warps 12 and 13
constexpr int F8_THREADS = 448;
constexpr int F8_PERSIST_ROWS = 256;       // query groups of the persistent grid
constexpr uint32_t F8_TMEM_COLS = 512;

// QP: parts of each query operand -- 2: hi and lo (the query to about 8
// significant bits, the parity path); 1: hi only (4 significant bits, the
// CSA2_LAYER_INDEX_E4M3_QUERY option: one column per head, half the MMA
// work of the accumulated case).
template <int QG, int QP = 2>
struct F8Cfg {
    static constexpr int STAGES = QG == 1 ? 6 : (QG == 2 ? 5 : 4);    // 32 KB of codes per stage
    // hi and lo query parts: stacked along N (one MMA per K step, the epilogue
    // adds the two columns; the fewest MMA instructions) while two tile slots of
    // 2 x 64 QG columns fit in tensor memory, else accumulated into the same
    // columns by two MMAs per K step (half the epilogue's reads)
    static constexpr bool STACKED = QP == 2 && QG <= 2;
    static constexpr int N = (STACKED ? 64 : 32) * QG;                // MMA N
    static constexpr int PARTS = STACKED ? 1 : QP;                    // MMAs per K step and half
    static constexpr int SLOT_COLS = 2 * N;                           // accumulator of a tile (two halves)
    static constexpr int SLOTS = (int)F8_TMEM_COLS / SLOT_COLS;       // 4, 2, 2: even, so that each slot
    static constexpr int ISSUERS = 2;                                 // belongs to one issuer (tile parity)
    static constexpr int WRITERS = QG >= 2 ? 2 : 1;                   // query-operand warps
    static constexpr uint32_t IDESC = tc::idesc_e4m3(128, N);
    static_assert(QG == 1 || QG == 2 || QG == 4, "1, 2 or 4 queries per group");
    static_assert(QP == 1 || QP == 2, "one or two query parts");
    static_assert(SLOTS >= 2 && SLOTS % 2 == 0, "an even number of tile slots");
};

template <int QG, int QP>
struct F8Smem {
    static constexpr int ST = F8Cfg<QG, QP>::STAGES, SL = F8Cfg<QG, QP>::SLOTS;
    uint8_t a[ST][F8_TILE * 128];          // e4m3 keys, 128-byte swizzle (cp.async); rows 128 h .. of half h
    uint8_t b[2][QG * 64 * 128];           // per segment parity: the hi and lo rows of every query
    float sc[ST][F8_TILE];                 // fp32 scales of the stage's entries (cp.async)
    float wq[2][QG][32];                   // w_h * 2^e_h of each query, per segment parity
    uint64_t full[ST], empty[ST], tfull[SL], tempty[SL];
    uint64_t bfree[2], wready[2], wfree[2];
    uint32_t tmem;
    int abort;
    int32_t prefix[F8_PERSIST_ROWS + 1];
    int32_t rowcnt[F8_PERSIST_ROWS];       // entries scanned per query group (persistent grid)
};

// Scales copied for the entries of a page whose id lies outside the cache:
// they score -inf.
__device__ __align__(16) float g_neg_inf_scales[64] = {
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY,
    -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY};

// Entries scored by row r: every visible entry of the paged cache, or (DENSE)
// the first pool_len[r] of a dense per-row copy of a candidate pool's keys.
template <bool DENSE>
__device__ __forceinline__ int64_t f8_row_entries(const csa2_batch &bt, const int32_t *pool_len, int64_t ld, int r)
{
    if (!DENSE) return visible_entries(bt, r);
    const int64_t n = pool_len[r];
    return n < 0 ? 0 : (n > ld ? ld : n);
}

// Query group g of QG consecutive queries of one sequence: its first row r0,
// its sequence b, its number of queries qn (the last group of a sequence may
// be partial) and the entries it scans (the largest of its rows').
template <int QG, bool DENSE>
__device__ __forceinline__ int64_t f8_group(const csa2_batch &bt, const int32_t *pool_len, int64_t ld, int g,
                                            int &r0, int &b, int &qn)
{
    const int gps = (bt.nq + QG - 1) / QG;         // groups per sequence
    b = g / gps;
    const int i0 = (g - b * gps) * QG;
    r0 = b * bt.nq + i0;
    qn = bt.nq - i0 < QG ? bt.nq - i0 : QG;
    int64_t n = 0;
    for (int q = 0; q < qn; q++) {
        const int64_t e = f8_row_entries<DENSE>(bt, pool_len, ld, r0 + q);
        n = e > n ? e : n;
    }
    return n;
}

// DENSE = false: row r scans the visible entries of the paged cache c, in
// groups of QG rows of one sequence.
// DENSE = true (QG = 1): row r scans entries 0 .. pool_len[r] of rows of ld
// slots stored one after the other in c.ik_codes / c.ik_scales (page j of row
// r is page r * ld / 64 + j; no block table), scores only.
// `polls` bounds each pipeline wait: when one runs out the CTA sets its abort
// flag and CSA2_DEV_TIMEOUT, every role leaves its loop, and the teardown
// awaits the CTA's own copies and last MMA commit before freeing memory.
template <bool PERSIST, bool DENSE, int QG, int QP>
__global__ void __launch_bounds__(F8_THREADS, 1) k_index_f8(csa2_cache c, csa2_batch bt,
                                                            const uint16_t *__restrict__ qi,
                                                            const float *__restrict__ w,
                                                            const int32_t *__restrict__ pool_len,
                                                            float *__restrict__ scores,
                                                            float *__restrict__ block_max,
                                                            int32_t *__restrict__ n_visible, int64_t ld,
                                                            int bf16_scores, uint32_t polls)
{
    using Cfg = F8Cfg<QG, QP>;
    constexpr int ST = Cfg::STAGES, SL = Cfg::SLOTS, N = Cfg::N;
    static_assert(!DENSE || QG == 1, "a dense pool copy has one query per row");
    extern __shared__ uint8_t smem_raw[];
    F8Smem<QG, QP> &S = *reinterpret_cast<F8Smem<QG, QP> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    static_assert(F8Smem<QG, QP>::SL == SL && F8Smem<QG, QP>::ST == ST, "the barriers match the pipeline");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = bt.batch * bt.nq;
    const int groups = bt.batch * ((bt.nq + QG - 1) / QG);

    if (tid == 0) {
        for (int i = 0; i < ST; i++) {
            tc::mbar_init(&S.full[i], F8_PROD);
            tc::mbar_init(&S.empty[i], F8_EPI);      // the epilogue warps, after the tile's MMAs and scale reads
        }
        for (int i = 0; i < SL; i++) {
            tc::mbar_init(&S.tfull[i], 1);
            tc::mbar_init(&S.tempty[i], F8_EPI);     // the epilogue warps, once they have read it
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&S.bfree[i], Cfg::ISSUERS);
            tc::mbar_init(&S.wready[i], 32 * Cfg::WRITERS);
            tc::mbar_init(&S.wfree[i], F8_EPI);
        }
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == F8_MMA_WARP) tc::tmem_alloc(&S.tmem, F8_TMEM_COLS);
    // launched as a programmatic dependent: the set-up above is local; the
    // batch, cache and queries are read below, once the previous kernel is done
    pdl_launch_dependents();
    pdl_wait();

    int64_t g0, g1, nv_grp = 0;                   // nv_grp: the per-group grid's entry count
    if (!DENSE && blockIdx.x == 0 && (PERSIST || blockIdx.y == 0) && n_visible)
        for (int r = tid; r < rows; r += F8_THREADS) n_visible[r] = (int32_t)visible_entries(bt, r);
    if (PERSIST) {
        for (int gi = tid; gi < groups; gi += F8_THREADS) {
            int r0, b, qn;
            const int64_t nv = f8_group<QG, DENSE>(bt, pool_len, ld, gi, r0, b, qn);
            S.rowcnt[gi] = (int32_t)nv;
            S.prefix[gi + 1] = (int32_t)((nv + F8_TILE - 1) / F8_TILE);
        }
        __syncthreads();
        if (tid == 0) {
            S.prefix[0] = 0;
            for (int gi = 0; gi < groups; gi++) S.prefix[gi + 1] += S.prefix[gi];
        }
        __syncthreads();
        const int64_t total = S.prefix[groups];
        g0 = total * blockIdx.x / gridDim.x;
        g1 = total * (blockIdx.x + 1) / gridDim.x;
    } else {
        int r0, b, qn;
        const int64_t nv = f8_group<QG, DENSE>(bt, pool_len, ld, (int)blockIdx.y, r0, b, qn);
        const int64_t T = (nv + F8_TILE - 1) / F8_TILE;
        nv_grp = nv;
        g0 = T * blockIdx.x / gridDim.x;
        g1 = T * (blockIdx.x + 1) / gridDim.x;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    volatile int *abort = &S.abort;

    // every role walks the same segments (consecutive tiles of one query group)
    int grp = PERSIST ? 0 : (int)blockIdx.y;
    int64_t g = g0, it = 0;
    int seg = 0;
    int last_slot = -1;
    uint32_t last_par = 0;

    while (g < g1 && !*abort) {
        int64_t j0, nt;
        if (PERSIST) {
            while (S.prefix[grp + 1] <= g) grp++;
            j0 = g - S.prefix[grp];
            nt = std::min<int64_t>(g1, S.prefix[grp + 1]) - g;
        } else {
            j0 = g;
            nt = g1 - g;
        }
        // the group's sequence, first row and query count (QG = 1: the row itself)
        const int gps = QG == 1 ? 1 : (bt.nq + QG - 1) / QG;
        const int b = QG == 1 ? grp / bt.nq : grp / gps;
        const int r0 = QG == 1 ? grp : b * bt.nq + (grp - b * gps) * QG;
        const int qn = QG == 1 ? 1 : min(QG, bt.nq - (grp - b * gps) * QG);
        const int64_t nvis = PERSIST ? (int64_t)S.rowcnt[grp] : nv_grp;   // entries scanned

        if (warp < 4) {
            // ---------------- producers: page ids of 32 tiles at a time (one lane per
            // tile), then per tile sixteen 16-byte chunks of codes per thread (thread t:
            // chunk t % 8 of rows t / 8 + 16 j); warps 0-1 also the tile's 256 scales
            const uint32_t a0 = tc::smem_u32(S.a[0]);
            const int pt = warp * 32 + lane;
            int32_t my_pg[4] = {-1, -1, -1, -1};
            for (int64_t i = 0; i < nt; i++) {
                if ((i & 31) == 0) {
                    const int64_t e = (j0 + i + lane) * F8_TILE;     // tile i + lane
#pragma unroll
                    for (int h = 0; h < 4; h++) {
                        const int64_t e0 = e + 64 * h;
                        my_pg[h] = -2;                                // -2: beyond the visible entries
                        if (i + lane < nt && e0 < nvis) {
                            const int32_t pg = DENSE ? (int32_t)(r0 * (ld >> 6) + (e0 >> 6))
                                                     : __ldg(c.block_table + (int64_t)b * c.max_pages + (e0 >> 6));
                            my_pg[h] = pg >= 0 && ((int64_t)pg + 1) * CSA2_PAGE <= c.num_slots ? pg : -1;
                        }
                    }
                }
                int32_t pgs[4];
#pragma unroll
                for (int h = 0; h < 4; h++) pgs[h] = __shfl_sync(0xffffffffu, my_pg[h], (int)(i & 31));
                const int64_t ti = it + i;
                const int stage = (int)(ti % ST);
                const int k = (int)(ti / ST);
                const bool ok = k == 0 || tc::mbar_wait_or_abort(&S.empty[stage], (uint32_t)((k - 1) & 1), abort, polls);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) {
                        *abort = 1;
                        flag(c.status, CSA2_DEV_TIMEOUT);
                    }
                    break;
                }
                const uint32_t dst = a0 + (uint32_t)stage * (F8_TILE * 128);
#pragma unroll
                for (int jj = 0; jj < 16; jj++) {
                    const int e = pt + F8_PROD * jj;                  // 16-byte chunk of the tile
                    const int row = e >> 3, ch = e & 7, h = jj >> 2;  // rows 64 h .. 64 h + 63: page h
                    if (pgs[h] >= 0)
                        cp_async16(dst + (uint32_t)row * 128u + ((uint32_t)(ch ^ (row & 7)) << 4),
                                   c.ik_codes + ((int64_t)pgs[h] * CSA2_PAGE + (row & 63)) * 128 + ch * 16);
                }
                if (warp < 2) {
                    const int q = pt;                                 // entries 4 q .. 4 q + 3
                    const int h = q >> 4;
                    const float *src = pgs[h] >= 0 ? c.ik_scales + (int64_t)pgs[h] * CSA2_PAGE + 4 * (q & 15)
                                                   : g_neg_inf_scales + 4 * (q & 15);
                    if (pgs[h] != -2) cp_async16(tc::smem_u32(&S.sc[stage][4 * q]), src);
                    if (pgs[h] == -1 && (q & 15) == 0) flag(c.status, CSA2_DEV_BAD_PAGE);
                }
                cp_async_arrive(&S.full[stage]);
            }
        } else if (warp >= F8_MMA_WARP) {
            // ---------------- query operands (warps 12 and 13 split the group's queries)
            // and MMA issue (lane 0 of warp 12: even tiles, of warp 13: odd tiles; warp
            // 12 all of them when there is a single issuer)
            const int is = warp - F8_MMA_WARP;
            bool ok = true;
            if (is < Cfg::WRITERS) {
                // the operand and weights of segment seg-2 must be done with: its MMAs
                // completed (bfree) and the epilogue finished its tiles (wfree)
                if (seg >= 2 && lane == 0) {
                    const uint32_t par = (uint32_t)(((seg >> 1) - 1) & 1);
                    ok = tc::mbar_wait_or_abort(&S.bfree[seg & 1], par, abort, polls) &&
                         tc::mbar_wait_or_abort(&S.wfree[seg & 1], par, abort, polls);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok) {
                    for (int q = is; q < qn; q += Cfg::WRITERS) {
                        // stacked: query q's hi rows 64 q .., lo rows 64 q + 32 ..; accumulated:
                        // hi rows 32 q .., lo rows 32 QG + 32 q ..
                        uint8_t *bh = S.b[seg & 1] + (Cfg::STACKED ? 64 * q : 32 * q) * 128;
                        uint8_t *bl = S.b[seg & 1] + (Cfg::STACKED ? 64 * q + 32 : 32 * QG + 32 * q) * 128;
                        write_query_operand(bh, bl, S.wq[seg & 1][q], qi + (int64_t)(r0 + q) * 4096,
                                            w + (int64_t)(r0 + q) * 32);
                    }
                    tc::fence_proxy_async_smem();
                    tc::mbar_arrive(&S.wready[seg & 1]);
                }
            }
            if (is < Cfg::ISSUERS) {
                if (lane == 0 && ok) ok = tc::mbar_wait_or_abort(&S.wready[seg & 1], (uint32_t)((seg >> 1) & 1), abort, polls);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) {
                    if (lane == 0) {
                        *abort = 1;
                        flag(c.status, CSA2_DEV_TIMEOUT);
                    }
                } else {
                    if (lane == 0) {
                        const uint32_t a0 = tc::smem_u32(S.a[0]);
                        const uint32_t b0 = tc::smem_u32(S.b[seg & 1]);
                        for (int64_t i = (is - it) & 1; i < nt; i += 2) {   // tiles ti with ti % 2 == is
                            const int64_t ti = it + i;
                            const int stage = (int)(ti % ST);
                            if (!tc::mbar_wait_or_abort(&S.full[stage], (uint32_t)((ti / ST) & 1), abort, polls)) {
                                *abort = 1;
                                flag(c.status, CSA2_DEV_TIMEOUT);
                                break;
                            }
                            // the producers' cp.async writes, acquired through the barrier, made
                            // visible to the tensor core's (async-proxy) operand reads
                            tc::fence_proxy_async_smem();
                            const uint32_t as = a0 + (uint32_t)stage * (F8_TILE * 128);
                            const int slot = (int)(ti % SL);
                            if (ti >= SL &&
                                !tc::mbar_wait_or_abort(&S.tempty[slot], (uint32_t)(((ti / SL) - 1) & 1), abort, polls)) {
                                *abort = 1;
                                flag(c.status, CSA2_DEV_TIMEOUT);
                                break;
                            }
                            tc::tc_fence_after();
#pragma unroll
                            for (int hf = 0; hf < 2; hf++)       // two halves of 128 entries
#pragma unroll
                                for (int kk = 0; kk < 4; kk++)   // K = 128 codes in steps of 32
#pragma unroll
                                    for (int part = 0; part < Cfg::PARTS; part++)   // (hi, then lo)
                                        tc::mma_f8(tmem + (uint32_t)(slot * Cfg::SLOT_COLS + hf * N),
                                                   tc::smem_desc(as + hf * (128 * 128) + kk * 32, 16, 1024,
                                                                 tc::kSwizzle128B),
                                                   tc::smem_desc(b0 + (uint32_t)(part * N * 128) + kk * 32, 16, 1024,
                                                                 tc::kSwizzle128B),
                                                   Cfg::IDESC, (kk | part) > 0);
                            // the stage is released by the epilogue, which reads its scales only
                            // after this commit: the MMAs are done with the codes by then
                            tc::mma_commit(&S.tfull[slot]);
                            last_slot = slot;
                            last_par = (uint32_t)((ti / SL) & 1);
                        }
                        tc::mma_commit(&S.bfree[seg & 1]);
                    }
                    __syncwarp();
                }
            }
        } else {
            // ---------------- epilogue: warps 4-11, half (warp - 4) / 4, TMEM lanes by warp % 4
            const int qd = warp & 3, hf = (warp - F8_EPI_WARP) >> 2;
            const bool wok = tc::mbar_wait_or_abort(&S.wready[seg & 1], (uint32_t)((seg >> 1) & 1), abort, polls);
            if (!__all_sync(0xffffffffu, wok)) {
                if (lane == 0) {
                    *abort = 1;
                    flag(c.status, CSA2_DEV_TIMEOUT);
                }
                break;
            }
            int32_t nvq[QG];                              // each query's own visible range (< 2^31)
#pragma unroll
            for (int q = 0; q < QG; q++)
                nvq[q] = QG == 1 ? (int32_t)nvis : (q < qn ? (int32_t)f8_row_entries<DENSE>(bt, pool_len, ld, r0 + q) : 0);
            const int64_t rowp = (int64_t)hf * 128 + qd * 32 + lane;
            for (int64_t i = 0; i < nt; i++) {
                const int64_t ti = it + i;
                const int stage = (int)(ti % ST);
                const int slot = (int)(ti % SL);
                // the MMAs of tile ti are done, so its stage's data has landed: the wait on
                // full[stage] returns at once and acquires the producers' scale copies (the
                // stage cannot refill before this warp's arrival on empty[stage] below)
                bool ok = tc::mbar_wait_or_abort(&S.tfull[slot], (uint32_t)((ti / SL) & 1), abort, polls) &&
                          tc::mbar_wait_or_abort(&S.full[stage], (uint32_t)((ti / ST) & 1), abort, polls);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) {
                        *abort = 1;
                        flag(c.status, CSA2_DEV_TIMEOUT);
                    }
                    break;
                }
                tc::tc_fence_after();
                const uint32_t ta = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(slot * Cfg::SLOT_COLS + hf * N);
                const float sc_cur = S.sc[stage][rowp];
                const int64_t p = (j0 + i) * F8_TILE + rowp;
                float res[QG];
                if constexpr (Cfg::STACKED) {
#pragma unroll
                    for (int q = 0; q < QG; q++) {
                        const float *wv = S.wq[seg & 1][q];   // broadcast shared-memory reads
                        float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // four independent chains
                        if (q < qn) {
#pragma unroll
                            for (int c16 = 0; c16 < 2; c16++) {   // heads 16 c16 .. 16 c16 + 15: hi + lo columns
                                uint32_t dh[16], dl[16];
                                tc::tmem_ld16(ta + 64u * q + 16u * c16, dh);
                                tc::tmem_ld16(ta + 64u * q + 32u + 16u * c16, dl);
                                tc::tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 16; j++) {
                                    const float x = __uint_as_float(dh[j]) + __uint_as_float(dl[j]);
                                    part[j & 3] = fmaf(wv[16 * c16 + j], fmaxf(x, 0.0f), part[j & 3]);
                                }
                            }
                        }
                        res[q] = (part[0] + part[1]) + (part[2] + part[3]);
                    }
                } else if constexpr (QG == 1) {
                    // one column per head (one query part)
                    uint32_t d0[32];
                    tc::tmem_ld32(ta, d0);
                    tc::tmem_ld_wait();
                    const float *w0 = S.wq[seg & 1][0];
                    float p0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int j = 0; j < 32; j++) p0[j & 3] = fmaf(w0[j], fmaxf(__uint_as_float(d0[j]), 0.0f), p0[j & 3]);
                    res[0] = (p0[0] + p0[1]) + (p0[2] + p0[3]);
                } else {
                    // one column per head (hi . k + lo . k, or hi . k alone); two queries'
                    // columns in flight per tensor-memory wait
#pragma unroll
                    for (int q = 0; q < QG; q += 2) {
                        uint32_t d0[32], d1[32];
                        tc::tmem_ld32(ta + 32u * q, d0);
                        tc::tmem_ld32(ta + 32u * (q + 1), d1);
                        tc::tmem_ld_wait();
                        const float *w0 = S.wq[seg & 1][q], *w1 = S.wq[seg & 1][q + 1];
                        float p0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, p1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int j = 0; j < 32; j++) {
                            p0[j & 3] = fmaf(w0[j], fmaxf(__uint_as_float(d0[j]), 0.0f), p0[j & 3]);
                            p1[j & 3] = fmaf(w1[j], fmaxf(__uint_as_float(d1[j]), 0.0f), p1[j & 3]);
                        }
                        res[q] = (p0[0] + p0[1]) + (p0[2] + p0[3]);
                        res[q + 1] = (p1[0] + p1[1]) + (p1[2] + p1[3]);
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&S.tempty[slot]);
                    tc::mbar_arrive(&S.empty[stage]);
                }
#pragma unroll
                for (int q = 0; q < QG; q++) {
                    if (q >= qn) break;
                    const bool valid = p < nvq[q];
                    const int64_t rq = r0 + q;
                    float sc = -INFINITY;
                    if (valid) {
                        if (sc_cur != -INFINITY) sc = res[q] * sc_cur;
                        if (bf16_scores) {             // kept as bf16 (nearest even); maxima of the rounded
                            const __nv_bfloat16 hb = __float2bfloat16_rn(sc);
                            sc = __bfloat162float(hb);
                            if (scores) reinterpret_cast<__nv_bfloat16 *>(scores)[rq * ld + p] = hb;
                        } else if (scores) {
                            scores[rq * ld + p] = sc;
                        }
                    }
                    if (!DENSE && block_max) {
                        float m = valid ? sc : -INFINITY;
#pragma unroll
                        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if ((lane & 7) == 0 && valid) block_max[rq * (ld / 8) + (p >> 3)] = m;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.wfree[seg & 1]);   // this warp is done with seg's weights
        }
        g += nt;
        it += nt;
        seg++;
    }

    // ---- teardown: nothing in flight may outlive the CTA's shared and tensor memory
    if (warp < 4) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (*abort && (tid == F8_MMA_WARP * 32 || tid == (F8_MMA_WARP + 1) * 32) && last_slot >= 0)
        tc::mbar_wait(&S.tfull[last_slot], last_par, 1u << 20);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == F8_MMA_WARP) tc::tmem_dealloc(tmem, F8_TMEM_COLS);
}

// ---------------------------------------------------------------- host side
template <bool DENSE, int QG, int QP>
static int launch_f8_q(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                       const int32_t *pool_len, float *scores, float *block_max, int32_t *n_visible, int64_t ld,
                       cudaStream_t st, bool bf16, int sms)
{
    const int groups = bt.batch * ((bt.nq + QG - 1) / QG);
    const size_t smem = sizeof(F8Smem<QG, QP>) + 1024;
    int s = CSA2_OK;
    if constexpr (QG == 1)
        s = kernel_smem_limit((const void *)k_index_f8<true, DENSE, QG, QP>, smem);
    if (s || (s = kernel_smem_limit((const void *)k_index_f8<false, DENSE, QG, QP>, smem))) return s;
    const int64_t per_row = DENSE ? ld : bt.max_entries;
    const int64_t tiles_row = std::max<int64_t>(1, (per_row + F8_TILE - 1) / F8_TILE);
    // the persistent grid (ragged single-query batches) for QG = 1; query groups
    // (equal lengths within a sequence) take a grid of CTAs per group
    if constexpr (QG == 1) {
        if (groups <= F8_PERSIST_ROWS) {
            const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)groups * tiles_row, sms));
            return launch_pdl(k_index_f8<true, DENSE, QG, QP>, dim3(grid), dim3(F8_THREADS), smem, st, c, bt, qi, w,
                              pool_len, scores, block_max, n_visible, ld, (int)bf16, wait_polls());
        }
    }
    if (groups > 65535) return CSA2_ERR_SHAPE;   // groups run along the grid's y dimension
    const int x = (int)std::max<int64_t>(1, std::min<int64_t>(tiles_row, ((int64_t)sms + groups - 1) / groups));
    return launch_pdl(k_index_f8<false, DENSE, QG, QP>, dim3(x, groups), dim3(F8_THREADS), smem, st, c, bt, qi, w,
                      pool_len, scores, block_max, n_visible, ld, (int)bf16, wait_polls());
}

// Queries per group: the largest of 4, 2, 1 that the per-sequence query count
// fills (a dense pool copy holds one query's keys per row).
template <bool DENSE, int QP>
static int launch_f8(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                     const int32_t *pool_len, float *scores, float *block_max, int32_t *n_visible, int64_t ld,
                     cudaStream_t st, bool bf16)
{
    const int sms = device_sms();
    if (sms <= 0) return CSA2_ERR_CUDA;
    if (DENSE || bt.nq < 2)
        return launch_f8_q<DENSE, 1, QP>(c, bt, qi, w, pool_len, scores, block_max, n_visible, ld, st, bf16, sms);
    if (bt.nq < 4)
        return launch_f8_q<false, 2, QP>(c, bt, qi, w, pool_len, scores, block_max, n_visible, ld, st, bf16, sms);
    return launch_f8_q<false, 4, QP>(c, bt, qi, w, pool_len, scores, block_max, n_visible, ld, st, bf16, sms);
}

int launch_index_scan(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                      float *scores, float *block_max, int32_t *n_visible, int64_t ld, cudaStream_t st,
                      bool bf16_scores, bool one_part_query)
{
    if (one_part_query)
        return launch_f8<false, 1>(c, bt, qi, w, nullptr, scores, block_max, n_visible, ld, st, bf16_scores);
    return launch_f8<false, 2>(c, bt, qi, w, nullptr, scores, block_max, n_visible, ld, st, bf16_scores);
}

// Dense copy of the indexer keys of each row's candidate pool: slot e of row r
// gets the codes and scale of position pool[r][e] (one thread per 16-byte
// chunk, all of a row's lookups in flight at once).  A position that is not a
// visible entry, or whose page id lies outside the cache, gets zero codes and
// a -inf scale (it scores -inf) and is flagged.
__global__ void __launch_bounds__(256) k_gather_pool(csa2_cache c, csa2_batch bt, const int32_t *__restrict__ pool,
                                                     const int32_t *__restrict__ pool_len, int64_t ld,
                                                     uint8_t *__restrict__ codes, float *__restrict__ scales)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t r = blockIdx.y;
    const int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int64_t e = t >> 3;
    const int ch = (int)(t & 7);
    int64_t n = pool_len[r];
    n = n < 0 ? 0 : (n > ld ? ld : n);
    if (e >= n) return;
    const int b = (int)(r / bt.nq);
    const int64_t nvis = visible_entries(bt, r);
    const int32_t p = __ldg(pool + r * ld + e);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    float s = -INFINITY;
    if (p >= 0 && p < nvis) {
        const int32_t pg = __ldg(c.block_table + (int64_t)b * c.max_pages + (p >> 6));
        if (pg >= 0 && ((int64_t)pg + 1) * CSA2_PAGE <= c.num_slots) {
            const int64_t slot = (int64_t)pg * CSA2_PAGE + (p & 63);
            v = __ldg(reinterpret_cast<const uint4 *>(c.ik_codes + slot * 128) + ch);
            s = __ldg(c.ik_scales + slot);
        } else if (ch == 0) {
            flag(c.status, CSA2_DEV_BAD_PAGE);
        }
    } else if (ch == 0) {
        flag(c.status, CSA2_DEV_BAD_INDEX);
    }
    reinterpret_cast<uint4 *>(codes + (r * ld + e) * 128)[ch] = v;
    if (ch == 0) scales[r * ld + e] = s;
}

int launch_gather_pool(const csa2_cache &c, const csa2_batch &bt, const int32_t *pool, const int32_t *pool_len,
                       int64_t ld, uint8_t *codes, float *scales, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    return launch_pdl(k_gather_pool, dim3((unsigned)((ld * 8 + 255) / 256), (unsigned)rows), dim3(256), 0, st, c, bt,
                      pool, pool_len, ld, codes, scales);
}

// Scores of the dense pool copy (rows of ld slots, codes [rows][ld][128] and
// scales [rows][ld]) for slots 0 .. pool_len[r] of each row.
int launch_index_dense(const uint8_t *codes, const float *scales, const csa2_batch &bt, const uint16_t *qi,
                       const float *w, const int32_t *pool_len, int64_t ld, float *scores, cudaStream_t st,
                       bool bf16_scores)
{
    if (ld % CSA2_PAGE) return CSA2_ERR_SHAPE;
    csa2_cache d = {};
    d.ik_codes = const_cast<uint8_t *>(codes);
    d.ik_scales = const_cast<float *>(scales);
    d.num_slots = (int64_t)bt.batch * bt.nq * ld;
    return launch_f8<true, 2>(d, bt, qi, w, pool_len, scores, nullptr, nullptr, ld, st, bf16_scores);
}

}  // namespace csa2
