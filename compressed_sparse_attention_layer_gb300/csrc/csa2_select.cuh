// The cluster radix select shared by the Top-K kernels and the Reindex
// layer's fused rescoring: the k largest order keys of a row whose slices sit
// in the shared memory of the CTAs of one thread-block cluster (ties to the
// lower slot, ranks ascending with the slot).
#pragma once

#include <cooperative_groups.h>

#include "csa2_internal.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

constexpr int TK_THREADS = 512;
constexpr int TK_SLICE = 16384;            // keys staged per CTA (64 KB)
constexpr int TK_MAX_K = 4096;

struct TkShared {
    uint32_t hist[2048];                   // this CTA's slice counts
    uint32_t own[2048];                    // cluster totals of the bins this rank owns
    int own_total;                         // their sum
    int warp_sums[32];
    int cnt[2];                            // this CTA's (count > T, count == T)
    uint32_t digit;
    int above;
    uint32_t kmin, kmax;                   // this CTA's key range
    int ncand;                             // keys >= the bound, compacted
    uint32_t bin_count;                    // cluster-wide keys in the crossing bin
    uint32_t ndirect;                      // rank 0: keys of a small crossing bin gathered here
    uint32_t direct[32];
    uint32_t T;
    int need_eq;
};

// 32-bit load from the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_ld(const void *p, int rank)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p)), ra, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// Find the bin holding the kk-th largest key among those counted, and the
// count above that bin, from the CL slice histograms of the cluster.  Each CTA
// first totals its own 256 bins across the cluster (8 remote loads for 256
// threads); every CTA then reads the CL slice totals, finds the slice with
// the crossing, fetches that slice's 256 totals and scans them: the same
// decision everywhere.  Ends with the cluster synchronised.
template <int CL>
__device__ void cluster_digit(cg::cluster_group &cluster, TkShared &sh, int kk, uint32_t &digit, int &above)
{
    const int tid = threadIdx.x;
    const int me = (int)cluster.block_rank();
    constexpr int BPR = 2048 / CL;                   // bins owned per rank
    constexpr int PER = BPR > TK_THREADS ? BPR / TK_THREADS : 1;   // bins per thread
    constexpr int ACTIVE = BPR / PER;                // threads holding bins
    // ---- 1. own bins, cluster totals
    int v = 0;
    if (tid < ACTIVE) {
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const int bin = tid * PER + j;
            uint32_t acc = 0;
#pragma unroll
            for (int q = 0; q < CL; q++) acc += dsmem_ld(&sh.hist[BPR * me + bin], q);
            sh.own[bin] = acc;
            v += (int)acc;
        }
    }
    int tot = 0;
    (void)block_exclusive_scan<TK_THREADS>(v, sh.warp_sums, &tot);
    if (tid == 0) sh.own_total = tot;
    cluster.sync();
    // ---- 2. the slice holding the crossing (ranks from the top bins down)
    if (tid == 0) {
        int acc = 0, slice = 0, slice_above = 0;
        for (int q = CL - 1; q >= 0; q--) {
            const int t = (int)dsmem_ld(&sh.own_total, q);
            if (acc < kk && acc + t >= kk) {
                slice = q;
                slice_above = acc;
            }
            acc += t;
        }
        sh.digit = (uint32_t)slice;
        sh.above = slice_above;
    }
    __syncthreads();
    const int slice = (int)sh.digit, slice_above = sh.above;
    // ---- 3. the crossing bin inside that slice, bins in descending order
    int c[PER];
    int csum = 0;
#pragma unroll
    for (int j = 0; j < PER; j++) {
        c[j] = tid < ACTIVE ? (int)dsmem_ld(&sh.own[BPR - 1 - (tid * PER + j)], slice) : 0;
        csum += c[j];
    }
    const int excl = block_exclusive_scan<TK_THREADS>(csum, sh.warp_sums, nullptr);
    if (tid < ACTIVE && slice_above + excl < kk && slice_above + excl + csum >= kk) {
        int acc = slice_above + excl;
#pragma unroll
        for (int j = 0; j < PER; j++) {
            if (acc + c[j] >= kk) {
                sh.digit = (uint32_t)(BPR * slice + BPR - 1 - (tid * PER + j));
                sh.above = acc;
                sh.bin_count = (uint32_t)c[j];
                break;
            }
            acc += c[j];
        }
    }
    __syncthreads();
    digit = sh.digit;
    above = sh.above;
}

// Top k of a row of n keys; this CTA holds keys[0 .. m) = slots [lo, lo + m).
// emit(rank, slot) for every selected slot of this slice, rank ascending with
// the slot across the whole row.
template <int CL, class Emit>
__device__ void cluster_select(cg::cluster_group &cluster, const uint32_t *keys, uint32_t *cand, int64_t lo, int m,
                               int64_t n, int k, TkShared &sh, Emit emit)
{
    const int tid = threadIdx.x;
    if (n <= k) {                                    // everything is selected: rank = slot
        for (int i = tid; i < m; i += TK_THREADS) emit((int)(lo + i), lo + i);
        return;
    }
    // ---- a lower bound L of the k-th largest key and the row's maximum
    // (cluster-wide): the keys of TPG consecutive threads form a group (the
    // cluster has CL * TK_THREADS / TPG >= k groups); every non-empty group
    // holds a key >= its maximum, so at least k keys are >= L = the smallest
    // group maximum (an empty group makes L = 0, no bound).  Digits are
    // relative to L and only keys >= L are counted.
    {
        int tpg = (CL * TK_THREADS) / k;                 // threads per group, a power of two <= 32
        tpg = tpg >= 32 ? 32 : (tpg >= 16 ? 16 : (tpg >= 8 ? 8 : (tpg >= 4 ? 4 : (tpg >= 2 ? 2 : 1))));
        uint32_t gm = 0u, mx = 0u;
        for (int i = tid; i < m; i += TK_THREADS) gm = max(gm, keys[i]);
        for (int o = 1; o < tpg; o <<= 1) gm = max(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        uint32_t mn = k <= (CL * TK_THREADS) ? gm : 0u;  // the bound needs k groups
        mx = gm;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (tid == 0) {
            sh.kmin = 0xFFFFFFFFu;
            sh.kmax = 0u;
        }
        __syncthreads();
        if ((tid & 31) == 0) {
            atomicMin(&sh.kmin, mn);
            atomicMax(&sh.kmax, mx);
        }
    }
    cluster.sync();
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int q = 0; q < CL; q++) {
        const TkShared *o = cluster.map_shared_rank(&sh, q);
        kmin = min(kmin, o->kmin);
        kmax = max(kmax, o->kmax);
    }
    const uint32_t range = kmax - kmin;
    const int nbits = range ? 32 - __clz(range) : 1;
    // this CTA's keys >= the bound, compacted (thread by thread) so that every
    // radix round reads only them
    {
        int cnt = 0;
        for (int i = tid; i < m; i += TK_THREADS) cnt += keys[i] >= kmin;
        int tot = 0;
        int pos = block_exclusive_scan<TK_THREADS>(cnt, sh.warp_sums, &tot);
        for (int i = tid; i < m; i += TK_THREADS) {
            const uint32_t key = keys[i];
            if (key >= kmin) cand[pos++] = key;
        }
        if (tid == 0) sh.ncand = tot;
        __syncthreads();
    }
    const int nc = sh.ncand;
    uint32_t prefix = 0, mask = 0;                   // over rel = key - kmin, keys >= kmin only
    int kk = k;
    bool direct = false;
    if (tid == 0) sh.ndirect = 0u;                   // (cluster-synchronised before any use)
#pragma unroll 1
    for (int top = nbits; top > 0;) {
        const int width = top < 11 ? top : 11;
        const int shift = top - width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int b = tid; b < 2048; b += TK_THREADS) sh.hist[b] = 0;
        __syncthreads();
        for (int i = tid; i < nc; i += TK_THREADS) {
            const uint32_t rel = cand[i] - kmin;
            if ((rel & mask) == prefix) atomicAdd(&sh.hist[(rel >> shift) & dmask], 1u);
        }
        cluster.sync();                              // every slice counted
        uint32_t d;
        int above;
        cluster_digit<CL>(cluster, sh, kk, d, above);
        prefix |= d << shift;
        mask |= dmask << shift;
        kk -= above;
        top = shift;
        if (top > 0 && sh.bin_count <= 32u) {
            // a crossing bin of at most 32 keys (cluster-wide): gathered in rank 0,
            // whose first warp ranks them directly
            uint32_t *cnt0 = cluster.map_shared_rank(&sh.ndirect, 0);
            uint32_t *dir0 = cluster.map_shared_rank(sh.direct, 0);
            for (int i = tid; i < nc; i += TK_THREADS) {
                const uint32_t rel = cand[i] - kmin;
                if ((rel & mask) == prefix) dir0[atomicAdd(cnt0, 1u) & 31u] = cand[i];
            }
            cluster.sync();                          // every key gathered
            if (cluster.block_rank() == 0 && tid < 32) {
                const int nd = (int)(sh.ndirect < 32u ? sh.ndirect : 32u);
                const uint32_t v = tid < nd ? sh.direct[tid] : 0u;
                int gt = 0, ge = 0;
                for (int i = 0; i < nd; i++) {
                    const uint32_t u = sh.direct[i];
                    gt += u > v;
                    ge += u >= v;
                }
                // the kk-th largest of the bin (every lane holding it writes the same)
                if (tid < nd && gt < kk && ge >= kk) {
                    sh.T = v;
                    sh.need_eq = kk - gt;
                }
            }
            cluster.sync();                          // T written
            direct = true;
            break;
        }
        cluster.sync();                              // every CTA done reading before the reset
    }
    uint32_t T = prefix + kmin;
    int need_eq = kk;                                // ties with T that are selected, lowest slots first
    if (direct) {
        T = *cluster.map_shared_rank(&sh.T, 0);
        need_eq = *cluster.map_shared_rank(&sh.need_eq, 0);
    }

    // ---- counts of this thread's chunk, of this slice, and of the slices before it
    const int chunk = ((m + TK_THREADS - 1) / TK_THREADS) | 1;    // odd: no bank conflicts
    const int a = tid * chunk < m ? tid * chunk : m;
    const int e = a + chunk < m ? a + chunk : m;
    int gt = 0, eq = 0;
    for (int i = a; i < e; i++) {
        const uint32_t u = keys[i];
        gt += u > T;
        eq += u == T;
    }
    // one scan of both counts packed in 16-bit halves (a slice holds at most 16,384 keys)
    int tot_pk = 0;
    const int pk = block_exclusive_scan<TK_THREADS>((gt << 16) | eq, sh.warp_sums, &tot_pk);
    const int gt_local = pk >> 16, eq_local = pk & 0xFFFF;
    const int tot_gt = tot_pk >> 16, tot_eq = tot_pk & 0xFFFF;
    if (tid == 0) {
        sh.cnt[0] = tot_gt;
        sh.cnt[1] = tot_eq;
    }
    cluster.sync();
    int gt_slices = 0, eq_slices = 0;
    const int me = (int)cluster.block_rank();
    for (int q = 0; q < me; q++) {
        const int *cq = cluster.map_shared_rank(sh.cnt, q);
        gt_slices += cq[0];
        eq_slices += cq[1];
    }
    cluster.sync();                                  // counts read before any CTA exits
    const int eq_prior = eq_slices + eq_local;       // ties in slots before this chunk
    int take = need_eq - eq_prior;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    int off = gt_slices + gt_local + (eq_prior < need_eq ? eq_prior : need_eq);
    int seen = 0;
    for (int i = a; i < e; i++) {
        const uint32_t u = keys[i];
        if (u > T) {
            emit(off++, lo + i);
        } else if (u == T && seen < take) {
            emit(off++, lo + i);
            seen++;
        }
    }
}

}  // namespace csa2
