// Sparse MQA + sliding-window attention, many-row schedule: persistent
// two-CTA clusters that each take whole query rows.
//
// The same computation as csa2_attn_tc.cu -- every key is its own value
// ("DeepSeek-V4 report explainer" §4.3), one softmax over the selected
// entries and the window ("DeepSeek-V4.1-Flash 架构详解" §1 table, §3;
// explainer §3.3), with the sink and the output re-rotation of the merge --
// scheduled for calls with many query rows (prefill, several query tokens per
// sequence, large decode groups), where one cluster per (row, key chunk)
// leaves every chunk paying the whole dependent chain (launch, query load,
// key lookups, two products, two exchanges) and the partial outputs make a
// round trip through memory.
//
// A cluster of two CTAs (CTA d: dims 256 d .. 256 d + 255) takes rows
// r = cluster, cluster + clusters, ... and walks each row's chunks in order
// (chunks 0..n-2 the selected entries, 128 each; the last the window); with
// new_rows, it first quantises its rows' own window rows into the ring:
//   - the query slice is loaded once per row;
//   - per chunk: dequantise the keys (already in registers) into the key
//     tile; partial S^T = K_d Q_d^T (M = keys, N = 64 heads); the other CTA's
//     heads go to it by one bulk copy; CTA d sums its 32 heads' partials and
//     runs an online softmax over the row: running maximum m, P = exp(S - m)
//     as bf16 hi + lo, the running sum l, and the factor alpha = exp(m_old -
//     m) by which the output so far shrinks; P rows and alpha go to the other
//     CTA; [O_hi | O_lo]_c^T = V_d^T [P_hi | P_lo]^T, and each thread keeps its
//     (dim, 32 heads) of the row's output in registers: acc = alpha acc + O_c;
//   - after the last chunk: o = acc x mult, mult = f / L with the sink folded
//     in (the same arithmetic as the merge kernel), the RoPE dims rotated
//     back, lse = M + log L.
// The keys are fetched ahead: while a chunk's first product is issued, the
// next chunk's codes (its page already known) and the index of the chunk
// after it are loaded, and that index's page after the product's read-out,
// so the codes have a whole chunk to arrive.
// 512 threads: four per key (64 dims each) for the loads and dequantisation,
// sixteen per owned head for the softmax, one tensor-memory lane each in the
// read-outs.
#include "csa2_attn_common.cuh"

namespace csa2 {

static_assert(AC_CL == 2, "the row schedule pairs two CTAs");
static_assert(AC_MT == 2, "two M-tiles of 128 dims per CTA");
// Tensor memory: [O_hi | O_lo]^T of M-tile mt in columns 128 mt .. 128 mt + 127
// (N = 128: the hi and lo rows of P side by side, half as many products as two
// N = 64 halves); S^T in columns 256 .. 319.
constexpr uint32_t AR_TMEM_COLS = 512;
constexpr uint32_t AR_S_COL = 256;
constexpr uint32_t AR_XS_BYTES = 2 * AC_OWN * 4;                      // alpha and mult of the owned heads
constexpr uint32_t AR_P_IN_BYTES = 4 * AC_P_ROWS_BYTES + AR_XS_BYTES;

// Per-row values every thread needs, computed once by one thread.
struct RowInfo {
    int64_t t;      // the query's token position
    int64_t lo;     // first window token
    int64_t vis;    // entries visible to the query
    int64_t dlo;    // de-duplicated entries dlo .. dhi (empty: dlo > dhi)
    int64_t dhi;
    int32_t b;      // sequence
    int32_t pad_;
};

struct ArSmem {
    uint8_t k[AC_SLABS * AC_KEYS * 128];           // key tile [slab of 64 dims][128 keys][128 B]   64 KB
    uint8_t q[AC_SLABS * CSA2_HEADS * 128];        // query slice [slab][64 heads][128 B]           32 KB
    float pout[CSA2_HEADS][AC_KEYS];               // this CTA's partial logits [head][key]         32 KB
                                                   // (also the RoPE exchange at the end of a row)
    uint8_t p[2 * 2 * CSA2_HEADS * 128];           // probability operand [slab of 64 keys][hi 64 | 32 KB
                                                   // lo 64 rows][128 B]; the other CTA's rows copied in
    float ps[AC_OWN][AC_KEYS];                     // the other CTA's partials of this CTA's heads  16 KB
    uint32_t e2m1_pair[256][32];                   // byte -> bf16x2 of its two E2M1 codes, per lane 32 KB
    float xs[AC_CL][2][AC_OWN];                    // per owning CTA: alpha and mult of its heads
    float kscale[AC_KEYS];                         // window row scale (1 for entries), -1: no key
    RowInfo ri[2];                                 // rows 2i and 2i + 1 of this cluster
    uint64_t mbar;                                 // the products' commits (two per chunk)
    uint64_t sbar;                                 // the other CTA's partial logits have landed
    uint64_t pbar;                                 // the other CTA's probability rows have landed
    uint32_t tmem;
};

// Bounded wait on a phase; after a timeout (flagged) the same phase is awaited
// once more with a long limit, so that both CTAs keep the same sequence of
// phases.  False only if that also runs out.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, uint32_t polls, int32_t *status)
{
    if (tc::mbar_wait(bar, parity, polls)) return true;
    flag(status, CSA2_DEV_TIMEOUT);
    return tc::mbar_wait(bar, parity, 1u << 22);
}

__global__ void __cluster_dims__(AC_CL, 1, 1) __launch_bounds__(AC_THREADS, 1)
    k_attn_rows(csa2_cache c, csa2_batch bt, const uint16_t *__restrict__ q, float sm_scale,
                const int32_t *__restrict__ idx, int k, csa2_swa swa, float *__restrict__ o,
                float *__restrict__ lse, int nchunks, int64_t rows, RopeTurns turns, uint32_t polls)
{
    extern __shared__ uint8_t smem_raw[];
    ArSmem &S = *reinterpret_cast<ArSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int key = tid & (AC_KEYS - 1), hf = tid >> 7;          // key row; 64-dim slab of this CTA
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16; // tensor-memory lane quarter of this warp
    const uint32_t dq = cluster_rank(), peer = dq ^ 1u;
    const int64_t ncl = gridDim.x / AC_CL, cl = blockIdx.x / AC_CL;
    const int64_t my_rows = cl < rows ? (rows - 1 - cl) / ncl + 1 : 0;
    const int64_t n_items = my_rows * nchunks;
    const bool rope = swa.rope_base > 0.0f;

    if (tid == 0) {
        tc::mbar_init(&S.mbar, 1);
        tc::mbar_init(&S.sbar, 1);
        tc::mbar_init(&S.pbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem, AR_TMEM_COLS);
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&S.sbar, AC_S_BYTES);        // the first chunk's exchanges
        tc::mbar_arrive_expect_tx(&S.pbar, AR_P_IN_BYTES);
    }
    // first half of a cluster barrier: this CTA's mbarriers are initialised; the
    // matching wait comes before the first copy into the other CTA
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
#pragma unroll
    for (int ch = tid; ch < 256 * 32 / 4; ch += AC_THREADS) {
        const uint32_t v = e2m1x2_to_bf16x2((uint32_t)ch >> 3);
        reinterpret_cast<uint4 *>(&S.e2m1_pair[0][0])[ch] = make_uint4(v, v, v, v);
    }
    // the first row's query slice into L2 (no value is consumed before the wait)
    constexpr int LPH = AC_DIMS * 2 / 128;         // 128-byte lines per head of the slice
    if (my_rows > 0 && tid < CSA2_HEADS * LPH)
        prefetch_l2(q + (cl * CSA2_HEADS + tid / LPH) * CSA2_HEAD_DIM + AC_DIMS * dq + 64 * (tid % LPH));
    pdl_wait();

    auto row_of = [&](int64_t i) { return cl + i * ncl; };
    auto row_info = [&](RowInfo &R, int64_t r) {
        const int b = (int)(r / bt.nq);
        const int64_t t = bt.q_pos[r];
        const int64_t s0 = swa.start ? swa.start[b] : 0;
        int64_t lo = t - (CSA2_SWA_WINDOW - 1);
        lo = lo < s0 ? s0 : lo;
        lo = lo < 0 ? 0 : lo;
        R.t = t;
        R.lo = lo;
        R.vis = visible_entries(bt, r);
        const bool dedup = (swa.flags & CSA2_ATTN_DEDUP_WINDOW) && bt.m == 1;
        R.dlo = dedup ? lo : 1;                    // the window's entries, m = 1
        R.dhi = dedup ? t : 0;
        R.b = b;
    };
    if (tid == 0 && my_rows > 0) row_info(S.ri[0], row_of(0));
    if (swa.new_rows) {
        // decode (one query per sequence): each row's own window row, quantised as
        // the FP8 quantiser would, into ring row t % rows before any of this
        // cluster's rows attends -- one warp per row; each CTA writes its half of
        // the codes (the half it reads back) and both write the same scale
        for (int64_t i = warp; i < my_rows; i += AC_THREADS / 32) {
            const int64_t r = row_of(i);
            const int64_t off = (r / bt.nq) * swa.rows + bt.q_pos[r] % swa.rows;
            const float4 *nr = reinterpret_cast<const float4 *>(swa.new_rows + r * CSA2_HEAD_DIM);
            float4 v[4];
            float amax = 0.0f;
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                v[c4] = __ldg(nr + c4 * 32 + lane);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[c4].x), fabsf(v[c4].y)), fmaxf(fabsf(v[c4].z), fabsf(v[c4].w))));
            }
#pragma unroll
            for (int of = 16; of; of >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, of));
            const float sc = fp8_row_scale(amax);
            uint32_t *ring = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(swa.codes)) + off * (CSA2_HEAD_DIM / 4);
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {       // float4 chunks 64 dq + 32 h2 + lane: this CTA's dims
                const float4 x = dq == 0 ? v[h2] : v[2 + h2];
                ring[64 * dq + 32 * h2 + lane] = f32x2_to_e4m3x2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc)) |
                                                 (f32x2_to_e4m3x2(__fdiv_rn(x.z, sc), __fdiv_rn(x.w, sc)) << 16);
            }
            if (lane == 0) const_cast<float *>(swa.scales)[off] = sc;
        }
        __threadfence_block();                     // read back by this CTA (L2 loads) below
    }
    __syncthreads();

    // ---- a chunk's keys in three steps (registers only): its index, the index's
    //      page, the codes.  The loop keeps the index and page two chunks ahead and
    //      the codes one chunk ahead.
    uint4 kc[4];
    uint32_t ksc = 0;
    float kscale = 1.0f;
    bool valid = false;
    auto load_index = [&](int64_t i, int ch) -> int32_t {
        const int j = ch * AC_KEYS + key;
        return ch != nchunks - 1 && j < k ? __ldg(idx + row_of(i) * k + j) : -1;
    };
    auto load_page = [&](int ch, const RowInfo &R, int32_t p, int32_t &page) -> bool {
        if (ch == nchunks - 1 || p < 0 || (p >= R.dlo && p <= R.dhi)) return false;
        if (p >= R.vis) {
            if (hf == 0 && dq == 0) flag(c.status, CSA2_DEV_BAD_INDEX);
            return false;
        }
        page = __ldg(c.block_table + (int64_t)R.b * c.max_pages + (p >> 6));
        return true;
    };
    auto load_codes = [&](int ch, const RowInfo &R, int32_t p, int32_t page, bool ok) {
        valid = false;
        kscale = 1.0f;
        if (ch != nchunks - 1) {
            if (ok) {
                const int64_t slot = (int64_t)page * CSA2_PAGE + (p & 63);
                if (page < 0 || slot >= c.num_slots) {
                    flag(c.status, CSA2_DEV_BAD_PAGE);
                } else {
                    const uint4 *src =
                        reinterpret_cast<const uint4 *>(c.kv_codes + slot * 256 + AC_DIMS / 2 * dq) + 2 * hf;
                    kc[0] = __ldg(src);
                    kc[1] = __ldg(src + 1);
                    ksc = c.kv_format == CSA2_KV_FP4_E4M3
                              ? __ldg(reinterpret_cast<const uint32_t *>(c.kv_scales + slot * 32 + AC_DIMS / 16 * dq) + hf)
                              : __ldg(reinterpret_cast<const uint16_t *>(c.kv_scales + slot * 16 + AC_DIMS / 32 * dq) + hf);
                    valid = true;
                }
            }
        } else if (R.lo + key <= R.t) {
            const int64_t off = (int64_t)R.b * swa.rows + (R.lo + key) % swa.rows;
            const uint4 *src = reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM + AC_DIMS * dq) + 4 * hf;
#pragma unroll
            for (int u = 0; u < 4; u++) kc[u] = __ldcg(src + u);   // L2: rows this kernel wrote
            kscale = __ldcg(swa.scales + off);
            valid = true;
        }
    };
    // the chunk after the current one (index, page) and the one after that
    int32_t p1 = -1, page1 = -1, p2 = -1, page2 = -1;
    bool ok1 = false, ok2 = false;
    if (n_items > 0) {
        // chunk 0 now; chunk 1 (same row: every row has at least two chunks) to step 2
        int32_t p0 = load_index(0, 0), page0 = -1;
        const bool ok0 = load_page(0, S.ri[0], p0, page0);
        load_codes(0, S.ri[0], p0, page0, ok0);
        if (n_items > 1) {
            p1 = load_index(0, 1);
            ok1 = load_page(1, S.ri[0], p1, page1);
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // the other CTA's mbarriers exist
    const uint32_t tmem = S.tmem;

    // this thread's share of the output: dim 128 mt + 32 (warp & 3) + lane of this
    // CTA's slice, heads 32 hh .. 32 hh + 31 (owned by CTA hh)
    const int eu = warp >> 2, emt = eu >> 1, ehh = eu & 1;
    const int edim = AC_DIMS * (int)dq + 128 * emt + 32 * (warp & 3) + lane;
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; j++) acc[j] = 0.0f;
    // the owned head of this thread's softmax group: its running max and sum
    const int shl = tid >> 4, sh = AC_OWN * (int)dq + shl, spart = tid & 15;
    float m_run = -INFINITY, l_run = 0.0f;
    const float z = swa.sink ? swa.sink[sh] : -INFINITY;
    bool hard = false;

    // read out the finished chunk's O^T into acc; after a row's last chunk write o
    auto epilogue = [&](int64_t i, bool last) {
        const float *al = &S.xs[ehh][0][0];
        {                                          // hi, then lo
            const uint32_t col = 128u * (uint32_t)emt + 32u * (uint32_t)ehh;
            uint32_t ov[32];
            tc::tmem_ld32(tmem + lane_base + col, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j++) acc[j] = fmaf(acc[j], al[j], __uint_as_float(ov[j]));
            tc::tmem_ld32(tmem + lane_base + 64u + col, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j++) acc[j] += __uint_as_float(ov[j]);
        }
        if (!last) return;
        const float *mu = &S.xs[ehh][1][0];
#pragma unroll
        for (int j = 0; j < 32; j++) acc[j] *= mu[j];
        const int64_t r = row_of(i);
        // RoPE dims 448+i (lane quarter 2 of M-tile 1 of CTA 1) pair with 480+i
        // (quarter 3): the two warps of a head half swap values through pout
        if (rope && dq == 1 && emt == 1 && (warp & 3) >= 2) {
            const int qd = (warp & 3) - 2;
            float(*xch)[2][32][32] = reinterpret_cast<float(*)[2][32][32]>(&S.pout[0][0]);
#pragma unroll
            for (int j = 0; j < 32; j++) xch[ehh][qd][j][lane] = acc[j];
            tc::named_bar_sync(1, 128);
            float sn, cs;
            rope_sincos(S.ri[i & 1].t, turns.phi[lane], &sn, &cs);
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const float oth = xch[ehh][qd ^ 1][j][lane];
                // (a, b) -> (a cos + b sin, -a sin + b cos); qd 0 holds a, qd 1 holds b
                acc[j] = qd == 0 ? fmaf(acc[j], cs, oth * sn) : fmaf(acc[j], cs, -oth * sn);
            }
        }
        float *dst = o + (r * CSA2_HEADS + 32 * ehh) * CSA2_HEAD_DIM + edim;
#pragma unroll
        for (int j = 0; j < 32; j++) {
            dst[(int64_t)j * CSA2_HEAD_DIM] = acc[j];
            acc[j] = 0.0f;
        }
    };

    int64_t i = 0;                                 // row of the item (of this cluster's rows), chunk
    int ch = 0;
    for (int64_t it = 0; it < n_items; it++) {
        if (it > 0 && ++ch == nchunks) {
            ch = 0;
            i++;
        }
        const bool window = ch == nchunks - 1;
        const int64_t r = row_of(i);
        // the next item
        const int64_t ni = window ? i + 1 : i;
        const int nch = window ? 0 : ch + 1;
        const int64_t ni2 = nch == nchunks - 1 ? ni + 1 : ni;   // the chunk after that
        const int nch2 = nch == nchunks - 1 ? 0 : nch + 1;
        // ---- A: the previous chunk's product has finished: this chunk's keys into
        //      the key tile (and the row's query slice), then the previous chunk's
        //      output share
        if (it > 0) {
            hard = __syncthreads_or(!wait_phase(&S.mbar, 1, polls, c.status));
            if (hard) break;
            tc::tc_fence_after();
        }
        if (valid) {
            if (window) store_window_key(S.k, key, kc, hf);
            else if (c.kv_format == CSA2_KV_FP4_E4M3) store_main_key<true>(S.k, key, kc, ksc, hf, S.e2m1_pair, (uint32_t)lane);
            else store_main_key<false>(S.k, key, kc, ksc, hf, S.e2m1_pair, (uint32_t)lane);
        } else {
            zero_key(S.k, key, hf);
        }
        if (hf == 0) S.kscale[key] = valid ? kscale : -1.0f;
        if (ch == 0) {
            constexpr int QCH = AC_DIMS / 8;       // 16-byte chunks per head
            const uint4 *src = reinterpret_cast<const uint4 *>(q + r * CSA2_HEADS * CSA2_HEAD_DIM + AC_DIMS * dq);
            uint4 qv[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int e = tid + AC_THREADS * u;
                qv[u] = __ldg(src + (e / QCH) * (CSA2_HEAD_DIM / 8) + (e % QCH));
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int e = tid + AC_THREADS * u;
                *reinterpret_cast<uint4 *>(S.q + tc::sw128_offset(e / QCH, 8 * (e % QCH), CSA2_HEADS)) = qv[u];
            }
            // the next row's query slice into L2
            if (i + 1 < my_rows && tid < CSA2_HEADS * LPH)
                prefetch_l2(q + (row_of(i + 1) * CSA2_HEADS + tid / LPH) * CSA2_HEAD_DIM + AC_DIMS * dq +
                            64 * (tid % LPH));
        }
        if (it > 0) epilogue(ch == 0 ? i - 1 : i, ch == 0);
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();

        // ---- B: partial S^T = K_d Q_d^T over this CTA's dims
        if (tid == 0) {
            const uint32_t k0 = tc::smem_u32(S.k), q0 = tc::smem_u32(S.q);
#pragma unroll
            for (int kk = 0; kk < AC_DIMS / 16; kk++) {   // 16 dims per step
                const uint32_t off = (uint32_t)(kk >> 2) * (AC_KEYS * 128) + (uint32_t)(kk & 3) * 32u;
                const uint32_t offq = (uint32_t)(kk >> 2) * (CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                tc::mma_f16(tmem + AR_S_COL, tc::smem_desc(k0 + off, 16, 1024, tc::kSwizzle128B),
                            tc::smem_desc(q0 + offq, 16, 1024, tc::kSwizzle128B), AC_IDESC_S, kk > 0);
            }
            tc::mma_commit(&S.mbar);
        }
        // while the products run: the next chunk's codes (its page is known) and the
        // index of the chunk after it; the row after this one's scalars
        if (it + 1 < n_items) load_codes(nch, S.ri[ni & 1], p1, page1, ok1);
        if (it + 2 < n_items) p2 = load_index(ni2, nch2);
        if (ch == 0 && tid == 32 && i + 1 < my_rows) row_info(S.ri[(i + 1) & 1], row_of(i + 1));

        // ---- D: read the partials out; the other CTA's heads go to it
        hard = __syncthreads_or(!wait_phase(&S.mbar, 0, polls, c.status));
        if (hard) break;
        tc::tc_fence_after();
        {
            const uint32_t col = 16u * (uint32_t)(warp >> 2);   // 16 heads per warp
            uint32_t a16[16];
            tc::tmem_ld16(tmem + AR_S_COL + lane_base + col, a16);
            tc::tmem_ld_wait();
            const int kr = (warp & 3) * 32 + lane;
#pragma unroll
            for (int j = 0; j < 16; j++) S.pout[col + j][kr] = __uint_as_float(a16[j]);
        }
        if (it + 2 < n_items) ok2 = load_page(nch2, S.ri[ni2 & 1], p2, page2);
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_to_peer(cluster_map(tc::smem_u32(&S.ps[0][0]), peer), tc::smem_u32(&S.pout[AC_OWN * peer][0]),
                         AC_S_BYTES, cluster_map(tc::smem_u32(&S.sbar), peer));
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }

        // ---- E: owned heads: online softmax over the row; P rows and alpha to the other CTA
        hard = __syncthreads_or(!wait_phase(&S.sbar, (uint32_t)(it & 1), polls, c.status));
        if (hard) break;
        if (tid == 0 && it + 1 < n_items) tc::mbar_arrive_expect_tx(&S.sbar, AC_S_BYTES);
        {
            float4 v[2][2];
            const float *mine = &S.pout[sh][0], *theirs = &S.ps[shl][0];
            // rank order (CTA 0's partial first): the same sum in every run
            const float *first = dq == 0 ? mine : theirs, *second = dq == 0 ? theirs : mine;
            v[0][0] = *reinterpret_cast<const float4 *>(first + 8 * spart);
            v[0][1] = *reinterpret_cast<const float4 *>(first + 8 * spart + 4);
            v[1][0] = *reinterpret_cast<const float4 *>(second + 8 * spart);
            v[1][1] = *reinterpret_cast<const float4 *>(second + 8 * spart + 4);
            const float4 ks0 = *reinterpret_cast<const float4 *>(&S.kscale[8 * spart]);
            const float4 ks1 = *reinterpret_cast<const float4 *>(&S.kscale[8 * spart + 4]);
            const float ks[8] = {ks0.x, ks0.y, ks0.z, ks0.w, ks1.x, ks1.y, ks1.z, ks1.w};   // -1: no key
            float lg[8];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float4 &a = v[0][j >> 2], &b2 = v[1][j >> 2];
                const int e = j & 3;
                const float s0 = e == 0 ? a.x : e == 1 ? a.y : e == 2 ? a.z : a.w;
                const float s1 = e == 0 ? b2.x : e == 1 ? b2.y : e == 2 ? b2.z : b2.w;
                lg[j] = ks[j] >= 0.0f ? (s0 + s1) * (sm_scale * ks[j]) : -INFINITY;
                mx = fmaxf(mx, lg[j]);
            }
#pragma unroll
            for (int of = 1; of < 16; of <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, of));
            const float m_new = fmaxf(m_run, mx);
            float e[8], l = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                e[j] = m_new != -INFINITY && lg[j] != -INFINITY ? __expf(lg[j] - m_new) : 0.0f;
                l += e[j];
            }
#pragma unroll
            for (int of = 1; of < 16; of <<= 1) l += __shfl_xor_sync(0xffffffffu, l, of);
            const float alpha = m_run == -INFINITY ? 0.0f : expf(m_run - m_new);
            l_run = fmaf(l_run, alpha, l);
            m_run = m_new;
            uint32_t hi2[4], lo2[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const float p0 = e[j] * fmaxf(ks[j], 0.0f), p1 = e[j + 1] * fmaxf(ks[j + 1], 0.0f);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
                const float2 hf2 = __bfloat1622float2(hi);
                const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf2.x, p1 - hf2.y);
                hi2[j >> 1] = *reinterpret_cast<const uint32_t *>(&hi);
                lo2[j >> 1] = *reinterpret_cast<const uint32_t *>(&lo);
            }
            const uint32_t chunk16 = (uint32_t)((spart & 7) ^ (sh & 7)) << 4;
            const uint32_t off_hi = (uint32_t)(spart >> 3) * (2 * CSA2_HEADS * 128) + (uint32_t)sh * 128u + chunk16;
            *reinterpret_cast<uint4 *>(S.p + off_hi) = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
            *reinterpret_cast<uint4 *>(S.p + off_hi + CSA2_HEADS * 128) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
            if (spart == 0) {
                S.xs[dq][0][shl] = alpha;
                if (window) {
                    // the sink joins the denominator (the merge kernel's arithmetic)
                    float M = m_run, L = l_run, f = 1.0f;
                    if (z != -INFINITY) {
                        if (M == -INFINITY || z > M) {
                            f = M == -INFINITY ? 0.0f : expf(M - z);
                            L = fmaf(L, f, 1.0f);
                            M = z;
                        } else {
                            L += expf(z - M);
                        }
                    }
                    S.xs[dq][1][shl] = L > 0.0f ? f / L : 0.0f;
                    lse[r * CSA2_HEADS + sh] = L > 0.0f ? M + logf(L) : -INFINITY;
                }
            }
            if (window) {
                m_run = -INFINITY;
                l_run = 0.0f;
            }
        }
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            const uint32_t p0 = tc::smem_u32(S.p), pb = cluster_map(tc::smem_u32(&S.pbar), peer);
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {       // (slab, half) = (q4 >> 1, q4 & 1)
                const uint32_t off = (uint32_t)(q4 >> 1) * (2 * CSA2_HEADS * 128) +
                                     ((uint32_t)(q4 & 1) * CSA2_HEADS + AC_OWN * dq) * 128u;
                bulk_to_peer(cluster_map(p0 + off, peer), p0 + off, AC_P_ROWS_BYTES, pb);
            }
            const uint32_t xs = tc::smem_u32(&S.xs[dq][0][0]);
            bulk_to_peer(cluster_map(xs, peer), xs, AR_XS_BYTES, pb);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }

        // ---- F: [O_hi | O_lo]^T = V_d^T [P_hi | P_lo]^T (M-tiles of 128 dims, K = 128
        //      keys, N = 128); the read-out adds the halves
        hard = __syncthreads_or(!wait_phase(&S.pbar, (uint32_t)(it & 1), polls, c.status));
        if (hard) break;
        if (tid == 0 && it + 1 < n_items) tc::mbar_arrive_expect_tx(&S.pbar, AR_P_IN_BYTES);
        tc::tc_fence_after();
        if (tid == 0) {
            const uint32_t k0 = tc::smem_u32(S.k), p0 = tc::smem_u32(S.p);
#pragma unroll
            for (int mt = 0; mt < AC_MT; mt++) {
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {   // 16 keys per step
                    const uint64_t ad = tc::smem_desc(k0 + (uint32_t)(2 * mt) * (AC_KEYS * 128) + (uint32_t)kk * 2048u,
                                                      AC_KEYS * 128, 1024, tc::kSwizzle128B);
                    const uint32_t boff = (uint32_t)(kk >> 2) * (2 * CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                    tc::mma_f16(tmem + 128u * (uint32_t)mt, ad, tc::smem_desc(p0 + boff, 16, 1024, tc::kSwizzle128B),
                                AC_IDESC_O, kk > 0);
                }
            }
            tc::mma_commit(&S.mbar);
        }
        p1 = p2;                                   // the chunk after next becomes the next
        page1 = page2;
        ok1 = ok2;
    }
    if (!hard && n_items > 0) {
        hard = __syncthreads_or(!wait_phase(&S.mbar, 1, polls, c.status));
        tc::tc_fence_after();
        if (!hard) epilogue(my_rows - 1, true);
    }
    pdl_launch_dependents();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, AR_TMEM_COLS);
    // neither CTA leaves while the other may still copy into its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

int launch_attn_rows(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale,
                     const int32_t *idx, int k, const csa2_swa &swa, float *o, float *lse, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    const int nchunks = (k + AC_KEYS - 1) / AC_KEYS + 1;
    const size_t smem = sizeof(ArSmem) + 1024;
    if (const int s = kernel_smem_limit((const void *)k_attn_rows, smem, 100)) return s;
    const int sms = device_sms();
    const int64_t ncl = std::min<int64_t>(rows, std::max(1, sms / AC_CL));
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t ac = {};
    ac.gridDim = dim3((unsigned)(AC_CL * ncl));
    ac.blockDim = dim3(AC_THREADS);
    ac.dynamicSmemBytes = smem;
    ac.stream = st;
    ac.attrs = pdl;
    ac.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&ac, k_attn_rows, c, bt, q, sm_scale, idx, k, swa, o, lse, nchunks,
                                             rows, rope_turns(swa.rope_base), wait_polls());
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace csa2
