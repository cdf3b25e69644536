// a7: lightning-indexer scores of a gathered list of entries on the tcgen05
// tensor cores -- a Reindex layer rescoring its candidate pool
// ("DeepSeek-V4.1-Flash 架构详解" §3 mode table, §3.2).  The same kernel
// also scores every visible entry (template flag POOL = false); the Full
// layer's scan itself runs on the TMA-fed e4m3 kernel.
//
// score(p) = s_p * sum_h w_h ReLU(qi_h . code_p)
// ("DeepSeek-V4 report explainer" §3.2).
//
// Per 128-entry tile: D[128 entries x 32 heads] = A[128 x 128] * B[32 x 128]^T
// with A = the e4m3 key codes widened to f16 (exact) and B = the indexer query
// in f16, each head scaled by a power of two 2^-e_h that brings its largest
// element into [2^14, 2^15) (exact; 2^e_h is folded into w_h).  The
// accumulator lives in tensor memory; the epilogue applies ReLU, the head
// weights and the entry's fp32 scale in registers.
//
// CTA = 4 warps; thread t owns entry t of a tile: it loads the entry's 128
// code bytes (eight 16-byte loads, two tiles ahead in registers), widens
// them, stores them into the 128-byte-swizzled K-major A tile, and later
// reads TMEM lane t for the epilogue.  Two shared-memory stages and two TMEM
// accumulators let the MMA of tile i+1 run while tile i is scored.  A
// persistent grid walks one global list of (row, tile) work items so ragged
// batches stay balanced.
#include <cuda_fp16.h>

#include <algorithm>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int TS_THREADS = 128;
constexpr int TS_TILE = 128;              // entries per tile (MMA M)
constexpr int TS_HEADS = 32;              // indexer heads (MMA N)
constexpr int TS_PERSIST_ROWS = 256;      // rows handled by the persistent work list
constexpr uint32_t TS_IDESC = tc::idesc_f16(TS_TILE, TS_HEADS, 0, 0, 0, 0);

struct TsSmem {
    uint8_t a[2][2 * TS_TILE * 128];      // [stage][slab of 64 dims][128 rows][128 B]
    uint8_t b[2 * TS_HEADS * 128];        // [slab][32 rows][128 B]
    float w[TS_HEADS];                    // w_h * 2^e_h
    uint64_t mbar[2];
    uint32_t tmem;
    int32_t prefix[TS_PERSIST_ROWS + 1];
};

// Two e4m3 bytes (low half of `v`) -> f16x2, exact.
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t v)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)(v & 0xFFFFu)));
    return r;
}

struct KeyRegs {
    uint4 c[8];
    float scale;
    int state;        // 0 = no entry (zeros), 1 = valid, 2 = bad slot
};

__device__ __forceinline__ void key_load(const csa2_cache &c, int b, int64_t p, int64_t nvis, KeyRegs &k)
{
    k.state = 0;
    k.scale = 0.0f;
    if (p < nvis) {
        const int64_t slot = entry_slot(c, b, p);
        if (slot >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(c.ik_codes + slot * 128);
#pragma unroll
            for (int i = 0; i < 8; i++) k.c[i] = __ldg(src + i);
            k.scale = __ldg(c.ik_scales + slot);
            k.state = 1;
            return;
        }
        k.state = 2;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) k.c[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Widen the 128 codes of one entry to f16 and store them as row `row` of the
// swizzled A tile.
__device__ __forceinline__ void key_store(uint8_t *a, uint32_t row, const KeyRegs &k)
{
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint4 u = k.c[i];
        uint4 lo, hi;
        lo.x = cvt_e4m3x2(u.x);
        lo.y = cvt_e4m3x2(u.x >> 16);
        lo.z = cvt_e4m3x2(u.y);
        lo.w = cvt_e4m3x2(u.y >> 16);
        hi.x = cvt_e4m3x2(u.z);
        hi.y = cvt_e4m3x2(u.z >> 16);
        hi.z = cvt_e4m3x2(u.w);
        hi.w = cvt_e4m3x2(u.w >> 16);
        *reinterpret_cast<uint4 *>(a + tc::sw128_offset(row, 16 * i, TS_TILE)) = lo;
        *reinterpret_cast<uint4 *>(a + tc::sw128_offset(row, 16 * i + 8, TS_TILE)) = hi;
    }
}

// B operand for row r: head h scaled by 2^-e_h into f16, w_h * 2^e_h.
__device__ __forceinline__ void load_query(TsSmem &S, const uint16_t *qr, const float *wr)
{
    const int tid = threadIdx.x;
    const int h = tid >> 2, part = tid & 3;           // 4 threads per head, 32 dims each
    const uint16_t *src = qr + h * 128 + part * 32;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v[i] = bf16_to_f32(src[i]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (amax > 0.0f) {
        const uint32_t u = __float_as_uint(amax);
        const int ex = (int)((u >> 23) & 0xFF);
        const int fl = ex ? ex - 127 : (31 - __clz(u & 0x7FFFFF)) - 149;
        e = fl - 14;
        e = e < -126 ? -126 : (e > 113 ? 113 : e);   // keeps 2^e and 2^-e normal floats
    }
    const float f = exp2i(-e);                       // exact scaling by a power of two
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        uint4 o;
        uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const __half2 hv = __floats2half2_rn(v[i + 2 * j] * f, v[i + 2 * j + 1] * f);
            ow[j] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        *reinterpret_cast<uint4 *>(S.b + tc::sw128_offset(h, part * 32 + i, TS_HEADS)) = o;
    }
    if (part == 0) S.w[h] = wr[h] * exp2i(e);
}

__device__ __forceinline__ void issue_tile_mma(const TsSmem &S, int stage, uint32_t d_tmem)
{
    const uint32_t a0 = tc::smem_u32(S.a[stage]);
    const uint32_t b0 = tc::smem_u32(S.b);
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {                 // K = 128 in steps of 16
        const uint32_t off = (uint32_t)(kk & 3) * 32u;      // 16 f16 = 32 B within the swizzled row
        const uint64_t ad = tc::smem_desc(a0 + (kk >> 2) * (TS_TILE * 128) + off, 16, 1024, tc::kSwizzle128B);
        const uint64_t bd = tc::smem_desc(b0 + (kk >> 2) * (TS_HEADS * 128) + off, 16, 1024, tc::kSwizzle128B);
        tc::mma_f16(d_tmem, ad, bd, TS_IDESC, kk > 0);
    }
}

// Entries scored by row r: every visible entry (the Full layer's scan) or the
// first pool_len[r] positions of its candidate pool (a Reindex layer).
template <bool POOL>
__device__ __forceinline__ int64_t row_entries(const csa2_batch &bt, const int32_t *pool_len, int64_t ld, int r)
{
    if (!POOL) return visible_entries(bt, r);
    int64_t n = pool_len[r];
    return n < 0 ? 0 : (n > ld ? ld : n);
}

template <bool PERSIST, bool POOL>
__global__ void __launch_bounds__(TS_THREADS) k_index_tc(csa2_cache c, csa2_batch bt,
                                                         const uint16_t *__restrict__ qi,
                                                         const float *__restrict__ w,
                                                         const int32_t *__restrict__ pool,
                                                         const int32_t *__restrict__ pool_len,
                                                         float *__restrict__ scores,
                                                         float *__restrict__ block_max,
                                                         int32_t *__restrict__ n_visible, int64_t ld)
{
    extern __shared__ uint8_t smem_raw[];
    TsSmem &S = *reinterpret_cast<TsSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int rows = bt.batch * bt.nq;

    if (tid == 0) {
        tc::mbar_init(&S.mbar[0], 1);
        tc::mbar_init(&S.mbar[1], 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem, 64);
    pdl_launch_dependents();                      // programmatic dependent launch: inputs are read
    pdl_wait();                                   // below, once the previous kernel is done

    // ---- this CTA's range of global tiles
    int64_t g0, g1;
    if (PERSIST) {
        for (int r = tid; r < rows; r += TS_THREADS) {
            const int64_t nv = row_entries<POOL>(bt, pool_len, ld, r);
            S.prefix[r + 1] = (int32_t)((nv + TS_TILE - 1) / TS_TILE);
            if (!POOL && blockIdx.x == 0 && n_visible) n_visible[r] = (int32_t)nv;
        }
        __syncthreads();
        if (tid == 0) {
            S.prefix[0] = 0;
            for (int r = 0; r < rows; r++) S.prefix[r + 1] += S.prefix[r];
        }
        __syncthreads();
        const int64_t total = S.prefix[rows];
        g0 = total * blockIdx.x / gridDim.x;
        g1 = total * (blockIdx.x + 1) / gridDim.x;
    } else {
        const int r = blockIdx.y;
        const int64_t nv = row_entries<POOL>(bt, pool_len, ld, r);
        const int64_t T = (nv + TS_TILE - 1) / TS_TILE;
        if (!POOL && blockIdx.x == 0 && tid == 0 && n_visible) n_visible[r] = (int32_t)nv;
        g0 = T * blockIdx.x / gridDim.x;
        g1 = T * (blockIdx.x + 1) / gridDim.x;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    uint32_t parity[2] = {0u, 0u};
    bool aborted = false;

    int r = PERSIST ? 0 : (int)blockIdx.y;
    int64_t g = g0;
    while (g < g1 && !aborted) {
        // ---- one segment: consecutive tiles of one row
        int64_t j0, nt;
        if (PERSIST) {
            while (S.prefix[r + 1] <= g) r++;
            j0 = g - S.prefix[r];
            nt = std::min<int64_t>(g1, S.prefix[r + 1]) - g;
        } else {
            j0 = g;
            nt = g1 - g;
        }
        g += nt;
        const int b = r / bt.nq;
        const int64_t nvis = visible_entries(bt, r);
        const int64_t n = row_entries<POOL>(bt, pool_len, ld, r);
        const int32_t *prow = POOL ? pool + (int64_t)r * ld : nullptr;
        // slot i of the row -> entry position (pool rows list positions)
        auto load_slot = [&](int64_t i, KeyRegs &kr) {
            if (!POOL) {
                key_load(c, b, i, nvis, kr);
                return;
            }
            int64_t p = i < n ? (int64_t)prow[i] : nvis;
            if (i < n && (p < 0 || p >= nvis)) {
                flag(c.status, CSA2_DEV_BAD_INDEX);
                p = nvis;
            }
            key_load(c, b, p, nvis, kr);
            if (i < n && kr.state == 0) kr.state = 2;
        };
        load_query(S, qi + (int64_t)r * 4096, w + (int64_t)r * 32);

        KeyRegs ka, kb;                             // tiles of even / odd index
        load_slot(j0 * TS_TILE + tid, ka);
        key_store(S.a[0], tid, ka);
        float scale_even = ka.scale;
        int state_even = ka.state;
        float scale_odd = 0.0f;
        int state_odd = 0;
        if (nt > 1) load_slot((j0 + 1) * TS_TILE + tid, kb);
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::tc_fence_after();
            issue_tile_mma(S, 0, tmem);
            tc::mma_commit(&S.mbar[0]);
        }

        for (int64_t i = 0; i < nt; i++) {
            const int s = (int)(i & 1);
            float scale_cur;
            int state_cur;
            // stage tile i+1 (registers loaded one iteration ago), start loading tile i+2
            if (s == 0) {
                scale_cur = scale_even;
                state_cur = state_even;
                if (i + 1 < nt) {
                    key_store(S.a[1], tid, kb);
                    scale_odd = kb.scale;
                    state_odd = kb.state;
                }
                if (i + 2 < nt) load_slot((j0 + i + 2) * TS_TILE + tid, ka);
            } else {
                scale_cur = scale_odd;
                state_cur = state_odd;
                if (i + 1 < nt) {
                    key_store(S.a[0], tid, ka);
                    scale_even = ka.scale;
                    state_even = ka.state;
                }
                if (i + 2 < nt) load_slot((j0 + i + 2) * TS_TILE + tid, kb);
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncthreads();
            if (tid == 0 && i + 1 < nt) {
                tc::tc_fence_after();
                issue_tile_mma(S, s ^ 1, tmem + (uint32_t)(s ^ 1) * 32u);
                tc::mma_commit(&S.mbar[s ^ 1]);
            }
            // ---- epilogue of tile i
            const bool ok = tc::mbar_wait(&S.mbar[s], parity[s]);
            parity[s] ^= 1u;
            if (__syncthreads_or(!ok)) {
                if (tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);
                aborted = true;
                break;
            }
            tc::tc_fence_after();
            uint32_t acc[32];
            tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)s * 32u, acc);
            tc::tmem_ld_wait();
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < 32; h++) sc = fmaf(S.w[h], fmaxf(__uint_as_float(acc[h]), 0.0f), sc);
            sc *= scale_cur;
            if (state_cur != 1) sc = -INFINITY;
            const int64_t p = (j0 + i) * TS_TILE + tid;
            const bool valid = p < n;
            if (valid && scores) scores[(int64_t)r * ld + p] = sc;
            if (!POOL && block_max) {
                float m = valid ? sc : -INFINITY;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if ((tid & 7) == 0 && valid) block_max[(int64_t)r * (ld / 8) + (p >> 3)] = m;
            }
            tc::tc_fence_before();
        }
        // the segment's MMAs have all been waited for: the B operand may change
        __syncthreads();
    }
    if (aborted) {
        // let any MMA still in flight finish before the accumulator is freed
        if (tid == 0) {
            tc::mbar_wait(&S.mbar[0], parity[0], 1u << 20);
            tc::mbar_wait(&S.mbar[1], parity[1], 1u << 20);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

static int g_num_sms = 0;

template <bool POOL>
static int launch_index(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                        const int32_t *pool, const int32_t *pool_len, float *scores, float *block_max,
                        int32_t *n_visible, int64_t ld, cudaStream_t st)
{
    const int rows = bt.batch * bt.nq;
    const size_t smem = sizeof(TsSmem) + 1024;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_index_tc<true, POOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(k_index_tc<false, POOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (!g_num_sms) {
            int dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        }
        attr = true;
    }
    const int per_sm = 3;
    const int64_t per_row = POOL ? ld : bt.max_entries;
    const int64_t tiles_row = std::max<int64_t>(1, (per_row + TS_TILE - 1) / TS_TILE);
    if (rows <= TS_PERSIST_ROWS) {
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(rows * tiles_row, (int64_t)g_num_sms * per_sm));
        return launch_pdl(k_index_tc<true, POOL>, dim3(grid), dim3(TS_THREADS), smem, st, c, bt, qi, w, pool,
                          pool_len, scores, block_max, n_visible, ld);
    }
    const int x = (int)std::max<int64_t>(1, std::min<int64_t>(tiles_row, ((int64_t)g_num_sms * per_sm + rows - 1) / rows));
    return launch_pdl(k_index_tc<false, POOL>, dim3(x, rows), dim3(TS_THREADS), smem, st, c, bt, qi, w, pool, pool_len,
                      scores, block_max, n_visible, ld);
}

// a7: a Reindex layer rescoring its candidate pool ("DeepSeek-V4.1-Flash 架构详解" §3.2).
int launch_index_pool(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                      const int32_t *pool, const int32_t *pool_len, int64_t ld, float *scores, cudaStream_t st)
{
    return launch_index<true>(c, bt, qi, w, pool, pool_len, scores, nullptr, nullptr, ld, st);
}

}  // namespace csa2
