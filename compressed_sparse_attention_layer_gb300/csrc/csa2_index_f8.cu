// a4: the Full layer's lightning-indexer scan, TMA-fed e4m3 keys on the
// kind::f8f6f4 tensor cores.
//
// score(p) = s_p * sum_h w_h ReLU(qi_h . code_p) and the maximum of each
// aligned block of 8 positions ("DeepSeek-V4 report explainer" §3.2;
// "DeepSeek-V4.1-Flash" research note §3.2; "DeepSeek-V4.1-Flash 架构详解"
// §3.2).
//
// The keys stay e4m3 end to end: TMA copies each 64-entry page of codes
// (8 KB) into a 128-byte-swizzled shared-memory tile, which is directly the
// K-major A operand (M = 128 entries, K = 128 codes).  The indexer query is
// the B operand split into two e4m3 parts per head, hi = e4m3(q'), lo =
// e4m3(q' - hi), q' = q * 2^-e_h with max|q'| in [128, 256).  Per K step two
// N = 32 products (A x hi, then A x lo) accumulate into the same fp32
// D[128 entries x 32 heads] in tensor memory; the epilogue applies ReLU,
// w_h * 2^e_h and the entry's scale.
//
// Warp roles (192 threads): warp 0 issues TMA into a 12-stage ring, warp 1
// writes the query operand of each row and issues the MMAs (one thread),
// warps 2-5 drain four tensor-memory accumulators.  A persistent grid walks
// one global list of (row, tile) items so ragged batches stay balanced.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int F8_STAGES = 12;
constexpr int F8_ACC = 8;                  // tensor-memory accumulators of 32 columns
constexpr int F8_THREADS = 192;
constexpr int F8_TILE = 128;
constexpr int F8_PERSIST_ROWS = 256;
constexpr uint32_t F8_IDESC = tc::idesc_e4m3(128, 32);

struct F8Smem {
    uint8_t a[F8_STAGES][F8_TILE * 128];   // e4m3 keys, 128-byte swizzle (TMA)
    uint8_t b[2][64 * 128];                // query hi (rows 0-31) and lo (rows 32-63), per segment parity
    float wq[2][32];                       // w_h * 2^e_h, per segment parity
    uint64_t full[F8_STAGES], empty[F8_STAGES], tfull[F8_ACC], tempty[F8_ACC];
    uint64_t bfree[2], wready[2], wfree[2];
    uint32_t tmem;
    int abort;
    int32_t prefix[F8_PERSIST_ROWS + 1];
};

// e_h with max|q_h| * 2^-e_h in [128, 256).
__device__ __forceinline__ int head_exponent(float amax)
{
    if (!(amax > 0.0f)) return 0;
    const uint32_t u = __float_as_uint(amax);
    const int ex = (int)((u >> 23) & 0xFF);
    const int fl = ex ? ex - 127 : (31 - __clz(u & 0x7FFFFF)) - 149;
    const int e = fl - 7;
    return e < -126 ? -126 : (e > 120 ? 120 : e);
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte offset of element k of row `row` in a K-major 128-byte-swizzled tile of
// one-byte elements (128 elements per row).
__device__ __forceinline__ uint32_t sw128_b8(uint32_t row, uint32_t k)
{
    return row * 128u + ((((k >> 4) ^ (row & 7u)) << 4) | (k & 15u));
}

// Warp 1: the two-part e4m3 query operand of row r and w_h * 2^e_h; lane h = head h.
__device__ __forceinline__ void write_query_operand(uint8_t *b, float *wq, const uint16_t *qr, const float *wr)
{
    const int h = threadIdx.x & 31;
    const uint4 *src = reinterpret_cast<const uint4 *>(qr + h * 128);
    uint4 raw[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        raw[i] = __ldg(src + i);
        const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] & 0xFFFF0000u)));
        }
    }
    const int e = head_exponent(amax);
    const float f = exp2i(-e);
    wq[h] = wr[h] * exp2i(e);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {               // 16 dims per 16-byte chunk of the operand
        uint32_t hiw[4], low[4];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint32_t w4[4] = {raw[i + half].x, raw[i + half].y, raw[i + half].z, raw[i + half].w};
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                float v[4] = {__uint_as_float(w4[j] << 16) * f, __uint_as_float(w4[j] & 0xFFFF0000u) * f,
                              __uint_as_float(w4[j + 1] << 16) * f, __uint_as_float(w4[j + 1] & 0xFFFF0000u) * f};
                const uint32_t h01 = e4m3x2(v[0], v[1]), h23 = e4m3x2(v[2], v[3]);
                const float r0 = v[0] - e4m3_to_f32(h01 & 0xFF), r1 = v[1] - e4m3_to_f32(h01 >> 8);
                const float r2 = v[2] - e4m3_to_f32(h23 & 0xFF), r3 = v[3] - e4m3_to_f32(h23 >> 8);
                hiw[half * 2 + j / 2] = h01 | (h23 << 16);
                low[half * 2 + j / 2] = e4m3x2(r0, r1) | (e4m3x2(r2, r3) << 16);
            }
        }
        const uint32_t k = (uint32_t)i * 8;        // first dim of this 16-dim chunk
        *reinterpret_cast<uint4 *>(b + sw128_b8(h, k)) = make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
        *reinterpret_cast<uint4 *>(b + sw128_b8(32 + h, k)) = make_uint4(low[0], low[1], low[2], low[3]);
    }
}

template <bool PERSIST>
__global__ void __launch_bounds__(F8_THREADS, 1) k_index_f8(const __grid_constant__ CUtensorMap tmap, csa2_cache c,
                                                            csa2_batch bt, const uint16_t *__restrict__ qi,
                                                            const float *__restrict__ w, float *__restrict__ scores,
                                                            float *__restrict__ block_max,
                                                            int32_t *__restrict__ n_visible, int64_t ld)
{
    extern __shared__ uint8_t smem_raw[];
    F8Smem &S = *reinterpret_cast<F8Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = bt.batch * bt.nq;

    if (tid == 0) {
        for (int i = 0; i < F8_STAGES; i++) {
            tc::mbar_init(&S.full[i], 1);
            tc::mbar_init(&S.empty[i], 1);
        }
        for (int i = 0; i < F8_ACC; i++) {
            tc::mbar_init(&S.tfull[i], 1);
            tc::mbar_init(&S.tempty[i], 4);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&S.bfree[i], 1);
            tc::mbar_init(&S.wready[i], 32);
            tc::mbar_init(&S.wfree[i], 4);
        }
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(&S.tmem, F8_ACC * 32);

    int64_t g0, g1;
    if (PERSIST) {
        for (int r = tid; r < rows; r += F8_THREADS) {
            const int64_t nv = visible_entries(bt, r);
            S.prefix[r + 1] = (int32_t)((nv + F8_TILE - 1) / F8_TILE);
            if (blockIdx.x == 0 && n_visible) n_visible[r] = (int32_t)nv;
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
        const int64_t nv = visible_entries(bt, r);
        const int64_t T = (nv + F8_TILE - 1) / F8_TILE;
        if (blockIdx.x == 0 && tid == 0 && n_visible) n_visible[r] = (int32_t)nv;
        g0 = T * blockIdx.x / gridDim.x;
        g1 = T * (blockIdx.x + 1) / gridDim.x;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    volatile int *abort = &S.abort;

    // every role walks the same segments (consecutive tiles of one row)
    int r = PERSIST ? 0 : (int)blockIdx.y;
    int64_t g = g0, it = 0;
    int seg = 0;
    int last_full_k[F8_STAGES];
#pragma unroll
    for (int i = 0; i < F8_STAGES; i++) last_full_k[i] = -1;
    int64_t last_tile = -1;

    while (g < g1 && !*abort) {
        int64_t j0, nt;
        if (PERSIST) {
            while (S.prefix[r + 1] <= g) r++;
            j0 = g - S.prefix[r];
            nt = std::min<int64_t>(g1, S.prefix[r + 1]) - g;
        } else {
            j0 = g;
            nt = g1 - g;
        }
        const int b = r / bt.nq;
        const int64_t nvis = visible_entries(bt, r);

        if (warp == 0) {
            // ---------------- TMA producer: page ids of 32 tiles at a time, one lane per tile
            int32_t my_pg[2] = {-1, -1};
            for (int64_t i = 0; i < nt; i++) {
                if ((i & 31) == 0) {
                    const int64_t pt = (j0 + i + lane) * F8_TILE;     // tile i + lane
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int64_t e0 = pt + 64 * h;
                        my_pg[h] = -2;                                // -2: beyond the visible entries
                        if (i + lane < nt && e0 < nvis)
                            my_pg[h] = __ldg(c.block_table + (int64_t)b * c.max_pages + (e0 >> 6));
                    }
                }
                const int32_t pg0 = __shfl_sync(0xffffffffu, my_pg[0], (int)(i & 31));
                const int32_t pg1 = __shfl_sync(0xffffffffu, my_pg[1], (int)(i & 31));
                if (lane == 0) {
                    const int64_t ti = it + i;
                    const int stage = (int)(ti % F8_STAGES);
                    const int k = (int)(ti / F8_STAGES);
                    bool ok = true;
                    if (k > 0 && !tc::mbar_wait_or_abort(&S.empty[stage], (uint32_t)((k - 1) & 1), abort)) {
                        *abort = 1;
                        flag(c.status, CSA2_DEV_TIMEOUT);
                        ok = false;
                    }
                    if (ok) {
                        const int32_t pgs[2] = {pg0, pg1};
                        uint32_t bytes = 0;
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            if (pgs[h] == -2) continue;
                            if (pgs[h] >= 0 && ((int64_t)pgs[h] + 1) * CSA2_PAGE <= c.num_slots) bytes += 64 * 128;
                            else flag(c.status, CSA2_DEV_BAD_PAGE);
                        }
                        tc::mbar_arrive_expect_tx(&S.full[stage], bytes);
#pragma unroll
                        for (int h = 0; h < 2; h++)
                            if (pgs[h] >= 0 && ((int64_t)pgs[h] + 1) * CSA2_PAGE <= c.num_slots)
                                tc::tma_load_2d(S.a[stage] + h * 64 * 128, &tmap, 0, pgs[h] * CSA2_PAGE,
                                                &S.full[stage]);
                        last_full_k[stage] = k;
                    }
                }
                if (__shfl_sync(0xffffffffu, *abort, 0)) break;
            }
        } else if (warp == 1) {
            // ---------------- query operand + MMA issue
            // the operand and weights of segment seg-2 must be done with: its MMAs
            // completed (bfree) and the epilogue finished its tiles (wfree)
            bool ok = true;
            if (seg >= 2 && lane == 0) {
                const uint32_t par = (uint32_t)(((seg >> 1) - 1) & 1);
                ok = tc::mbar_wait_or_abort(&S.bfree[seg & 1], par, abort) &&
                     tc::mbar_wait_or_abort(&S.wfree[seg & 1], par, abort);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) {
                    *abort = 1;
                    flag(c.status, CSA2_DEV_TIMEOUT);
                }
            } else {
                write_query_operand(S.b[seg & 1], S.wq[seg & 1], qi + (int64_t)r * 4096, w + (int64_t)r * 32);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&S.wready[seg & 1]);
                __syncwarp();
                if (lane == 0) {
                    const uint32_t a0 = tc::smem_u32(S.a[0]);
                    const uint32_t b0 = tc::smem_u32(S.b[seg & 1]);
                    for (int64_t i = 0; i < nt; i++) {
                        const int64_t ti = it + i;
                        const int stage = (int)(ti % F8_STAGES);
                        const int acc = (int)(ti % F8_ACC);
                        if (!tc::mbar_wait_or_abort(&S.full[stage], (uint32_t)((ti / F8_STAGES) & 1), abort) ||
                            (ti >= F8_ACC &&
                             !tc::mbar_wait_or_abort(&S.tempty[acc], (uint32_t)(((ti / F8_ACC) - 1) & 1), abort))) {
                            *abort = 1;
                            flag(c.status, CSA2_DEV_TIMEOUT);
                            break;
                        }
                        tc::tc_fence_after();
                        const uint32_t as = a0 + (uint32_t)stage * (F8_TILE * 128);
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) {     // K = 128 codes in steps of 32
                            const uint64_t ad = tc::smem_desc(as + kk * 32, 16, 1024, tc::kSwizzle128B);
                            tc::mma_f8(tmem + (uint32_t)acc * 32u, ad,
                                       tc::smem_desc(b0 + kk * 32, 16, 1024, tc::kSwizzle128B), F8_IDESC, kk > 0);
                            tc::mma_f8(tmem + (uint32_t)acc * 32u, ad,
                                       tc::smem_desc(b0 + 32 * 128 + kk * 32, 16, 1024, tc::kSwizzle128B), F8_IDESC,
                                       1);
                        }
                        tc::mma_commit(&S.empty[stage]);
                        tc::mma_commit(&S.tfull[acc]);
                        last_tile = ti;
                    }
                    tc::mma_commit(&S.bfree[seg & 1]);
                }
                __syncwarp();
            }
        } else {
            // ---------------- epilogue: warps 2-5, TMEM lanes by warp % 4
            const int qd = warp & 3;
            const bool wok = tc::mbar_wait_or_abort(&S.wready[seg & 1], (uint32_t)((seg >> 1) & 1), abort);
            if (!__all_sync(0xffffffffu, wok)) {
                if (lane == 0) {
                    *abort = 1;
                    flag(c.status, CSA2_DEV_TIMEOUT);
                }
                break;
            }
            float wv[32];
#pragma unroll
            for (int h = 0; h < 32; h++) wv[h] = S.wq[seg & 1][h];
            // the scale of this lane's entry, two tiles ahead: page id for tile i+2,
            // scale for tile i+1, use for tile i
            const int64_t rowp = (int64_t)qd * 32 + lane;
            auto page_of = [&](int64_t i) -> int32_t {
                const int64_t p = (j0 + i) * F8_TILE + rowp;
                if (i >= nt || p >= nvis) return -2;
                return __ldg(c.block_table + (int64_t)b * c.max_pages + (p >> 6));
            };
            auto scale_of = [&](int64_t i, int32_t pg) -> float {
                const int64_t p = (j0 + i) * F8_TILE + rowp;
                if (pg == -2) return 0.0f;
                const int64_t slot = (int64_t)pg * CSA2_PAGE + (p & 63);
                if (pg < 0 || slot >= c.num_slots) return -INFINITY;            // bad page: score -inf
                return __ldg(c.ik_scales + slot);
            };
            int32_t pg_next = page_of(1);
            float sc_cur = scale_of(0, page_of(0));
            for (int64_t i = 0; i < nt; i++) {
                const int32_t pg_next2 = page_of(i + 2);
                const float sc_next = scale_of(i + 1, pg_next);
                const int64_t ti = it + i;
                const int acc = (int)(ti % F8_ACC);
                bool ok = tc::mbar_wait_or_abort(&S.tfull[acc], (uint32_t)((ti / F8_ACC) & 1), abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) {
                        *abort = 1;
                        flag(c.status, CSA2_DEV_TIMEOUT);
                    }
                    break;
                }
                tc::tc_fence_after();
                uint32_t d[32];
                tc::tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)acc * 32u, d);
                tc::tmem_ld_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&S.tempty[acc]);
                const int64_t p = (j0 + i) * F8_TILE + rowp;
                const bool valid = p < nvis;
                float sc = -INFINITY;
                if (valid) {
                    if (sc_cur != -INFINITY) {
                        float acc_s = 0.0f;
#pragma unroll
                        for (int h = 0; h < 32; h++)
                            acc_s = fmaf(wv[h], fmaxf(__uint_as_float(d[h]), 0.0f), acc_s);
                        sc = acc_s * sc_cur;
                    }
                    if (scores) scores[(int64_t)r * ld + p] = sc;
                }
                if (block_max) {
                    float m = valid ? sc : -INFINITY;
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if ((lane & 7) == 0 && valid) block_max[(int64_t)r * (ld / 8) + (p >> 3)] = m;
                }
                sc_cur = sc_next;
                pg_next = pg_next2;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.wfree[seg & 1]);   // this warp is done with seg's weights
        }
        g += nt;
        it += nt;
        seg++;
    }

    // ---- teardown: nothing in flight may outlive the CTA's shared and tensor memory
    __syncthreads();
    if (*abort) {
        if (tid == 0)
            for (int s = 0; s < F8_STAGES; s++)
                if (last_full_k[s] >= 0) tc::mbar_wait(&S.full[s], (uint32_t)(last_full_k[s] & 1), 1u << 20);
        if (tid == 32 && last_tile >= 0)
            tc::mbar_wait(&S.tfull[last_tile % F8_ACC], (uint32_t)((last_tile / F8_ACC) & 1), 1u << 20);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, F8_ACC * 32);
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;
static int g_sms = 0;

static int make_key_map(const csa2_cache &c, CUtensorMap *map)
{
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    });
    if (!g_encode) return CSA2_ERR_CUDA;
    const cuuint64_t dims[2] = {128, (cuuint64_t)c.num_slots};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 64};
    const cuuint32_t es[2] = {1, 1};
    const CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c.ik_codes, dims, strides, box, es,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? CSA2_OK : CSA2_ERR_CUDA;
}

int launch_index_scan(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi, const float *w,
                      float *scores, float *block_max, int32_t *n_visible, int64_t ld, cudaStream_t st)
{
    CUtensorMap map;
    int s = make_key_map(c, &map);
    if (s) return s;
    const int rows = bt.batch * bt.nq;
    const size_t smem = sizeof(F8Smem) + 1024;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_index_f8<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(k_index_f8<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    const int64_t tiles_row = std::max<int64_t>(1, (bt.max_entries + F8_TILE - 1) / F8_TILE);
    if (rows <= F8_PERSIST_ROWS) {
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)rows * tiles_row, g_sms));
        k_index_f8<true><<<grid, F8_THREADS, smem, st>>>(map, c, bt, qi, w, scores, block_max, n_visible, ld);
    } else {
        const int x = (int)std::max<int64_t>(1, std::min<int64_t>(tiles_row, ((int64_t)g_sms + rows - 1) / rows));
        k_index_f8<false><<<dim3(x, rows), F8_THREADS, smem, st>>>(map, c, bt, qi, w, scores, block_max, n_visible,
                                                                   ld);
    }
    return launch_status();
}

}  // namespace csa2
