// a9: sparse MQA + sliding-window attention on the tcgen05 tensor cores.
//
// Every key is its own value ("DeepSeek-V4 report explainer" §4.3) and one
// softmax covers the selected entries and the window ("DeepSeek-V4.1-Flash
// 架构详解" §1 table, §3; explainer §3.3).
//
// Split over keys: CTA (row, chunk) takes 128 keys -- chunks 0..3 the selected
// entries idx[128c .. 128c+127], the last chunk the window rows -- and all 64
// heads:
//   1. dequantise its keys into a 128 x 512 bf16 tile (MXFP4 e2m1 * 2^X is
//      exact in bf16; window codes e4m3 are exact, their fp32 row scale is
//      applied to the logit and to the probability instead);
//   2. S^T[128 keys x 64 heads] = K Q^T   (M = keys, N = heads, K = 512 dims);
//   3. per-head max m_c and sum l_c over the chunk, P = exp(S - m_c) split into
//      bf16 hi + lo (P = hi + lo to 2^-17);
//   4. O^T[512 dims x 64 heads] = V^T P^T with the same key tile read as an
//      MN-major operand (4 M-tiles of 128 dims, K = 128 keys, hi and lo);
//   5. the unnormalised partial O_c and (m_c, l_c) go to the workspace.
// A second kernel merges the chunks of each row: O = sum_c e^(m_c-M) O_c / L.
#include <cuda_bf16.h>

#include <algorithm>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int AC_THREADS = 128;
constexpr int AC_KEYS = 128;                       // keys per chunk (MMA M of the first product)
constexpr int AC_MAX_CHUNKS = CSA2_TOPK / AC_KEYS + 1;
constexpr uint32_t AC_IDESC_S = tc::idesc_f16(128, 64, 1, 1, 0, 0);   // K-major A and B
constexpr uint32_t AC_IDESC_O = tc::idesc_f16(128, 64, 1, 1, 1, 0);   // MN-major A (V^T)

struct AcSmem {
    uint8_t k[8 * AC_KEYS * 128];                  // [slab of 64 dims][128 keys][128 B]   128 KB
    union {
        uint8_t q[8 * CSA2_HEADS * 128];           // [slab][64 heads][128 B]              64 KB
        struct {
            float red[CSA2_HEADS][AC_KEYS];        // logits, transposed                  32 KB
            uint8_t p_hi[2 * CSA2_HEADS * 128];    // [slab of 64 keys][64 heads][128 B]  16 KB
            uint8_t p_lo[2 * CSA2_HEADS * 128];    //                                     16 KB
        } s;
    } u;
    float m[CSA2_HEADS], l[CSA2_HEADS];
    uint64_t mbar;
    uint32_t tmem;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// MXFP4 entry -> bf16 row of the key tile (exact).
__device__ __forceinline__ void store_main_key(uint8_t *ktile, uint32_t row, const uint8_t *codes,
                                               const uint8_t *scales)
{
    const uint4 sc = __ldg(reinterpret_cast<const uint4 *>(scales));
    const uint8_t *scb = reinterpret_cast<const uint8_t *>(&sc);
    const uint4 *src = reinterpret_cast<const uint4 *>(codes);
#pragma unroll 4
    for (int i = 0; i < 16; i++) {                 // 16 bytes = 32 elements = one MX block
        const uint4 u = __ldg(src + i);
        const float f = exp2i((int)scb[i] - 127 < -126 ? -126 : (int)scb[i] - 127);
        const float f2 = (int)scb[i] - 127 < -126 ? 0.5f : 1.0f;      // X = -127
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {              // 8 elements -> one 16-byte chunk
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const uint32_t b = (wd[j] >> (8 * e)) & 0xFFu;
                ow[e] = pack_bf16x2(e2m1_to_f32(b & 15u) * f * f2, e2m1_to_f32(b >> 4) * f * f2);
            }
            *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 32 * i + 8 * j, AC_KEYS)) = o;
        }
    }
}

// FP8 window row -> bf16 row of the key tile (codes only; exact).
__device__ __forceinline__ void store_window_key(uint8_t *ktile, uint32_t row, const uint8_t *codes)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(codes);
#pragma unroll 4
    for (int i = 0; i < 32; i++) {                 // 16 codes per load
        const uint4 u = __ldg(src + i);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
        uint4 o0, o1;
        uint32_t *a = reinterpret_cast<uint32_t *>(&o0);
        uint32_t *b = reinterpret_cast<uint32_t *>(&o1);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const uint32_t w = wd[e];
            const uint32_t v = pack_bf16x2(e4m3_to_f32(w & 0xFFu), e4m3_to_f32((w >> 8) & 0xFFu));
            const uint32_t v2 = pack_bf16x2(e4m3_to_f32((w >> 16) & 0xFFu), e4m3_to_f32(w >> 24));
            if (e < 2) {
                a[2 * e] = v;
                a[2 * e + 1] = v2;
            } else {
                b[2 * (e - 2)] = v;
                b[2 * (e - 2) + 1] = v2;
            }
        }
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 16 * i, AC_KEYS)) = o0;
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 16 * i + 8, AC_KEYS)) = o1;
    }
}

__device__ __forceinline__ void zero_key(uint8_t *ktile, uint32_t row)
{
#pragma unroll 8
    for (int i = 0; i < 64; i++)
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 8 * i, AC_KEYS)) = make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(AC_THREADS) k_attn_tc(csa2_cache c, csa2_batch bt,
                                                        const uint16_t *__restrict__ q, float sm_scale,
                                                        const int32_t *__restrict__ idx, int k, csa2_swa swa,
                                                        float *__restrict__ part_o, float *__restrict__ part_ml,
                                                        int nchunks)
{
    extern __shared__ uint8_t smem_raw[];
    AcSmem &S = *reinterpret_cast<AcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const int chunk = blockIdx.y;
    const int b = (int)(r / bt.nq);
    const bool window = chunk == nchunks - 1;

    if (tid == 0) {
        tc::mbar_init(&S.mbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem, 512);

    // ---- queries: 64 x 512 bf16, coalesced 16-byte loads into the swizzled B tile
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(q + r * CSA2_HEADS * CSA2_HEAD_DIM);
#pragma unroll 4
        for (int i = 0; i < 32; i++) {
            const int e = 8 * (tid + AC_THREADS * i);
            const uint4 v = __ldg(src + tid + AC_THREADS * i);
            *reinterpret_cast<uint4 *>(S.u.q + tc::sw128_offset(e >> 9, e & 511, CSA2_HEADS)) = v;
        }
    }

    // ---- this thread's key: dequantise into row tid of the key tile
    float kscale = 1.0f;          // multiplies the logit and the probability (window rows)
    bool valid = false;
    if (!window) {
        const int j = chunk * AC_KEYS + tid;
        if (j < k) {
            const int32_t p = idx[r * k + j];
            if (p >= 0) {
                if (p >= visible_entries(bt, r)) {
                    flag(c.status, CSA2_DEV_BAD_INDEX);
                } else {
                    const int64_t slot = entry_slot(c, b, p);
                    if (slot >= 0) {
                        store_main_key(S.k, tid, c.kv_codes + slot * 256, c.kv_scales + slot * 16);
                        valid = true;
                    }
                }
            }
        }
    } else {
        const int64_t t = bt.q_pos[r];
        const int64_t s0 = swa.start ? swa.start[b] : 0;
        int64_t lo = t - (CSA2_SWA_WINDOW - 1);
        lo = lo < s0 ? s0 : lo;
        lo = lo < 0 ? 0 : lo;
        if (lo + tid <= t) {
            const int64_t row = (lo + tid) % swa.rows;
            const int64_t off = (int64_t)b * swa.rows + row;
            store_window_key(S.k, tid, swa.codes + off * CSA2_HEAD_DIM);
            kscale = swa.scales[off];
            valid = true;
        }
    }
    if (!valid) zero_key(S.k, tid);

    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;

    // ---- S^T = K Q^T
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k), q0 = tc::smem_u32(S.u.q);
#pragma unroll
        for (int kk = 0; kk < 32; kk++) {          // 512 dims in steps of 16
            const uint32_t off = (uint32_t)(kk >> 2) * (AC_KEYS * 128) + (uint32_t)(kk & 3) * 32u;
            const uint32_t offq = (uint32_t)(kk >> 2) * (CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
            tc::mma_f16(tmem, tc::smem_desc(k0 + off, 16, 1024, tc::kSwizzle128B),
                        tc::smem_desc(q0 + offq, 16, 1024, tc::kSwizzle128B), AC_IDESC_S, kk > 0);
        }
        tc::mma_commit(&S.mbar);
    }
    bool ok = tc::mbar_wait(&S.mbar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);
        goto teardown;
    }
    tc::tc_fence_after();
    {
        // ---- logits of this thread's key for the 64 heads, transposed into smem
        const float lscale = sm_scale * kscale;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            uint32_t acc[32];
            tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)half * 32u, acc);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; h++)
                S.u.s.red[half * 32 + h][tid] = valid ? __uint_as_float(acc[h]) * lscale : -INFINITY;
        }
        __syncthreads();
        // ---- per-head max and sum over the chunk: two threads per head
        {
            const int h = tid >> 1, part = tid & 1;
            float mx = -INFINITY;
            for (int j = part; j < AC_KEYS; j += 2) mx = fmaxf(mx, S.u.s.red[h][j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            float sum = 0.0f;
            if (mx != -INFINITY)
                for (int j = part; j < AC_KEYS; j += 2) sum += expf(S.u.s.red[h][j] - mx);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            if (part == 0) {
                S.m[h] = mx;
                S.l[h] = sum;
            }
        }
        __syncthreads();
        // ---- P^T (times the window scale) as bf16 hi + lo, K-major rows = heads
#pragma unroll 4
        for (int h = 0; h < CSA2_HEADS; h++) {
            const float mx = S.m[h];
            const float p = (valid && mx != -INFINITY) ? expf(S.u.s.red[h][tid] - mx) * kscale : 0.0f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(p);
            const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
            const uint32_t off = tc::sw128_offset(h, tid, CSA2_HEADS);
            *reinterpret_cast<__nv_bfloat16 *>(S.u.s.p_hi + off) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(S.u.s.p_lo + off) = lo;
        }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- O^T = V^T P^T: 4 tiles of 128 dims, K = 128 keys, hi then lo
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k);
        const uint32_t ph = tc::smem_u32(S.u.s.p_hi), pl = tc::smem_u32(S.u.s.p_lo);
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            const uint32_t d = tmem + 64u + 64u * (uint32_t)mt;
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {       // 16 keys per step
                const uint64_t ad = tc::smem_desc(k0 + (uint32_t)(2 * mt) * (AC_KEYS * 128) + (uint32_t)kk * 2048u,
                                                  AC_KEYS * 128, 1024, tc::kSwizzle128B);
                const uint32_t boff = (uint32_t)(kk >> 2) * (CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                tc::mma_f16(d, ad, tc::smem_desc(ph + boff, 16, 1024, tc::kSwizzle128B), AC_IDESC_O, kk > 0);
                tc::mma_f16(d, ad, tc::smem_desc(pl + boff, 16, 1024, tc::kSwizzle128B), AC_IDESC_O, 1);
            }
        }
        tc::mma_commit(&S.mbar);
    }
    ok = tc::mbar_wait(&S.mbar, 1);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);
        goto teardown;
    }
    tc::tc_fence_after();
    {
        // ---- partial output: thread = dim within the M-tile, 64 heads per tile
        const int64_t base = (r * AC_MAX_CHUNKS + chunk) * (int64_t)CSA2_HEADS;
        float *po = part_o + base * CSA2_HEAD_DIM;
#pragma unroll 1
        for (int mt = 0; mt < 4; mt++) {
            const int d = 128 * mt + warp * 32 + (tid & 31);
#pragma unroll
            for (int half = 0; half < 2; half++) {
                uint32_t acc[32];
                tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 64u + 64u * (uint32_t)mt + 32u * (uint32_t)half,
                              acc);
                tc::tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 32; h++) po[(int64_t)(half * 32 + h) * CSA2_HEAD_DIM + d] = __uint_as_float(acc[h]);
            }
        }
        if (tid < CSA2_HEADS) {
            part_ml[(base + tid) * 2] = S.m[tid];
            part_ml[(base + tid) * 2 + 1] = S.l[tid];
        }
    }
teardown:
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// o = sum_c e^(m_c - M) O_c / sum_c e^(m_c - M) l_c, lse = M + log L; one CTA per
// (row, 8 heads), thread = 2 dims.
__global__ void __launch_bounds__(256) k_attn_combine(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_ml, int nchunks,
                                                      float *__restrict__ o, float *__restrict__ lse)
{
    const int64_t r = blockIdx.x;
    const int h0 = blockIdx.y * 8;
    const int tid = threadIdx.x;
#pragma unroll 1
    for (int hh = 0; hh < 8; hh++) {
        const int h = h0 + hh;
        float M = -INFINITY;
        for (int ch = 0; ch < nchunks; ch++)
            M = fmaxf(M, part_ml[((r * AC_MAX_CHUNKS + ch) * CSA2_HEADS + h) * 2]);
        float L = 0.0f;
        float2 acc = make_float2(0.0f, 0.0f);
        if (M != -INFINITY) {
            for (int ch = 0; ch < nchunks; ch++) {
                const int64_t base = (r * AC_MAX_CHUNKS + ch) * CSA2_HEADS + h;
                const float mc = part_ml[base * 2];
                if (mc == -INFINITY) continue;
                const float wgt = expf(mc - M);
                L += wgt * part_ml[base * 2 + 1];
                const float2 v = *reinterpret_cast<const float2 *>(part_o + base * CSA2_HEAD_DIM + 2 * tid);
                acc.x = fmaf(wgt, v.x, acc.x);
                acc.y = fmaf(wgt, v.y, acc.y);
            }
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        *reinterpret_cast<float2 *>(o + (r * CSA2_HEADS + h) * CSA2_HEAD_DIM + 2 * tid) =
            make_float2(acc.x * inv, acc.y * inv);
        if (tid == 0) lse[r * CSA2_HEADS + h] = L > 0.0f ? M + logf(L) : -INFINITY;
    }
}

size_t attn_workspace_bytes(int64_t rows)
{
    const size_t po = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4;
    const size_t ml = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * 2 * 4;
    return ((po + 255) & ~(size_t)255) + ml;
}

int launch_attn(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale, const int32_t *idx,
                int k, const csa2_swa &swa, float *o, float *lse, void *ws, size_t ws_bytes, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    if (ws_bytes < attn_workspace_bytes(rows) || !ws) return CSA2_ERR_WORKSPACE;
    const size_t po_bytes = ((size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4 + 255) & ~(size_t)255;
    float *part_o = static_cast<float *>(ws);
    float *part_ml = reinterpret_cast<float *>(static_cast<char *>(ws) + po_bytes);
    const int nchunks = (k + AC_KEYS - 1) / AC_KEYS + 1;
    const size_t smem = sizeof(AcSmem) + 1024;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    k_attn_tc<<<dim3((unsigned)rows, nchunks), AC_THREADS, smem, st>>>(c, bt, q, sm_scale, idx, k, swa, part_o,
                                                                       part_ml, nchunks);
    int s = launch_status();
    if (s) return s;
    k_attn_combine<<<dim3((unsigned)rows, CSA2_HEADS / 8), 256, 0, st>>>(part_o, part_ml, nchunks, o, lse);
    return launch_status();
}

}  // namespace csa2
