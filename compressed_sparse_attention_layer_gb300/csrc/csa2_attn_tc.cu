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

constexpr int AC_THREADS = 256;                   // two threads per key
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

// Half (`half` = 0: dims 0..255, 1: dims 256..511) of an MXFP4 entry -> bf16
// row of the key tile (exact).
__device__ __forceinline__ void store_main_key(uint8_t *ktile, uint32_t row, const uint8_t *codes,
                                               const uint8_t *scales, int half)
{
    const uint2 sc = __ldg(reinterpret_cast<const uint2 *>(scales) + half);
    const uint8_t *scb = reinterpret_cast<const uint8_t *>(&sc);
    const uint4 *src = reinterpret_cast<const uint4 *>(codes) + 8 * half;
#pragma unroll 4
    for (int ii = 0; ii < 8; ii++) {               // 16 bytes = 32 elements = one MX block
        const int i = ii + 8 * half;
        const uint4 u = __ldg(src + ii);
        const int X = (int)scb[ii] - 127;
        const float f = exp2i(X < -126 ? -126 : X);
        const float f2 = X < -126 ? 0.5f : 1.0f;      // X = -127
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

// Half of an FP8 window row -> bf16 row of the key tile (codes only; exact).
__device__ __forceinline__ void store_window_key(uint8_t *ktile, uint32_t row, const uint8_t *codes, int half)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(codes) + 16 * half;
#pragma unroll 4
    for (int ii = 0; ii < 16; ii++) {              // 16 codes per load
        const int i = ii + 16 * half;
        const uint4 u = __ldg(src + ii);
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

__device__ __forceinline__ void zero_key(uint8_t *ktile, uint32_t row, int half)
{
#pragma unroll 8
    for (int i = 32 * half; i < 32 * half + 32; i++)
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
    const int key = tid & (AC_KEYS - 1), half = tid >> 7;   // key row; half of the dims / heads
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // TMEM lane quarter of this warp
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
        for (int i = 0; i < 16; i++) {
            const int e = 8 * (tid + AC_THREADS * i);
            const uint4 v = __ldg(src + tid + AC_THREADS * i);
            *reinterpret_cast<uint4 *>(S.u.q + tc::sw128_offset(e >> 9, e & 511, CSA2_HEADS)) = v;
        }
    }

    // ---- this thread's key: dequantise its half into row `key` of the key tile
    float kscale = 1.0f;          // multiplies the logit and the probability (window rows)
    bool valid = false;
    if (!window) {
        const int j = chunk * AC_KEYS + key;
        if (j < k) {
            const int32_t p = idx[r * k + j];
            if (p >= 0) {
                if (p >= visible_entries(bt, r)) {
                    if (half == 0) flag(c.status, CSA2_DEV_BAD_INDEX);
                } else {
                    const int64_t slot = entry_slot(c, b, p);
                    if (slot >= 0) {
                        store_main_key(S.k, key, c.kv_codes + slot * 256, c.kv_scales + slot * 16, half);
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
        if (lo + key <= t) {
            const int64_t row = (lo + key) % swa.rows;
            const int64_t off = (int64_t)b * swa.rows + row;
            store_window_key(S.k, key, swa.codes + off * CSA2_HEAD_DIM, half);
            kscale = swa.scales[off];
            valid = true;
        }
    }
    if (!valid) zero_key(S.k, key, half);

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
        // ---- logits of this key for this half's 32 heads, transposed into smem
        const float lscale = sm_scale * kscale;
        {
            uint32_t acc[32];
            tc::tmem_ld32(tmem + lane_base + (uint32_t)half * 32u, acc);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; h++)
                S.u.s.red[half * 32 + h][key] = valid ? __uint_as_float(acc[h]) * lscale : -INFINITY;
        }
        __syncthreads();
        // ---- per-head max and sum over the chunk: four threads per head
        {
            const int h = tid >> 2, part = tid & 3;
            float mx = -INFINITY;
            for (int j = part; j < AC_KEYS; j += 4) mx = fmaxf(mx, S.u.s.red[h][j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            float sum = 0.0f;
            if (mx != -INFINITY)
                for (int j = part; j < AC_KEYS; j += 4) sum += expf(S.u.s.red[h][j] - mx);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) {
                S.m[h] = mx;
                S.l[h] = sum;
            }
        }
        __syncthreads();
        // ---- P^T (times the window scale) as bf16 hi + lo, K-major rows = heads
#pragma unroll 4
        for (int hh = 0; hh < 32; hh++) {
            const int h = half * 32 + hh;
            const float mx = S.m[h];
            const float p = (valid && mx != -INFINITY) ? expf(S.u.s.red[h][key] - mx) * kscale : 0.0f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(p);
            const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
            const uint32_t off = tc::sw128_offset(h, key, CSA2_HEADS);
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
        // ---- partial output: lane = dim within the M-tile, this half's 32 heads
        const int64_t base = (r * AC_MAX_CHUNKS + chunk) * (int64_t)CSA2_HEADS;
        float *po = part_o + base * CSA2_HEAD_DIM;
#pragma unroll 1
        for (int mt = 0; mt < 4; mt++) {
            const int d = 128 * mt + (warp & 3) * 32 + (tid & 31);
            uint32_t acc[32];
            tc::tmem_ld32(tmem + lane_base + 64u + 64u * (uint32_t)mt + 32u * (uint32_t)half, acc);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; h++) po[(int64_t)(half * 32 + h) * CSA2_HEAD_DIM + d] = __uint_as_float(acc[h]);
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
// (row, 4 heads), thread = 4 consecutive dims (float4), all chunk loads in flight.
__global__ void __launch_bounds__(128) k_attn_combine(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_ml, int nchunks,
                                                      float *__restrict__ o, float *__restrict__ lse)
{
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
#pragma unroll
    for (int hh = 0; hh < 4; hh++) {
        const int h = blockIdx.y * 4 + hh;
        float mc[AC_MAX_CHUNKS], lc[AC_MAX_CHUNKS];
        float4 v[AC_MAX_CHUNKS];
        float M = -INFINITY;
#pragma unroll
        for (int ch = 0; ch < AC_MAX_CHUNKS; ch++) {
            if (ch < nchunks) {
                const int64_t base = (r * AC_MAX_CHUNKS + ch) * CSA2_HEADS + h;
                const float2 ml = *reinterpret_cast<const float2 *>(part_ml + base * 2);
                mc[ch] = ml.x;
                lc[ch] = ml.y;
                v[ch] = *reinterpret_cast<const float4 *>(part_o + base * CSA2_HEAD_DIM + 4 * tid);
                M = fmaxf(M, ml.x);
            } else {
                mc[ch] = -INFINITY;
                lc[ch] = 0.0f;
                v[ch] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float L = 0.0f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int ch = 0; ch < AC_MAX_CHUNKS; ch++) {
                if (mc[ch] == -INFINITY) continue;
                const float wgt = expf(mc[ch] - M);
                L = fmaf(wgt, lc[ch], L);
                acc.x = fmaf(wgt, v[ch].x, acc.x);
                acc.y = fmaf(wgt, v[ch].y, acc.y);
                acc.z = fmaf(wgt, v[ch].z, acc.z);
                acc.w = fmaf(wgt, v[ch].w, acc.w);
            }
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        *reinterpret_cast<float4 *>(o + (r * CSA2_HEADS + h) * CSA2_HEAD_DIM + 4 * tid) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
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
    k_attn_combine<<<dim3((unsigned)rows, CSA2_HEADS / 4), 128, 0, st>>>(part_o, part_ml, nchunks, o, lse);
    return launch_status();
}

}  // namespace csa2
