// a9: sparse MQA + sliding-window attention on the tcgen05 tensor cores.
//
// Every key is its own value ("DeepSeek-V4 report explainer" §4.3) and one
// softmax covers the selected entries and the window ("DeepSeek-V4.1-Flash
// 架构详解" §1 table, §3; explainer §3.3).
//
// Split over keys: CTA (row, chunk) takes 128 keys -- chunks 0..3 the selected
// entries idx[128c .. 128c+127], the last chunk the window rows -- and all 64
// heads:
//   1. dequantise its keys into a 128 x 512 bf16 tile: MXFP4 bytes through a
//      256-entry table (byte -> two bf16 magnitudes with signs) and one bf16x2
//      multiply by 2^X per block; window codes e4m3 by placing their bits in a
//      bf16 and one multiply by 2^120 -- both exact; the window's fp32 row scale
//      is applied to the logit and to the probability instead;
//   2. S^T[128 keys x 64 heads] = K Q^T   (M = keys, N = heads, K = 512 dims);
//   3. per-head max m_c and sum l_c over the chunk, P = exp(S - m_c) split into
//      bf16 hi + lo (P = hi + lo to 2^-17), stacked as one 128-row operand;
//   4. [O_hi | O_lo]^T[512 dims x 128] = V^T [P_hi | P_lo]^T with the same key
//      tile read as an MN-major operand (4 M-tiles of 128 dims, K = 128 keys,
//      N = 128); the epilogue adds the two halves;
//   5. the unnormalised partial O_c and (m_c, l_c) go to the workspace.
// A second kernel merges the chunks of each row: O = sum_c e^(m_c-M) O_c / L.
// 512 threads: four per key (128 dims each) for the loads and dequantisation,
// eight per head for the softmax statistics, one M-tile row each for the
// epilogue.
#include <cuda_bf16.h>

#include <algorithm>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int AC_THREADS = 512;
constexpr int AC_KEYS = 128;                       // keys per chunk (MMA M of the first product)
constexpr int AC_MAX_CHUNKS = CSA2_TOPK / AC_KEYS + 1;
constexpr uint32_t AC_IDESC_S = tc::idesc_f16(128, 64, 1, 1, 0, 0);   // K-major A and B
constexpr uint32_t AC_IDESC_O = tc::idesc_f16(128, 128, 1, 1, 1, 0);  // MN-major A (V^T), N = hi|lo

struct AcSmem {
    uint8_t k[8 * AC_KEYS * 128];                  // [slab of 64 dims][128 keys][128 B]   128 KB
    union {
        uint8_t q[8 * CSA2_HEADS * 128];           // [slab][64 heads][128 B]              64 KB
        struct {
            float red[CSA2_HEADS][AC_KEYS];        // logits, transposed                  32 KB
            uint8_t p[2 * 2 * CSA2_HEADS * 128];   // [slab of 64 keys][hi 64 | lo 64 rows][128 B] 32 KB
        } s;
    } u;
    uint32_t e2m1_pair[256];                       // byte -> bf16x2 of its two E2M1 codes
    float m[CSA2_HEADS], l[CSA2_HEADS];
    float kscale[AC_KEYS];
    int valid[AC_KEYS];
    uint64_t mbar;
    uint32_t tmem;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// a (bf16x2) * b (bf16x2), exact when the products are representable.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(0x80008000u));
    return r;
}

// 2^X (X in [-127, 127]) as a bf16, in both halves.
__device__ __forceinline__ uint32_t pow2_bf16x2(int X)
{
    const uint32_t h = X >= -126 ? (uint32_t)(X + 127) << 7 : 0x0040u;   // 2^-127 is subnormal
    return h | (h << 16);
}

// Quarter `qt` (dims 128 qt .. 128 qt + 127) of an MXFP4 entry -> bf16 row of
// the key tile (exact): the table gives the two E2M1 magnitudes of a byte with
// their signs, one bf16x2 multiply applies the block's 2^X.
__device__ __forceinline__ void store_main_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[4], uint32_t sc,
                                               int qt, const uint32_t *pair)
{
#pragma unroll
    for (int blk = 0; blk < 4; blk++) {            // 16 bytes = 32 elements = one MX block
        const uint32_t f = pow2_bf16x2((int)((sc >> (8 * blk)) & 0xFFu) - 127);
        const uint32_t w[4] = {c[blk].x, c[blk].y, c[blk].z, c[blk].w};
#pragma unroll
        for (int j = 0; j < 4; j++) {              // 4 bytes = 8 elements -> one 16-byte chunk
            uint4 o;
            o.x = bf16x2_mul(pair[w[j] & 0xFFu], f);
            o.y = bf16x2_mul(pair[(w[j] >> 8) & 0xFFu], f);
            o.z = bf16x2_mul(pair[(w[j] >> 16) & 0xFFu], f);
            o.w = bf16x2_mul(pair[w[j] >> 24], f);
            *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qt + 32 * blk + 8 * j, AC_KEYS)) = o;
        }
    }
}

// Two e4m3 codes (low bytes of the halves of v) -> bf16x2 of their values:
// sign and the 7 exponent/mantissa bits moved into bf16 position give the
// value times 2^-120, which one exact multiply by 2^120 restores (subnormal
// codes included).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t v)
{
    const uint32_t bits = ((v & 0x007F007Fu) << 4) | ((v & 0x00800080u) << 8);
    return bf16x2_mul(bits, 0x7B807B80u);          // 2^120 in both halves
}

// Quarter `qt` of an FP8 window row -> bf16 row of the key tile (codes only; exact).
__device__ __forceinline__ void store_window_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[8], int qt)
{
#pragma unroll
    for (int i = 0; i < 8; i++) {                  // 16 codes per load -> two 16-byte chunks
        const uint32_t w[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
        uint4 o0, o1;
        o0.x = e4m3x2_to_bf16x2(__byte_perm(w[0], 0, 0x4140));
        o0.y = e4m3x2_to_bf16x2(__byte_perm(w[0], 0, 0x4342));
        o0.z = e4m3x2_to_bf16x2(__byte_perm(w[1], 0, 0x4140));
        o0.w = e4m3x2_to_bf16x2(__byte_perm(w[1], 0, 0x4342));
        o1.x = e4m3x2_to_bf16x2(__byte_perm(w[2], 0, 0x4140));
        o1.y = e4m3x2_to_bf16x2(__byte_perm(w[2], 0, 0x4342));
        o1.z = e4m3x2_to_bf16x2(__byte_perm(w[3], 0, 0x4140));
        o1.w = e4m3x2_to_bf16x2(__byte_perm(w[3], 0, 0x4342));
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qt + 16 * i, AC_KEYS)) = o0;
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qt + 16 * i + 8, AC_KEYS)) = o1;
    }
}

__device__ __forceinline__ void zero_key(uint8_t *ktile, uint32_t row, int qt)
{
#pragma unroll 4
    for (int i = 16 * qt; i < 16 * qt + 16; i++)
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 8 * i, AC_KEYS)) = make_uint4(0, 0, 0, 0);
}

// 16 consecutive 32-bit TMEM columns of this warp's lane quarter.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__global__ void __launch_bounds__(AC_THREADS, 1) k_attn_tc(csa2_cache c, csa2_batch bt,
                                                           const uint16_t *__restrict__ q, float sm_scale,
                                                           const int32_t *__restrict__ idx, int k, csa2_swa swa,
                                                           float *__restrict__ part_o, float *__restrict__ part_ml,
                                                           int nchunks)
{
    extern __shared__ uint8_t smem_raw[];
    AcSmem &S = *reinterpret_cast<AcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int key = tid & (AC_KEYS - 1), qt = tid >> 7;          // key row; quarter of the dims / heads
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16; // TMEM lane quarter of this warp
    const int64_t r = blockIdx.x;
    const int chunk = blockIdx.y;
    const int b = (int)(r / bt.nq);
    const bool window = chunk == nchunks - 1;

    if (tid == 0) {
        tc::mbar_init(&S.mbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem, 512);
    if (tid < 256) {                               // E2M1 pair table
        const uint32_t lo = tid & 15u, hi = tid >> 4;
        S.e2m1_pair[tid] = pack_bf16x2(e2m1_to_f32(lo), e2m1_to_f32(hi));
    }

    // ---- this thread's key: locate it and start loading its quarter
    float kscale = 1.0f;          // multiplies the logit and the probability (window rows)
    bool valid = false;
    uint4 kc[8];
    uint32_t ksc = 0;
    if (!window) {
        const int j = chunk * AC_KEYS + key;
        if (j < k) {
            const int32_t p = idx[r * k + j];
            if (p >= 0) {
                if (p >= visible_entries(bt, r)) {
                    if (qt == 0) flag(c.status, CSA2_DEV_BAD_INDEX);
                } else {
                    const int64_t slot = entry_slot(c, b, p);
                    if (slot >= 0) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(c.kv_codes + slot * 256) + 4 * qt;
#pragma unroll
                        for (int i = 0; i < 4; i++) kc[i] = __ldg(src + i);
                        ksc = __ldg(reinterpret_cast<const uint32_t *>(c.kv_scales + slot * 16) + qt);
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
            const uint4 *src = reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM) + 8 * qt;
#pragma unroll
            for (int i = 0; i < 8; i++) kc[i] = __ldg(src + i);
            kscale = swa.scales[off];
            valid = true;
        }
    }

    // ---- queries: 64 x 512 bf16, coalesced 16-byte loads into the swizzled B tile
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(q + r * CSA2_HEADS * CSA2_HEAD_DIM);
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = __ldg(src + tid + AC_THREADS * i);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int e = 8 * (tid + AC_THREADS * i);
            *reinterpret_cast<uint4 *>(S.u.q + tc::sw128_offset(e >> 9, e & 511, CSA2_HEADS)) = v[i];
        }
    }
    if (qt == 0) {
        S.kscale[key] = kscale;
        S.valid[key] = valid;
    }
    __syncthreads();                               // the pair table is ready

    // ---- dequantise the key quarter into row `key` of the key tile
    if (valid) {
        if (window) {
            store_window_key(S.k, key, kc, qt);
        } else {
            const uint4 (&kc4)[4] = *reinterpret_cast<const uint4 (*)[4]>(kc);
            store_main_key(S.k, key, kc4, ksc, qt, S.e2m1_pair);
        }
    } else {
        zero_key(S.k, key, qt);
    }

    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;

    // ---- S^T = K Q^T
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k), q0 = tc::smem_u32(S.u.q);
#pragma unroll 1
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
        // ---- logits of this key for this quarter's 16 heads, transposed into smem
        const bool kv = S.valid[key];
        const float lscale = sm_scale * S.kscale[key];
        {
            uint32_t acc[16];
            tmem_ld16(tmem + lane_base + (uint32_t)qt * 16u, acc);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 16; h++)
                S.u.s.red[qt * 16 + h][key] = kv ? __uint_as_float(acc[h]) * lscale : -INFINITY;
        }
        __syncthreads();
        // ---- per-head max and sum over the chunk: eight threads per head
        {
            const int h = tid >> 3, part = tid & 7;
            float mx = -INFINITY;
#pragma unroll 4
            for (int j = part; j < AC_KEYS; j += 8) mx = fmaxf(mx, S.u.s.red[h][j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            float sum = 0.0f;
            if (mx != -INFINITY) {
#pragma unroll 4
                for (int j = part; j < AC_KEYS; j += 8) sum += expf(S.u.s.red[h][j] - mx);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if (part == 0) {
                S.m[h] = mx;
                S.l[h] = sum;
            }
        }
        __syncthreads();
        // ---- P^T (times the window scale) as bf16 hi + lo, K-major rows = heads
        const float vscale = S.kscale[key];
#pragma unroll 4
        for (int hh = 0; hh < 16; hh++) {
            const int h = qt * 16 + hh;
            const float mx = S.m[h];
            const float p = (kv && mx != -INFINITY) ? expf(S.u.s.red[h][key] - mx) * vscale : 0.0f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(p);
            const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
            *reinterpret_cast<__nv_bfloat16 *>(S.u.s.p + tc::sw128_offset(h, key, 2 * CSA2_HEADS)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(S.u.s.p + tc::sw128_offset(CSA2_HEADS + h, key, 2 * CSA2_HEADS)) = lo;
        }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- [O_hi | O_lo]^T = V^T [P_hi | P_lo]^T: 4 tiles of 128 dims, K = 128 keys,
    //      N = 128; the tile of dims 128 mt .. +127 lands in columns 128 mt .. +127
    //      (S has been read out, its columns are reused)
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k);
        const uint32_t p0 = tc::smem_u32(S.u.s.p);
#pragma unroll 1
        for (int mt = 0; mt < 4; mt++) {
            const uint32_t d = tmem + 128u * (uint32_t)mt;
#pragma unroll 1
            for (int kk = 0; kk < 8; kk++) {       // 16 keys per step
                const uint64_t ad = tc::smem_desc(k0 + (uint32_t)(2 * mt) * (AC_KEYS * 128) + (uint32_t)kk * 2048u,
                                                  AC_KEYS * 128, 1024, tc::kSwizzle128B);
                const uint32_t boff = (uint32_t)(kk >> 2) * (2 * CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                tc::mma_f16(d, ad, tc::smem_desc(p0 + boff, 16, 1024, tc::kSwizzle128B), AC_IDESC_O, kk > 0);
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
        // ---- partial output: warp group g takes M-tile g, lane = dim, 64 heads
        const int64_t base = (r * AC_MAX_CHUNKS + chunk) * (int64_t)CSA2_HEADS;
        float *po = part_o + base * CSA2_HEAD_DIM;
        const int mt = warp >> 2;
        const int d = 128 * mt + (warp & 3) * 32 + lane;
#pragma unroll 1
        for (int half = 0; half < 2; half++) {
            uint32_t ahi[32], alo[32];
            const uint32_t col = 128u * (uint32_t)mt + 32u * (uint32_t)half;
            tc::tmem_ld32(tmem + lane_base + col, ahi);
            tc::tmem_ld32(tmem + lane_base + col + 64u, alo);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; h++)
                po[(int64_t)(half * 32 + h) * CSA2_HEAD_DIM + d] = __uint_as_float(ahi[h]) + __uint_as_float(alo[h]);
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
