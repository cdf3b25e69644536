// a4/a7: lightning-indexer scores on CUDA cores.
//
// score(p) = scale_p * sum_h w_h * ReLU(qi_h . code_p)   (scale_p > 0, so the
// scale factors out of the ReLU), qi in fp32 shared memory, the 128 e4m3
// codes of one entry per thread.  Used for the candidate-pool rescoring of a
// Reindex layer (16,384 gathered entries per query) and for rows too short to
// fill a tensor-core tile.  "DeepSeek-V4 report explainer" §3.2;
// "DeepSeek-V4.1-Flash 架构详解" §3.2.
#include "csa2_internal.cuh"

namespace csa2 {

constexpr int IX_THREADS = 128;

// Dot products of one entry's 128 codes with the 32 indexer heads.
__device__ __forceinline__ float entry_score(const uint8_t *__restrict__ codes, float scale,
                                             const float4 (*qs)[32], const float *ws)
{
    float acc[32];
#pragma unroll
    for (int h = 0; h < 32; h++) acc[h] = 0.0f;
    const uint4 *src = reinterpret_cast<const uint4 *>(codes);
#pragma unroll 1
    for (int ch = 0; ch < 8; ch++) {
        const uint4 u = __ldg(src + ch);
        float kv[16];
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 16; i++) kv[i] = e4m3_to_f32((wd[i >> 2] >> (8 * (i & 3))) & 0xFFu);
#pragma unroll
        for (int h = 0; h < 32; h++) {
            float a = acc[h];
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                const float4 q = qs[h][ch * 4 + c4];
                a = fmaf(q.x, kv[4 * c4], a);
                a = fmaf(q.y, kv[4 * c4 + 1], a);
                a = fmaf(q.z, kv[4 * c4 + 2], a);
                a = fmaf(q.w, kv[4 * c4 + 3], a);
            }
            acc[h] = a;
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int h = 0; h < 32; h++) s = fmaf(ws[h], fmaxf(acc[h], 0.0f), s);
    return s * scale;
}

template <bool POOL>
__global__ void __launch_bounds__(IX_THREADS) k_index_simt(
    csa2_cache c, csa2_batch bt, const uint16_t *__restrict__ qi, const float *__restrict__ w,
    const int32_t *__restrict__ pool, const int32_t *__restrict__ pool_len,
    float *__restrict__ scores, float *__restrict__ block_max, int32_t *__restrict__ n_visible,
    int64_t ld)
{
    __shared__ float4 qs[32][32];
    __shared__ float ws[32];
    const int64_t r = blockIdx.y;
    const int b = (int)(r / bt.nq);
    const int tid = threadIdx.x;
    const int64_t nvis = visible_entries(bt, r);
    int64_t n = nvis;
    if (POOL) {
        n = pool_len[r];
        n = n < 0 ? 0 : (n > ld ? ld : n);
    }
    const int64_t i0 = (int64_t)blockIdx.x * IX_THREADS;
    if (!POOL && blockIdx.x == 0 && tid == 0 && n_visible) n_visible[r] = (int32_t)nvis;
    if (i0 >= n) return;
    {
        const uint16_t *qr = qi + r * 4096;
        float *qf = reinterpret_cast<float *>(qs);
        for (int e = tid; e < 4096; e += IX_THREADS) qf[e] = bf16_to_f32(qr[e]);
        if (tid < 32) ws[tid] = w[r * 32 + tid];
    }
    __syncthreads();
    const int64_t i = i0 + tid;
    float sc = -INFINITY;
    if (i < n) {
        const int64_t p = POOL ? (int64_t)pool[r * ld + i] : i;
        if (p < 0 || p >= nvis) {
            flag(c.status, CSA2_DEV_BAD_INDEX);
        } else {
            const int64_t slot = entry_slot(c, b, p);
            if (slot >= 0) sc = entry_score(c.ik_codes + slot * 128, c.ik_scales[slot], qs, ws);
        }
        if (scores) scores[r * ld + i] = sc;
    }
    if (!POOL && block_max) {
        float m = sc;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((tid & 7) == 0 && i < n) block_max[r * (ld / 8) + (i >> 3)] = m;
    }
}

int launch_index_pool_simt(const csa2_cache &c, const csa2_batch &bt, const uint16_t *qi,
                           const float *w, const int32_t *pool, const int32_t *pool_len, int64_t ld,
                           float *scores, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    dim3 grid((unsigned)ceil_div_i(ld, IX_THREADS), (unsigned)rows);
    k_index_simt<true><<<grid, IX_THREADS, 0, st>>>(c, bt, qi, w, pool, pool_len, scores, nullptr,
                                                    nullptr, ld);
    return launch_status();
}

// scores of the pool positions, gathered from a full score row
__global__ void k_gather_scores(const float *__restrict__ scores, int64_t ld,
                                const int32_t *__restrict__ pool, const int32_t *__restrict__ pool_len,
                                int64_t ld_pool, float *__restrict__ out)
{
    const int64_t r = blockIdx.y;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t n = pool_len[r];
    n = n < 0 ? 0 : (n > ld_pool ? ld_pool : n);
    if (i >= n) return;
    const int32_t p = pool[r * ld_pool + i];
    out[r * ld_pool + i] = (p >= 0 && p < ld) ? scores[r * ld + p] : -INFINITY;
}

int launch_gather_scores(const float *scores, int64_t ld, const int32_t *pool, const int32_t *pool_len,
                         int64_t ld_pool, int64_t rows, float *out, cudaStream_t st)
{
    dim3 grid((unsigned)ceil_div_i(ld_pool, 256), (unsigned)rows);
    k_gather_scores<<<grid, 256, 0, st>>>(scores, ld, pool, pool_len, ld_pool, out);
    return launch_status();
}

}  // namespace csa2
