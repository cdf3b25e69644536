// a9: sparse MQA + sliding-window attention on CUDA cores.
//
// Grid: one CTA per (query row, group of 4 heads).  The CTA lists its keys
// (selected MXFP4 entries, then the window rows), computes the logits of its
// 4 heads (one warp per key, 16 dims per lane, the key dequantised in
// registers), takes one softmax over all keys per head and accumulates
// o = P K with each thread owning 2 of the 512 dims.  Every key serves as
// its own value ("DeepSeek-V4 report explainer" §4.3), one softmax covers the
// compressed and window branches ("DeepSeek-V4.1-Flash 架构详解" §1 table, §3;
// explainer §3.3).  Dequantisation: MXFP4 e2m1 * 2^X is exact in fp32; the
// window value is e4m3 * s rounded once to fp32.
#include "csa2_internal.cuh"

namespace csa2 {

constexpr int AT_THREADS = 256;
constexpr int AT_HG = 4;                 // heads per CTA
constexpr int AT_MAXK = CSA2_TOPK + CSA2_SWA_WINDOW;

__global__ void __launch_bounds__(AT_THREADS) k_attn_simt(csa2_cache c, csa2_batch bt,
                                                          const uint16_t *__restrict__ q,
                                                          float sm_scale,
                                                          const int32_t *__restrict__ idx, int k,
                                                          csa2_swa swa, float *__restrict__ o,
                                                          float *__restrict__ lse)
{
    __shared__ int64_t key_slot[AT_MAXK];   // >= 0: main-KV slot; < 0: -(window row) - 1
    __shared__ float qs[AT_HG][CSA2_HEAD_DIM];
    __shared__ float lg[AT_HG][AT_MAXK];
    __shared__ float red_max[AT_HG], red_inv[AT_HG];
    __shared__ int warp_sums[32];
    __shared__ int n_main_sh;

    const int64_t r = blockIdx.x;
    const int h0 = blockIdx.y * AT_HG;
    const int b = (int)(r / bt.nq);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t t = bt.q_pos[r];
    const int64_t nvis = visible_entries(bt, r);

    // ---- key list: selected entries in idx order (ordered compaction), then window rows
    int64_t my_slot = -1;
    if (tid < k) {
        const int32_t p = idx[r * k + tid];
        if (p >= 0) {
            if (p >= nvis) flag(c.status, CSA2_DEV_BAD_INDEX);
            else my_slot = entry_slot(c, b, p);
        }
    }
    int valid = my_slot >= 0;
    int total = 0;
    int off = 0;
    {
        // k <= 512 = 2 * AT_THREADS: two rounds of 256
        int v0 = valid;
        off = block_exclusive_scan<AT_THREADS>(v0, warp_sums, &total);
        if (v0) key_slot[off] = my_slot;
        int64_t s2 = -1;
        if (tid + AT_THREADS < k) {
            const int32_t p = idx[r * k + tid + AT_THREADS];
            if (p >= 0) {
                if (p >= nvis) flag(c.status, CSA2_DEV_BAD_INDEX);
                else s2 = entry_slot(c, b, p);
            }
        }
        int v1 = s2 >= 0;
        int total1 = 0;
        int off1 = block_exclusive_scan<AT_THREADS>(v1, warp_sums, &total1);
        if (v1) key_slot[total + off1] = s2;
        total += total1;
    }
    const int n_main = total;
    const int64_t s0 = swa.start ? swa.start[b] : 0;
    int64_t lo = t - (CSA2_SWA_WINDOW - 1);
    if (lo < s0) lo = s0;
    if (lo < 0) lo = 0;
    const int n_win = t >= lo ? (int)(t - lo + 1) : 0;
    if (tid < n_win) key_slot[n_main + tid] = -((lo + tid) % swa.rows) - 1;
    if (tid == 0) n_main_sh = n_main;
    for (int e = tid; e < AT_HG * CSA2_HEAD_DIM; e += AT_THREADS)
        qs[e / CSA2_HEAD_DIM][e % CSA2_HEAD_DIM] =
            bf16_to_f32(q[(r * CSA2_HEADS + h0) * CSA2_HEAD_DIM + e]);
    __syncthreads();
    const int nk = n_main + n_win;

    const uint8_t *swa_codes = swa.codes + (int64_t)b * swa.rows * CSA2_HEAD_DIM;
    const float *swa_scales = swa.scales + (int64_t)b * swa.rows;

    // ---- logits: one warp per key, lane owns dims [16 lane, 16 lane + 16)
    for (int j = wid; j < nk; j += AT_THREADS / 32) {
        const int64_t ks = key_slot[j];
        float kv[16];
        if (ks >= 0) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(c.kv_codes + ks * 256) + lane);
            const float sc = exp2i((int)c.kv_scales[ks * 16 + (lane >> 1)] - 127);
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const uint32_t word = i < 8 ? u.x : u.y;
                kv[i] = e2m1_to_f32((word >> (4 * (i & 7))) & 15u) * sc;
            }
        } else {
            const int64_t row = -ks - 1;
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(swa_codes + row * CSA2_HEAD_DIM) + lane);
            const float sc = swa_scales[row];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 16; i++) kv[i] = e4m3_to_f32((wd[i >> 2] >> (8 * (i & 3))) & 0xFFu) * sc;
        }
#pragma unroll
        for (int h = 0; h < AT_HG; h++) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i++) a = fmaf(qs[h][16 * lane + i], kv[i], a);
#pragma unroll
            for (int o2 = 16; o2; o2 >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o2);
            if (lane == 0) lg[h][j] = a * sm_scale;
        }
    }
    __syncthreads();

    // ---- softmax statistics: warp h handles head h
    if (wid < AT_HG) {
        float mx = -INFINITY;
        for (int j = lane; j < nk; j += 32) mx = fmaxf(mx, lg[wid][j]);
#pragma unroll
        for (int o2 = 16; o2; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        float sum = 0.0f;
        for (int j = lane; j < nk; j += 32) {
            const float p = expf(lg[wid][j] - mx);
            lg[wid][j] = p;
            sum += p;
        }
#pragma unroll
        for (int o2 = 16; o2; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        if (lane == 0) {
            red_max[wid] = mx;
            red_inv[wid] = nk ? 1.0f / sum : 0.0f;
            lse[r * CSA2_HEADS + h0 + wid] = nk ? mx + logf(sum) : -INFINITY;
        }
    }
    __syncthreads();

    // ---- o = P K: thread owns dims d0 = 2 tid, d0 + 1
    const int d0 = 2 * tid;
    float acc[AT_HG][2];
#pragma unroll
    for (int h = 0; h < AT_HG; h++) acc[h][0] = acc[h][1] = 0.0f;
    for (int j = 0; j < nk; j++) {
        const int64_t ks = key_slot[j];
        float v0, v1;
        if (ks >= 0) {
            const uint32_t byte = c.kv_codes[ks * 256 + tid];
            const float sc = exp2i((int)c.kv_scales[ks * 16 + (d0 >> 5)] - 127);
            v0 = e2m1_to_f32(byte & 15u) * sc;
            v1 = e2m1_to_f32(byte >> 4) * sc;
        } else {
            const int64_t row = -ks - 1;
            const uint16_t two = *reinterpret_cast<const uint16_t *>(swa_codes + row * CSA2_HEAD_DIM + d0);
            const float sc = swa_scales[row];
            v0 = e4m3_to_f32(two & 0xFFu) * sc;
            v1 = e4m3_to_f32(two >> 8) * sc;
        }
#pragma unroll
        for (int h = 0; h < AT_HG; h++) {
            const float p = lg[h][j];
            acc[h][0] = fmaf(p, v0, acc[h][0]);
            acc[h][1] = fmaf(p, v1, acc[h][1]);
        }
    }
#pragma unroll
    for (int h = 0; h < AT_HG; h++) {
        float2 res = make_float2(acc[h][0] * red_inv[h], acc[h][1] * red_inv[h]);
        *reinterpret_cast<float2 *>(o + ((r * CSA2_HEADS + h0 + h) * CSA2_HEAD_DIM) + d0) = res;
    }
    (void)n_main_sh;
}

int launch_attn_simt(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale,
                     const int32_t *idx, int k, const csa2_swa &swa, float *o, float *lse, cudaStream_t st)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    dim3 grid((unsigned)rows, CSA2_HEADS / AT_HG);
    k_attn_simt<<<grid, AT_THREADS, 0, st>>>(c, bt, q, sm_scale, idx, k, swa, o, lse);
    return launch_status();
}

}  // namespace csa2

namespace csa2 {
size_t attn_workspace_bytes(int64_t) { return 0; }

int launch_attn(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale,
                const int32_t *idx, int k, const csa2_swa &swa, float *o, float *lse, void *, size_t,
                cudaStream_t st)
{
    return launch_attn_simt(c, bt, q, sm_scale, idx, k, swa, o, lse, st);
}
}  // namespace csa2
