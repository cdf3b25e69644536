// Scores of the candidate-pool positions, gathered from a Full layer's
// score row (input of the pool Top-512, "DeepSeek-V4.1-Flash 架构详解" §3.2).
#include "csa2_internal.cuh"

namespace csa2 {

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
