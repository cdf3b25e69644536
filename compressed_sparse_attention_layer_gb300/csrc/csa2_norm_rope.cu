// The attention inputs' prologue: RMSNorm of every 512-dim query head / KV
// entry, then the partial RoPE on its last 64 dims.
// "DeepSeek-V4 report explainer" §4.3 (queries and compressed KV normalised
// before the core attention; RoPE on the last 64 dims only, the output
// rotated back afterwards).
//
// Memory bound (2 KB read, 2 KB or 1 KB written per vector): one warp per
// vector, each lane four float4 loads (dims 4·lane + 128·c), the mean square
// by warp shuffle.  The RoPE pair (448+i, 480+i) sits in lanes 16+i/4 and
// 24+i/4 of the last chunk, so one shuffle across 8 lanes brings each lane its
// partner.  Angles: t·θ_i reduced modulo 2π exactly in 64-bit integer turns
// (rope_sincos), then sin / cos in fp32.
#include <cuda_bf16.h>

#include "csa2_internal.cuh"

namespace csa2 {

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// One warp per vector.  x may equal out_f32: each lane reads its 16 values
// before it writes them.
__global__ void __launch_bounds__(256) k_norm_rope(const float *x, int64_t nvec, int vecs,
                                                   const float *__restrict__ gamma, float eps,
                                                   const int64_t *__restrict__ pos, int rope, RopeTurns turns,
                                                   float *out_f32, uint16_t *out_bf16)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t v = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (v >= nvec) return;
    const float4 *src = reinterpret_cast<const float4 *>(x + v * CSA2_HEAD_DIM);
    float4 a[4];
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        a[c] = src[c * 32 + lane];
        ss = fmaf(a[c].x, a[c].x, ss);
        ss = fmaf(a[c].y, a[c].y, ss);
        ss = fmaf(a[c].z, a[c].z, ss);
        ss = fmaf(a[c].w, a[c].w, ss);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    // 1 / sqrt(mean square + eps), IEEE square root and division
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)CSA2_HEAD_DIM) + eps));
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const float4 g = gamma ? __ldg(reinterpret_cast<const float4 *>(gamma) + c * 32 + lane)
                               : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
        a[c].x = a[c].x * inv * g.x;
        a[c].y = a[c].y * inv * g.y;
        a[c].z = a[c].z * inv * g.z;
        a[c].w = a[c].w * inv * g.w;
    }
    if (rope) {
        // chunk 3 holds dims 384 + 4·lane .. +3: lanes 16..23 the first halves
        // (448 + i), lanes 24..31 the second (480 + i), i = 4·(lane & 7) + j
        float4 p;
        p.x = __shfl_xor_sync(0xffffffffu, a[3].x, 8);
        p.y = __shfl_xor_sync(0xffffffffu, a[3].y, 8);
        p.z = __shfl_xor_sync(0xffffffffu, a[3].z, 8);
        p.w = __shfl_xor_sync(0xffffffffu, a[3].w, 8);
        if (lane >= 16) {
            const int64_t t = pos[v / vecs];
            const bool first = lane < 24;
            float *own = &a[3].x;
            const float *par = &p.x;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float s, co;
                rope_sincos(t, turns.phi[4 * (lane & 7) + j], &s, &co);
                // (u, w) -> (u cos - w sin, u sin + w cos), u the first half
                own[j] = first ? own[j] * co - par[j] * s : par[j] * s + own[j] * co;
            }
        }
    }
    if (out_f32) {
        float4 *dst = reinterpret_cast<float4 *>(out_f32 + v * CSA2_HEAD_DIM);
#pragma unroll
        for (int c = 0; c < 4; c++) dst[c * 32 + lane] = a[c];
    } else {
        uint2 *dst = reinterpret_cast<uint2 *>(out_bf16 + v * CSA2_HEAD_DIM);
#pragma unroll
        for (int c = 0; c < 4; c++) dst[c * 32 + lane] = make_uint2(pack_bf16x2(a[c].x, a[c].y), pack_bf16x2(a[c].z, a[c].w));
    }
}

int launch_norm_rope(const float *x, int64_t rows, int vecs, const float *gamma, float eps, const int64_t *pos,
                     float rope_base, float *out_f32, uint16_t *out_bf16, cudaStream_t st)
{
    const int64_t nvec = rows * vecs;
    if (nvec == 0) return CSA2_OK;
    const RopeTurns turns = rope_turns(rope_base);
    const unsigned grid = (unsigned)((nvec + 7) / 8);
    return launch_pdl(k_norm_rope, dim3(grid), dim3(256), 0, st, x, nvec, vecs, gamma, eps, pos,
                      rope_base > 0.0f ? 1 : 0, turns, out_f32, out_bf16);
}

}  // namespace csa2
