// Device helpers shared by the lightning-indexer kernels (the Full layer's
// scan and the Reindex layer's pool rescoring): 16-byte cp.async copies and
// the two-part e4m3 query operand of the kind::f8f6f4 products.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

// 16-byte global -> shared copy through the load-store path (L1 bypassed).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

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

// The two-part e4m3 query operand of row r (hi rows at bh, lo rows at bl, 32
// each, 8-row aligned) and w_h * 2^e_h, written by one warp; lane h = head h.  Two passes over the head's 128 dims (the maximum,
// then the conversion) keep half of it in registers at a time.
__device__ __forceinline__ void write_query_operand(uint8_t *bh, uint8_t *bl, float *wq, const uint16_t *qr,
                                                    const float *wr)
{
    const int h = threadIdx.x & 31;
    const uint4 *src = reinterpret_cast<const uint4 *>(qr + h * 128);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const uint4 raw = __ldg(src + i);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] & 0xFFFF0000u)));
        }
    }
    const int e = head_exponent(amax);
    const float f = exp2i(-e);
    wq[h] = wr[h] * exp2i(e);
#pragma unroll 2
    for (int i = 0; i < 16; i += 2) {               // 16 dims per 16-byte chunk of the operand
        uint32_t hiw[4], low[4];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint4 raw = __ldg(src + i + half);
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
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
        *reinterpret_cast<uint4 *>(bh + sw128_b8(h, k)) = make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
        *reinterpret_cast<uint4 *>(bl + sw128_b8(h, k)) = make_uint4(low[0], low[1], low[2], low[3]);
    }
}

// The same operand written by eight warps: thread (h, c) -- lane 8 (h % 4) + c
// of warp h / 4 -- converts dims 16 c .. 16 c + 15 of head h (one 16-byte chunk
// of each part); the head's maximum is reduced over its eight lanes.  Values
// are identical to write_query_operand's.
__device__ __forceinline__ void write_query_chunk(uint8_t *bh, uint8_t *bl, float *wq, const uint16_t *qr,
                                                  const float *wr, int h, int c)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(qr + h * 128 + c * 16);
    const uint4 r0 = __ldg(src), r1 = __ldg(src + 1);
    const uint32_t w8[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w8[j] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w8[j] & 0xFFFF0000u)));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = head_exponent(amax);
    const float f = exp2i(-e);
    if (c == 0) wq[h] = wr[h] * exp2i(e);
    uint32_t hiw[4], low[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const float v[4] = {__uint_as_float(w8[j] << 16) * f, __uint_as_float(w8[j] & 0xFFFF0000u) * f,
                            __uint_as_float(w8[j + 1] << 16) * f, __uint_as_float(w8[j + 1] & 0xFFFF0000u) * f};
        const uint32_t h01 = e4m3x2(v[0], v[1]), h23 = e4m3x2(v[2], v[3]);
        const float q0 = v[0] - e4m3_to_f32(h01 & 0xFF), q1 = v[1] - e4m3_to_f32(h01 >> 8);
        const float q2 = v[2] - e4m3_to_f32(h23 & 0xFF), q3 = v[3] - e4m3_to_f32(h23 >> 8);
        hiw[j / 2] = h01 | (h23 << 16);
        low[j / 2] = e4m3x2(q0, q1) | (e4m3x2(q2, q3) << 16);
    }
    *reinterpret_cast<uint4 *>(bh + sw128_b8(h, 16 * c)) = make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
    *reinterpret_cast<uint4 *>(bl + sw128_b8(h, 16 * c)) = make_uint4(low[0], low[1], low[2], low[3]);
}

}  // namespace csa2
