// Pieces shared by the two schedules of the sparse + window attention
// (csa2_attn_tc.cu: one cluster per (row, key chunk) and a merge kernel;
// csa2_attn_rows.cu: persistent clusters that each take whole rows): the
// split of the work between the CTAs of a cluster, the cluster copy helpers
// and the exact dequantisation of FP4 / FP8 keys into a 128-byte-swizzled
// bf16 key tile.
#pragma once

#include <cuda_bf16.h>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

#ifndef CSA2_ATTN_CLUSTER
#define CSA2_ATTN_CLUSTER 2
#endif
constexpr int AC_KEYS = 128;                       // keys per chunk (MMA M of the first product)
constexpr int AC_CL = CSA2_ATTN_CLUSTER;           // CTAs per cluster, one per slice of the dims
constexpr int AC_DIMS = CSA2_HEAD_DIM / AC_CL;     // dims per CTA
constexpr int AC_SLABS = AC_DIMS / 64;             // 64-dim slabs per CTA = threads per key
constexpr int AC_THREADS = AC_KEYS * AC_SLABS;
constexpr int AC_OWN = CSA2_HEADS / AC_CL;         // heads reduced by each CTA
constexpr int AC_MT = AC_DIMS / 128;               // M-tiles of the value product
constexpr uint32_t AC_TMEM_COLS = AC_MT * 128;     // S^T in columns 0-63, then O^T tile mt at 128 mt
constexpr int AC_MAX_CHUNKS = CSA2_TOPK / AC_KEYS + 1;
constexpr uint32_t AC_IDESC_S = tc::idesc_f16(128, 64, 1, 1, 0, 0);    // K-major A and B
constexpr uint32_t AC_IDESC_O = tc::idesc_f16(128, 128, 1, 1, 1, 0);   // MN-major A (V^T), N = hi|lo
static_assert(AC_CL == 2 || AC_CL == 4, "two or four CTAs per cluster");
static_assert(AC_THREADS / 16 == AC_OWN, "sixteen threads per owned head");
constexpr uint32_t AC_P_ROWS_BYTES = AC_OWN * 128;                       // one CTA's rows of one half, one slab
constexpr uint32_t AC_P_IN_BYTES = (AC_CL - 1) * 4 * AC_P_ROWS_BYTES;   // probability bytes received
constexpr uint32_t AC_S_BYTES = AC_OWN * AC_KEYS * 4;                    // one CTA's partials of one owner
constexpr uint32_t AC_S_IN_BYTES = (AC_CL - 1) * AC_S_BYTES;            // partial-logit bytes received

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Bulk copy of `bytes` from this CTA's shared memory to shared memory of a CTA
// of the cluster (cluster address), completing `bytes` on the mbarrier at the
// cluster address `bar` (in the destination CTA).  Async proxy on both ends.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
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

// Two e4m3 codes (low bytes of the halves of v) -> bf16x2 of their values:
// sign and the 7 exponent/mantissa bits moved into bf16 position give the
// value times 2^-120, which one exact multiply by 2^120 restores (subnormal
// codes included).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t v)
{
    const uint32_t bits = ((v & 0x007F007Fu) << 4) | ((v & 0x00800080u) << 8);
    return bf16x2_mul(bits, 0x7B807B80u);          // 2^120 in both halves
}

// Slab `hf` (local dims 64 hf .. 64 hf + 63) of this CTA's slice of an FP4
// entry -> bf16 row of the key tile (exact): the table gives the two E2M1
// values of a byte with their signs (this lane's copy), one bf16x2 multiply
// applies the block scale.  MXFP4: sc holds the two E8M0 bytes of the slab's
// 32-element blocks (scale 2^X); FP4_E4M3: the four E4M3 bytes of its
// 16-element blocks (every E2M1 x E4M3 product is a bf16 value).
template <bool E4M3>
__device__ __forceinline__ void store_main_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[4], uint32_t sc,
                                               int hf, const uint32_t (*pair)[32], uint32_t lane)
{
#pragma unroll
    for (int blk = 0; blk < 2; blk++) {            // 16 bytes = 32 elements
        const uint32_t w[4] = {c[blk].x, c[blk].y, c[blk].z, c[blk].w};
#pragma unroll
        for (int j = 0; j < 4; j++) {              // 4 bytes = 8 elements -> one 16-byte chunk
            uint32_t f;
            if (E4M3) f = e4m3x2_to_bf16x2(((sc >> (8 * (2 * blk + (j >> 1)))) & 0xFFu) * 0x00010001u);
            else f = pow2_bf16x2((int)((sc >> (8 * blk)) & 0xFFu) - 127);
            uint4 o;
            o.x = bf16x2_mul(pair[w[j] & 0xFFu][lane], f);
            o.y = bf16x2_mul(pair[(w[j] >> 8) & 0xFFu][lane], f);
            o.z = bf16x2_mul(pair[(w[j] >> 16) & 0xFFu][lane], f);
            o.w = bf16x2_mul(pair[w[j] >> 24][lane], f);
            *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 64 * hf + 32 * blk + 8 * j, AC_KEYS)) = o;
        }
    }
}

// The two E2M1 codes of a byte (low nibble first) -> bf16x2 of their values:
// sign to bit 15, the three exponent/mantissa bits to bits 6-8 give the value
// times 2^-126 (0.5 as a bf16 subnormal), which one exact multiply by 2^126
// restores.
__device__ __forceinline__ uint32_t e2m1x2_to_bf16x2(uint32_t byte)
{
    const uint32_t lo = byte & 15u, hi = (byte >> 4) & 15u;
    const uint32_t bits = ((lo & 7u) << 6) | ((lo & 8u) << 12) | ((hi & 7u) << 22) | ((hi & 8u) << 28);
    return bf16x2_mul(bits, 0x7E807E80u);          // 2^126 in both halves
}

// Half `hf` of this CTA's slice of an FP8 window row -> bf16 row of the key
// tile (codes only; exact).
__device__ __forceinline__ void store_window_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[4], int hf)
{
#pragma unroll
    for (int i = 0; i < 4; i++) {                  // 16 codes per load -> two 16-byte chunks
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
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 64 * hf + 16 * i, AC_KEYS)) = o0;
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 64 * hf + 16 * i + 8, AC_KEYS)) = o1;
    }
}

__device__ __forceinline__ void zero_key(uint8_t *ktile, uint32_t row, int hf)
{
#pragma unroll
    for (int i = 0; i < 8; i++)
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 64 * hf + 8 * i, AC_KEYS)) = make_uint4(0, 0, 0, 0);
}

}  // namespace csa2
