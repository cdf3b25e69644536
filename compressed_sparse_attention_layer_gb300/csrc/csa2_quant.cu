// The CSA compressor and the MXFP4 / FP8 quantisers.
//
// These kernels are memory bound (a few bytes read per byte written), so the
// design goal is coalesced 16-byte accesses and enough threads in flight:
//  * compressor: one thread per (entry, channel) in double precision, so the
//    single rounding to fp32 at the end matches a double-precision reference;
//  * MXFP4: one thread per 32-element block (128 B in, 16 B codes + 1 B scale
//    out), 16 consecutive threads covering one 512-dim entry;
//  * FP8: one warp per row (dim 128 or 512), amax by warp shuffle;
//  * the three for a step's new entries in one launch (one CTA per entry).
#include <algorithm>

#include "csa2_internal.cuh"

namespace csa2 {

// e_j[d] = sum_i softmax_i(Z + bias) * C over the m tokens of group j.
// "DeepSeek-V4 report explainer" §3.1; "DeepSeek-V4.1-Flash 架构详解" §2, §3.2.
__device__ __forceinline__ float compress_channel(const uint16_t *__restrict__ C, const uint16_t *__restrict__ Z,
                                                  const float *__restrict__ bias, int m, int64_t j, int d)
{
    const int64_t base = j * m * CSA2_HEAD_DIM + d;
    // one token: its weight is exp(0) / exp(0) = 1 exactly, so the entry is C
    // (the general path below gives the same bits, through FP64 exp)
    if (m == 1) return bf16_to_f32(C[base]);
    double zmax = -INFINITY;
    for (int k = 0; k < m; k++) {
        double z = (double)bf16_to_f32(Z[base + (int64_t)k * CSA2_HEAD_DIM]) + (double)bias[k * CSA2_HEAD_DIM + d];
        zmax = z > zmax ? z : zmax;
    }
    double den = 0.0, num = 0.0;
    for (int k = 0; k < m; k++) {
        double z = (double)bf16_to_f32(Z[base + (int64_t)k * CSA2_HEAD_DIM]) + (double)bias[k * CSA2_HEAD_DIM + d];
        double p = exp(z - zmax);
        den += p;
        num += p * (double)bf16_to_f32(C[base + (int64_t)k * CSA2_HEAD_DIM]);
    }
    return (float)(num / den);
}

__global__ void __launch_bounds__(256) k_compress(const uint16_t *__restrict__ C,
                                                  const uint16_t *__restrict__ Z,
                                                  const float *__restrict__ bias, int m,
                                                  int64_t n_ent, float *__restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = n_ent * CSA2_HEAD_DIM;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = compress_channel(C, Z, bias, m, i / CSA2_HEAD_DIM, (int)(i % CSA2_HEAD_DIM));
}

// floor(log2(a)) of a finite a > 0, subnormals included.
__device__ __forceinline__ int floor_log2(float a)
{
    const uint32_t u = __float_as_uint(a);
    const int e = (int)((u >> 23) & 0xFF);
    if (e) return e - 127;
    return (31 - __clz(u & 0x7FFFFF)) - 149;
}

// E2M1 magnitude code of a >= 0, round to nearest with ties to the even
// mantissa, saturating at 6: thresholds are the midpoints of the grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}; a tie takes the even code (0, 2, 4, 6).
__device__ __forceinline__ uint32_t e2m1_code(float a)
{
    return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
           (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
           (uint32_t)(a > 5.0f);
}

// One 32-element block of an entry: 16 bytes of E2M1 codes and its E8M0
// scale.  "DeepSeek-V4.1-Flash 架构详解" §4 (OCP MXFP4).
__device__ __forceinline__ void quant_mxfp4_block(const float (&v)[32], uint8_t *__restrict__ code16,
                                                  uint8_t *__restrict__ scale1)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(v[i]));
    int X = 0;
    if (amax > 0.0f) {
        X = floor_log2(amax) - 2;
        X = X < -127 ? -127 : (X > 127 ? 127 : X);
    }
    const float inv = exp2i(-X);   // -X in [-125, 127]: a normal float, exact scaling
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const uint32_t c = e2m1_code(fabsf(v[i] * inv)) | ((__float_as_uint(v[i]) >> 31) << 3);
        packed[i >> 3] |= c << (4 * (i & 7));
    }
    *reinterpret_cast<uint4 *>(code16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    *scale1 = (uint8_t)(X + 127);
}

// One thread per 32-element block.
__global__ void __launch_bounds__(256) k_quant_mxfp4(const float *__restrict__ x, int64_t n,
                                                     const int64_t *__restrict__ slots,
                                                     uint8_t *__restrict__ codes,
                                                     uint8_t *__restrict__ scales, int64_t num_slots,
                                                     int32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t >= n * 16) return;
    const int64_t r = t >> 4;
    const int blk = (int)(t & 15);
    const int64_t dst = slots ? slots[r] : r;
    if (dst < 0) return;
    if (dst >= num_slots) {
        flag(status, CSA2_DEV_BAD_SLOT);
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(x + r * CSA2_HEAD_DIM + blk * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float4 f = __ldg(src + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    quant_mxfp4_block(v, codes + dst * 256 + blk * 16, scales + dst * 16 + blk);
}

// FP4 with one E4M3 scale per 16 elements ("DeepSeek-V4.1-Flash 架构详解" §4;
// "How DeepSeek V4.1 Flash beats 1.6T models"): one 16-element block, 8 bytes
// of codes and its scale byte.
__device__ __forceinline__ void quant_fp4e4m3_block(const float (&v)[16], uint8_t *__restrict__ code8,
                                                    uint8_t *__restrict__ scale1)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t sb = f32x2_to_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu;   // amax / 6 >= 0
    const float sv = e4m3_to_f32(sb);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const uint32_t sign = (__float_as_uint(v[i]) >> 31) << 3;
        const uint32_t c = sv == 0.0f ? sign : e2m1_code(fabsf(__fdiv_rn(v[i], sv))) | sign;
        packed[i >> 3] |= c << (4 * (i & 7));
    }
    *reinterpret_cast<uint2 *>(code8) = make_uint2(packed[0], packed[1]);
    *scale1 = (uint8_t)sb;
}

// One thread per 16-element block (64 B in, 8 B codes + 1 B scale out), 32
// threads per entry.
__global__ void __launch_bounds__(256) k_quant_fp4_e4m3(const float *__restrict__ x, int64_t n,
                                                        const int64_t *__restrict__ slots,
                                                        uint8_t *__restrict__ codes,
                                                        uint8_t *__restrict__ scales, int64_t num_slots,
                                                        int32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t >= n * 32) return;
    const int64_t r = t >> 5;
    const int blk = (int)(t & 31);
    const int64_t dst = slots ? slots[r] : r;
    if (dst < 0) return;
    if (dst >= num_slots) {
        if (blk == 0) flag(status, CSA2_DEV_BAD_SLOT);
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(x + r * CSA2_HEAD_DIM + blk * 16);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float4 f = __ldg(src + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    quant_fp4e4m3_block(v, codes + dst * 256 + blk * 8, scales + dst * 32 + blk);
}

// One row of DIM elements by one warp (lane l holds float4 chunks l, l + 32,
// ...): its fp32 scale and e4m3 codes.  "DeepSeek-V4.1-Flash" research note
// §3.3 (FP8 SWA KV).
template <int DIM>
__device__ __forceinline__ void quant_fp8_row(const float4 (&v)[DIM / 128], int lane, uint8_t *__restrict__ codes,
                                              float *__restrict__ scale1)
{
    constexpr int PER = DIM / 128;   // float4 chunks per lane
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < PER; c++)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[c].x), fabsf(v[c].y)), fmaxf(fabsf(v[c].z), fabsf(v[c].w))));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = fp8_row_scale(amax);
    uint32_t *dc = reinterpret_cast<uint32_t *>(codes);
#pragma unroll
    for (int c = 0; c < PER; c++) {
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[c].x, s), __fdiv_rn(v[c].y, s));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[c].z, s), __fdiv_rn(v[c].w, s));
        dc[c * 32 + lane] = lo | (hi << 16);
    }
    if (lane == 0) *scale1 = s;
}

// One warp per row.
template <int DIM>
__global__ void __launch_bounds__(256) k_quant_fp8(const float *__restrict__ x, int64_t n,
                                                   const int64_t *__restrict__ slots,
                                                   uint8_t *__restrict__ codes,
                                                   float *__restrict__ scales, int64_t num_slots,
                                                   int32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();
    constexpr int PER = DIM / 128;
    const int lane = threadIdx.x & 31;
    const int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (r >= n) return;
    const int64_t dst = slots ? slots[r] : r;
    if (dst < 0) return;
    if (dst >= num_slots) {
        if (lane == 0) flag(status, CSA2_DEV_BAD_SLOT);
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(x + r * DIM);
    float4 v[PER];
#pragma unroll
    for (int c = 0; c < PER; c++) v[c] = __ldg(src + c * 32 + lane);
    quant_fp8_row<DIM>(v, lane, codes + dst * DIM, scales + dst);
}

// The step's new entries in one launch: one CTA per entry j.  Thread d
// compresses channel d into shared memory (and the optional fp32 copy); the
// main-KV quantiser threads (16 MXFP4 or 32 FP4-E4M3 blocks) then read their
// blocks from it, and warp 2 quantises the entry's indexer key -- the same
// device functions as k_compress, k_quant_mxfp4 / k_quant_fp4_e4m3 and
// k_quant_fp8<128>, so the results are theirs bit for bit.
constexpr int AP_THREADS = CSA2_HEAD_DIM;
__global__ void __launch_bounds__(AP_THREADS) k_append_entries(
    const uint16_t *__restrict__ C, const uint16_t *__restrict__ Z, const float *__restrict__ bias, int m,
    const float *__restrict__ ik, const int64_t *__restrict__ slots, csa2_cache c, float *__restrict__ entries)
{
    __shared__ __align__(16) float e[CSA2_HEAD_DIM];
    pdl_launch_dependents();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t j = blockIdx.x;
    const float x = compress_channel(C, Z, bias, m, j, tid);
    e[tid] = x;
    if (entries) entries[j * CSA2_HEAD_DIM + tid] = x;
    const int64_t dst = slots ? slots[j] : j;
    const bool ok = dst >= 0 && dst < c.num_slots;
    if (dst >= c.num_slots && tid == 0) flag(c.status, CSA2_DEV_BAD_SLOT);
    if (ok && warp == 2) {                         // the indexer key (independent of the compressor)
        float4 v[1];
        v[0] = __ldg(reinterpret_cast<const float4 *>(ik + j * CSA2_IDX_DIM) + lane);
        quant_fp8_row<CSA2_IDX_DIM>(v, lane, c.ik_codes + dst * CSA2_IDX_DIM, c.ik_scales + dst);
    }
    __syncthreads();
    if (!ok) return;
    if (c.kv_format == CSA2_KV_FP4_E4M3) {
        if (tid < 32) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; i++) v[i] = e[16 * tid + i];
            quant_fp4e4m3_block(v, c.kv_codes + dst * 256 + tid * 8, c.kv_scales + dst * 32 + tid);
        }
    } else if (tid < 16) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = e[32 * tid + i];
        quant_mxfp4_block(v, c.kv_codes + dst * 256 + tid * 16, c.kv_scales + dst * 16 + tid);
    }
}

// ---------------------------------------------------------------- launchers
int launch_compress(const uint16_t *C, const uint16_t *Z, const float *bias, int m, int64_t n_tok,
                    float *out, cudaStream_t st)
{
    const int64_t n_ent = n_tok / m;
    if (n_ent == 0) return CSA2_OK;
    const int64_t total = n_ent * CSA2_HEAD_DIM;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 152 * 16);
    return launch_pdl(k_compress, dim3(grid), dim3(256), 0, st, C, Z, bias, m, n_ent, out);
}

int launch_quant_mxfp4(const float *x, int64_t n, const int64_t *slots, uint8_t *codes,
                       uint8_t *scales, int64_t num_slots, int32_t *status, cudaStream_t st)
{
    if (n == 0) return CSA2_OK;
    const int64_t threads = n * 16;
    return launch_pdl(k_quant_mxfp4, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, x, n, slots, codes,
                      scales, num_slots, status);
}

int launch_quant_fp4_e4m3(const float *x, int64_t n, const int64_t *slots, uint8_t *codes, uint8_t *scales,
                          int64_t num_slots, int32_t *status, cudaStream_t st)
{
    if (n == 0) return CSA2_OK;
    const int64_t threads = n * 32;
    return launch_pdl(k_quant_fp4_e4m3, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, x, n, slots, codes,
                      scales, num_slots, status);
}

int launch_append_entries(const uint16_t *C, const uint16_t *Z, const float *bias, int m, int64_t n_tok,
                          const float *ik, const int64_t *slots, const csa2_cache &c, float *entries, cudaStream_t st)
{
    const int64_t n_ent = n_tok / m;
    if (n_ent == 0) return CSA2_OK;
    return launch_pdl(k_append_entries, dim3((unsigned)n_ent), dim3(AP_THREADS), 0, st, C, Z, bias, m, ik, slots, c,
                      entries);
}

int launch_quant_fp8(const float *x, int64_t n, int dim, const int64_t *slots, uint8_t *codes,
                     float *scales, int64_t num_slots, int32_t *status, cudaStream_t st)
{
    if (n == 0) return CSA2_OK;
    const unsigned grid = (unsigned)((n * 32 + 255) / 256);
    if (dim == 128)
        return launch_pdl(k_quant_fp8<128>, dim3(grid), dim3(256), 0, st, x, n, slots, codes, scales, num_slots,
                          status);
    return launch_pdl(k_quant_fp8<512>, dim3(grid), dim3(256), 0, st, x, n, slots, codes, scales, num_slots, status);
}

}  // namespace csa2
