// Internal helpers shared by the CSA2 kernels (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "csa2.h"

namespace csa2 {

// ---------------------------------------------------------------- host side
// Last CUDA error recorded by an entry point on this thread.
void set_cuda_error(cudaError_t e);

inline int launch_status()
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return CSA2_OK;
}

// Launch `kernel` as a programmatic dependent of the previous kernel on the
// stream: its CTAs may start while that kernel drains and must execute
// pdl_wait() before reading anything it wrote.
template <class K, class... Args>
inline int launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

inline int ceil_div_i(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Per-device kernel set-up (thread-safe): raises `kernel`'s dynamic
// shared-memory limit to `bytes` on the current device -- the limit is a
// property of the kernel on each device -- the first time a launch there
// needs it, and with carveout >= 0 also sets its preferred shared-memory
// carveout (percent).  CSA2_ERR_CUDA if the runtime refuses.
int kernel_smem_limit(const void *kernel, size_t bytes, int carveout = -1);

// Number of SMs of the current device (looked up once per device); 0 if the
// runtime cannot say.
int device_sms();

// Polls a bounded device wait makes before it gives up (kernel argument of
// the tcgen05 kernels): 2^24 unless csa2_debug_set_wait_limit changed it.
uint32_t wait_polls();

// Workspace bytes csa2_layer needs for these arguments (io may be NULL: the
// most any call of the mode needs); 0 for invalid arguments.
size_t layer_workspace_need(int32_t mode, const csa2_batch *b, const csa2_layer_io *io);

inline bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// The pool's own selection input, written by the block-level Top-K as it
// writes the pool (host-side launch argument; all pointers NULL: not wanted).
struct PoolKeys {
    const void *scores = nullptr;  // the scan's score rows the pool indexes (fp32, or bf16 with bf16)
    int64_t ld_scores = 0;         // their row length, a multiple of 8
    bool bf16 = false;
    int k = 0;                     // the pool select's k: the bound holds only over >= k selected blocks
    uint32_t *keys = nullptr;      // [rows][pool slots] order keys of the pool's scores
    uint2 *bound = nullptr;        // [rows][bound_ld]: per cluster CTA, (lower bound, largest key)
    int bound_ld = 0;
};

// ---------------------------------------------------------------- device side
// Programmatic dependent launch: let the next kernel on the stream be
// scheduled now (it still waits for this grid before reading its results) /
// wait until the previous kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bring a line into L2.  Harmless before pdl_wait(): no value is consumed, and
// a later write by the previous kernel still goes through L2.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ void flag(int32_t *status, int32_t bit)
{
    if (status) atomicOr(status, bit);
}

// Slot of logical entry e of sequence b; -1 (and a flag) if the page id is
// outside the cache.
__device__ __forceinline__ int64_t entry_slot(const csa2_cache &c, int b, int64_t e)
{
    int32_t page = __ldg(c.block_table + (int64_t)b * c.max_pages + (e >> 6));
    int64_t slot = (int64_t)page * CSA2_PAGE + (e & 63);
    if (page < 0 || slot >= c.num_slots) {
        flag(c.status, CSA2_DEV_BAD_PAGE);
        return -1;
    }
    return slot;
}

// Entries visible to query row r = b*Q + i ([P3] §3.3 visibility rule).
__device__ __forceinline__ int64_t visible_entries(const csa2_batch &bt, int64_t r)
{
    int b = (int)(r / bt.nq);
    int64_t t = bt.q_pos[r];
    int64_t n = bt.n_entries[b];
    int64_t lim = (t + 1) / bt.m;
    if (lim < n) n = lim;
    if (n > bt.max_entries) n = bt.max_entries;
    if (n < 0) n = 0;
    return n;
}

// ---------------------------------------------------------------- RoPE angles
// The RoPE pair i (dims 448+i, 480+i) turns by t * theta_i, theta_i =
// rope_base^(-i/32), at token position t.  phi[i] holds theta_i / 2π as a
// 64-bit binary fraction (computed on the host in double precision), so that
// t * phi[i] modulo 2^64 is the angle reduced modulo 2π, exact for every
// int64 t up to phi's own rounding (relative 2^-53): no floating-point
// reduction of angles that reach 2^20 rad, and no double-precision work on
// the device.
struct RopeTurns {
    uint64_t phi[32];
};

inline RopeTurns rope_turns(float rope_base)
{
    RopeTurns r;
    for (int i = 0; i < 32; i++) {
        // theta_i <= 1, so theta_i / 2π < 1 and the fraction fits 64 bits
        const double f = rope_base > 0.0f ? pow((double)rope_base, -(double)i / 32.0) / 6.283185307179586 : 0.0;
        r.phi[i] = (uint64_t)ldexp(f, 64);
    }
    return r;
}

// sin and cos of t * theta for one pair: the top 32 bits of the turn fraction,
// read as signed, are the angle in units of 2^-31 π, in [-π, π).
__device__ __forceinline__ void rope_sincos(int64_t t, uint64_t phi, float *s, float *c)
{
    const uint64_t turns = (uint64_t)t * phi;
    const float x = (float)(int32_t)(uint32_t)(turns >> 32) * 4.656612873077393e-10f;   // 2^-31
    sincospif(x, s, c);
}

// FP8 e4m3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte)
{
    uint32_t s = (byte & 0x80u) << 24;
    uint32_t e = (byte >> 3) & 15u;
    uint32_t m = byte & 7u;
    float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
    return __uint_as_float(__float_as_uint(mag) | s);
}

// Two e4m3 bytes (low half of x) -> two halves of a __half2-packed pair via the
// hardware conversion (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
    return r;
}

// Two fp32 values -> two e4m3 bytes (lo in the low byte), round to nearest
// even, saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Per-row FP8 scale from the row's largest magnitude: amax / 448 (fp32 IEEE
// division), 1 for an all-zero row.
__device__ __forceinline__ float fp8_row_scale(float amax) { return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f); }

// E2M1 magnitude code (0..7) -> float magnitude.
__device__ __forceinline__ float e2m1_mag(uint32_t c)
{
    // 0, .5, 1, 1.5, 2, 3, 4, 6
    const uint32_t e = c >> 1, mb = c & 1u;
    return e ? __uint_as_float(((e + 126u) << 23) | (mb << 22)) : 0.5f * (float)mb;
}

__device__ __forceinline__ float e2m1_to_f32(uint32_t nib)
{
    float m = e2m1_mag(nib & 7u);
    return (nib & 8u) ? -m : m;
}

// 2^k for k in [-126, 127] as a float.
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// Monotone map of a float to an unsigned key (larger float -> larger key);
// -0.0 and +0.0 map to the same key.
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = lane < NT / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < NT / 32) warp_sums[lane] = s;   // inclusive
    }
    __syncthreads();
    int base = wid ? warp_sums[wid - 1] : 0;
    if (total) *total = warp_sums[NT / 32 - 1];
    int r = base + x - v;
    __syncthreads();
    return r;
}

}  // namespace csa2
