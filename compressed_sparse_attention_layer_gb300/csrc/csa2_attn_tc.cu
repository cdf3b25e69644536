// Sparse MQA + sliding-window attention on the tcgen05 tensor cores.
//
// Every key is its own value ("DeepSeek-V4 report explainer" §4.3) and one
// softmax covers the selected entries and the window ("DeepSeek-V4.1-Flash
// 架构详解" §1 table, §3; explainer §3.3).
//
// Work unit (row, chunk, half of the dims): 128 keys -- chunks 0..3 the
// selected entries idx[128c .. 128c+127], the last chunk the window rows --
// all 64 heads, and the output dims 256 d .. 256 d + 255.  One CTA per unit,
// 512 threads:
//   1. dequantise the chunk's keys into a 128 x 512 bf16 tile (four threads
//      per key, 128 dims each): MXFP4 bytes through a 256-entry table (byte ->
//      two bf16 magnitudes with signs) and one bf16x2 multiply by the block
//      scale; window codes e4m3 by placing their bits in a bf16 and one
//      multiply by 2^120 -- both exact; the window's fp32 row scale is applied
//      to the logit and to the probability instead;
//   2. S^T[128 keys x 64 heads] = K Q^T over all 512 dims (M = keys, N =
//      heads, 32 MMAs of K = 16).  The two CTAs of a chunk both compute these
//      logits: an MMA costs about the same from N = 16 to N = 64, so the
//      redundant product is cheaper than exchanging partial sums over halves
//      of the dims;
//   3. per head: the chunk's max m_c and sum l_c, and P = exp(S - m_c) as
//      bf16 hi + lo (P = hi + lo to 2^-17), written as the B operand of
//   4. [O_hi | O_lo]^T = V_d^T [P_hi | P_lo]^T for the CTA's 256 dims: the key
//      tile read as an MN-major operand (V = K), two M-tiles of 128 dims, K =
//      128 keys, N = 128 (16 MMAs); the epilogue adds the two halves and
//      writes the unnormalised partial O_c and (m_c, l_c) to the workspace;
//   5. the chunks of one (row, half) form a thread-block cluster: after a
//      cluster barrier each CTA merges a share of the half's outputs in one
//      round of loads, O = sum_c e^(m_c - M) O_c / (sum_c e^(m_c - M) l_c +
//      e^(z_h - M)), with the optional sink logit z_h, and rotates the
//      output's RoPE dims back.
// A decode row's window chunk also quantises the query token's own window
// row (csa2_swa.new_rows) exactly as the FP8 quantiser would, into its key
// tile and into the ring.
//
// Key tiles carried between layers (csa2_layer_io.kv_tiles): a Reuse layer
// attends to the same selected entries as the layer that selected them, so
// that layer also writes each selected chunk's dequantised tile -- the exact
// shared-memory image, 128 KB, and its key scales -- to global memory with
// bulk stores, and the Reuse layers that follow bulk-copy it back (one TMA
// stream per CTA) instead of gathering and dequantising the entries again.
// That matters most for the CTAs that start late, once the previous layer's
// CTAs have left their SMs.
#include <cuda_bf16.h>

#include <algorithm>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {

constexpr int AC_KEYS = 128;                       // keys per chunk (MMA M of the logit product)
constexpr int AC_HALVES = 2;                       // halves of the output dims per chunk
constexpr int AC_DH = CSA2_HEAD_DIM / AC_HALVES;   // output dims per CTA
constexpr int AC_THREADS = 512;                    // four threads per key (128 dims each) for the loads
constexpr int AC_SLABS = CSA2_HEAD_DIM / 64;       // 64-dim slabs of the key tile
constexpr int AC_MT = AC_DH / 128;                 // M-tiles of the value product
constexpr int AC_MAX_CHUNKS = CSA2_TOPK / AC_KEYS + 1;
constexpr uint32_t AC_TILE_BYTES = AC_SLABS * AC_KEYS * 128;        // one chunk's key tile
constexpr uint32_t AC_TILE_STRIDE = AC_TILE_BYTES + 1024;             // + its key scales, per chunk
constexpr uint32_t AC_TMEM_COLS = 512;             // O^T tile mt at 128 mt (hi 64 | lo 64), S^T at 256
constexpr uint32_t AC_S_COL = 256;
constexpr uint32_t AC_IDESC_S = tc::idesc_f16(128, CSA2_HEADS, 1, 1, 0, 0);       // K-major A and B
constexpr uint32_t AC_IDESC_O = tc::idesc_f16(128, 2 * CSA2_HEADS, 1, 1, 1, 0);   // MN-major A (V^T), N = hi|lo
static_assert(AC_THREADS == 4 * AC_KEYS, "four threads per key");
static_assert(AC_THREADS / 8 == CSA2_HEADS, "eight threads per head in the softmax");
static_assert(AC_THREADS / 32 == 4 * AC_MT * 2, "one warp per (M-tile, lane quarter, 32 heads) in the epilogue");

struct AcSmem {
    uint8_t k[AC_SLABS * AC_KEYS * 128];           // [slab of 64 dims][128 keys][128 B]   128 KB
    union {
        uint8_t q[AC_SLABS * CSA2_HEADS * 128];    // [slab][64 heads][128 B]              64 KB
        struct {                                   // once the logit product is done with Q:
            float s[CSA2_HEADS][AC_KEYS];          //   logits [head][key]                 32 KB
            uint8_t p[2 * 2 * CSA2_HEADS * 128];   //   [slab of 64 keys][hi 64 | lo 64 rows][128 B]
        } sp;
    } u;
    uint32_t e2m1_pair[256][32];                   // byte -> bf16x2 of its two E2M1 codes, one
                                                   // copy per lane (bank = lane: no conflicts)  32 KB
    float kscale[AC_KEYS];                         // window row scale (1 for entries), -1: no key
    uint64_t mbar;                                 // the products' commits
    uint64_t tbar;                                 // a carried key tile has landed
    uint32_t tmem;
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
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

// Quarter qq (dims 128 qq .. 128 qq + 127) of an FP4 entry -> bf16 row of the
// key tile (exact): the table gives the two E2M1 values of a byte with their
// signs (this lane's copy), one bf16x2 multiply applies the block scale.
// MXFP4: sc.x holds the four E8M0 bytes of the quarter's 32-element blocks
// (scale 2^X); FP4_E4M3: sc.x, sc.y the eight E4M3 bytes of its 16-element
// blocks (every E2M1 x E4M3 product is a bf16 value).
template <bool E4M3>
__device__ __forceinline__ void store_main_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[8], uint2 sc, int qq,
                                               const uint32_t (*pair)[32], uint32_t lane)
{
#pragma unroll
    for (int blk = 0; blk < 4; blk++) {            // 16 bytes = 32 elements
        const uint32_t w[4] = {c[blk].x, c[blk].y, c[blk].z, c[blk].w};
#pragma unroll
        for (int j = 0; j < 4; j++) {              // 4 bytes = 8 elements -> one 16-byte chunk
            uint32_t f;
            if (E4M3) {
                const int sb = 2 * blk + (j >> 1);                       // 16-element block of the quarter
                const uint32_t word = sb < 4 ? sc.x : sc.y;
                f = e4m3x2_to_bf16x2(((word >> (8 * (sb & 3))) & 0xFFu) * 0x00010001u);
            } else {
                f = pow2_bf16x2((int)((sc.x >> (8 * blk)) & 0xFFu) - 127);
            }
            uint4 o;
            o.x = bf16x2_mul(pair[w[j] & 0xFFu][lane], f);
            o.y = bf16x2_mul(pair[(w[j] >> 8) & 0xFFu][lane], f);
            o.z = bf16x2_mul(pair[(w[j] >> 16) & 0xFFu][lane], f);
            o.w = bf16x2_mul(pair[w[j] >> 24][lane], f);
            *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 32 * blk + 8 * j, AC_KEYS)) = o;
        }
    }
}

// Quarter qq of an FP8 window row -> bf16 row of the key tile (codes only; exact).
__device__ __forceinline__ void store_window_key(uint8_t *ktile, uint32_t row, const uint4 (&c)[8], int qq)
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
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 16 * i, AC_KEYS)) = o0;
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 16 * i + 8, AC_KEYS)) = o1;
    }
}

// Ring row `row` (its 128 codes of quarter qq, staged unswizzled at `stage`,
// 512 B per row) -> bf16 row of the key tile (exact).  Lane-rotated 16-byte
// chunks: the eight lanes of a shared-memory phase read eight different
// chunk columns of eight rows (no bank conflicts).
__device__ __forceinline__ void stage_window_key(uint8_t *ktile, const uint8_t *stage, uint32_t row, int qq,
                                                 uint32_t lane)
{
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t cc = ((uint32_t)i + lane) & 7u;                 // 16-code chunk of the quarter
        const uint4 c = *reinterpret_cast<const uint4 *>(stage + row * CSA2_HEAD_DIM + 128 * qq + 16 * cc);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint4 o0, o1;
        o0.x = e4m3x2_to_bf16x2(__byte_perm(w[0], 0, 0x4140));
        o0.y = e4m3x2_to_bf16x2(__byte_perm(w[0], 0, 0x4342));
        o0.z = e4m3x2_to_bf16x2(__byte_perm(w[1], 0, 0x4140));
        o0.w = e4m3x2_to_bf16x2(__byte_perm(w[1], 0, 0x4342));
        o1.x = e4m3x2_to_bf16x2(__byte_perm(w[2], 0, 0x4140));
        o1.y = e4m3x2_to_bf16x2(__byte_perm(w[2], 0, 0x4342));
        o1.z = e4m3x2_to_bf16x2(__byte_perm(w[3], 0, 0x4140));
        o1.w = e4m3x2_to_bf16x2(__byte_perm(w[3], 0, 0x4342));
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 16 * cc, AC_KEYS)) = o0;
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 16 * cc + 8, AC_KEYS)) = o1;
    }
}

__device__ __forceinline__ void zero_key(uint8_t *ktile, uint32_t row, int qq)
{
#pragma unroll
    for (int i = 0; i < 16; i++)
        *reinterpret_cast<uint4 *>(ktile + tc::sw128_offset(row, 128 * qq + 8 * i, AC_KEYS)) = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------- the kernel
// Grid: x = AC_HALVES * nchunks (one cluster per half d of the output dims
// holding its nchunks chunks: x = d * nchunks + chunk), y = query rows.
// Launched as a programmatic dependent of the previous kernel on the stream.
// `polls` bounds each wait for a product or a tile (CSA2_DEV_TIMEOUT when it
// runs out).  tile_mode: 0 no carried tiles, 1 write them, 2 read them after
// the dependency wait, 3 read them before it (written before the previous
// kernel's predecessor).
__global__ void __launch_bounds__(AC_THREADS, 1)
    k_attn_tc(csa2_cache c, csa2_batch bt, const uint16_t *__restrict__ q, float sm_scale,
              const int32_t *__restrict__ idx, int k, csa2_swa swa, int rope, RopeTurns turns,
              float *__restrict__ part_o, float *__restrict__ part_ml, float *__restrict__ o,
              float *__restrict__ lse, int nchunks, int early, uint8_t *__restrict__ tiles, int tile_mode,
              uint32_t polls)
{
    extern __shared__ uint8_t smem_raw[];
    AcSmem &S = *reinterpret_cast<AcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int key = tid & (AC_KEYS - 1), qq = tid >> 7;          // key row; quarter of the dims
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16; // TMEM lane quarter of this warp
    const int chunk = (int)blockIdx.x % nchunks;
    const int d = (int)blockIdx.x / nchunks;                     // output dims AC_DH d .. AC_DH d + AC_DH - 1
    const int64_t r = blockIdx.y;
    const int b = (int)(r / bt.nq);
    const bool window = chunk == nchunks - 1;
    const int64_t base = (r * AC_MAX_CHUNKS + chunk) * (int64_t)CSA2_HEADS;   // (row, chunk, head 0)
    const uint16_t *qr = q + r * CSA2_HEADS * CSA2_HEAD_DIM;
    // this chunk's carried tile (selected chunks only)
    uint8_t *tile_g = tiles && !window ? tiles + (r * (AC_MAX_CHUNKS - 1) + chunk) * (int64_t)AC_TILE_STRIDE : nullptr;
    const bool tread = tile_g && tile_mode >= 2, twrite = tile_g && tile_mode == 1;

    if (tid == 0) {
        tc::mbar_init(&S.mbar, 1);
        tc::mbar_init(&S.tbar, 1);
        tc::fence_mbar_init();
    }
    // the carried tile and its key scales, one bulk stream into the key tile
    auto load_tile = [&]() {
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(&S.tbar, AC_TILE_BYTES + AC_KEYS * 4);
#pragma unroll
            for (int sl = 0; sl < AC_SLABS; sl++)
                tc::bulk_load(S.k + sl * (AC_KEYS * 128), tile_g + sl * (AC_KEYS * 128), AC_KEYS * 128, &S.tbar);
            tc::bulk_load(S.kscale, tile_g + AC_TILE_BYTES, AC_KEYS * 4, &S.tbar);
        }
    };
    if (tread && tile_mode == 3) load_tile();
    if (warp == 0) tc::tmem_alloc(&S.tmem, AC_TMEM_COLS);
    // the row's queries (and a decode token's new window row) into L2 while the
    // previous kernel finishes: a prefetch carries no data into this CTA, so it
    // may run before the dependency wait
    prefetch_l2(reinterpret_cast<const uint8_t *>(qr) + 128 * tid);
    if (window && swa.new_rows && tid < CSA2_HEAD_DIM * 4 / 128)
        prefetch_l2(reinterpret_cast<const uint8_t *>(swa.new_rows + r * CSA2_HEAD_DIM) + 128 * tid);
    // E2M1 pair table (FP4 entries are dequantised here): 2048 16-byte chunks of
    // four copies each, consecutive per lane
    if (!window && !tread) {
#pragma unroll
        for (int ch = tid; ch < 256 * 32 / 4; ch += AC_THREADS) {
            const uint32_t v = e2m1x2_to_bf16x2((uint32_t)ch >> 3);
            reinterpret_cast<uint4 *>(&S.e2m1_pair[0][0])[ch] = make_uint4(v, v, v, v);
        }
    }
    // ---- this thread's key: locate it and load its 128 dims
    float kscale = 1.0f;          // multiplies the logit and the probability (window rows)
    bool valid = false;
    uint4 kc[8];
    uint2 ksc = make_uint2(0u, 0u);
    int64_t t = 0, lo = 0;
    int kn = -1;                  // the query's own token in the window chunk (when in it)
    // A ring of exactly 128 rows holds the whole window: row `key` of the tile is
    // ring slot `key`, loaded without waiting for the query's position (the keys'
    // order within a chunk does not change the softmax) as one bulk copy of the
    // sequence's 64 KB of codes into the query buffer (free until the queries
    // arrive) and its 512 B of scales into the E2M1 table's space (unused by the
    // window chunk); otherwise row `key` is the window's token lo + key.
    const bool ring_order = window && swa.rows == AC_KEYS && ((uintptr_t)swa.scales & 15) == 0;
    float *ring_sc = reinterpret_cast<float *>(&S.e2m1_pair[0][0]);
    auto load_ring = [&]() {
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(&S.tbar, AC_KEYS * CSA2_HEAD_DIM + AC_KEYS * 4);
#pragma unroll
            for (int i = 0; i < 4; i++)
                tc::bulk_load(S.u.q + i * (AC_KEYS * CSA2_HEAD_DIM / 4),
                              swa.codes + (int64_t)b * AC_KEYS * CSA2_HEAD_DIM + i * (AC_KEYS * CSA2_HEAD_DIM / 4),
                              AC_KEYS * CSA2_HEAD_DIM / 4, &S.tbar);
            tc::bulk_load(ring_sc, swa.scales + (int64_t)b * AC_KEYS, AC_KEYS * 4, &S.tbar);
        }
    };
    if (window) {
        t = bt.q_pos[r];
        const int64_t s0 = swa.start ? swa.start[b] : 0;
        lo = t - (CSA2_SWA_WINDOW - 1);
        lo = lo < s0 ? s0 : lo;
        lo = lo < 0 ? 0 : lo;
        kn = ring_order ? (int)(t & (AC_KEYS - 1)) : (int)(t - lo);
    }
    // the selected entry of this thread's key (main KV)
    auto load_selected = [&]() {
        const int64_t vis = visible_entries(bt, r);
        // window de-duplication (m = 1): a selected entry that is also a window row is dropped
        int64_t dlo = 1, dhi = 0;
        if ((swa.flags & CSA2_ATTN_DEDUP_WINDOW) && bt.m == 1) {
            dhi = bt.q_pos[r];
            const int64_t s0 = swa.start ? swa.start[b] : 0;
            dlo = dhi - (CSA2_SWA_WINDOW - 1);
            dlo = dlo < s0 ? s0 : dlo;
            dlo = dlo < 0 ? 0 : dlo;
        }
        const int j = chunk * AC_KEYS + key;
        if (j < k) {
            const int32_t p = idx[r * k + j];
            if (p >= 0 && !(p >= dlo && p <= dhi)) {
                if (p >= vis) {
                    if (qq == 0 && d == 0) flag(c.status, CSA2_DEV_BAD_INDEX);
                } else {
                    const int64_t slot = entry_slot(c, b, p);
                    if (slot >= 0) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(c.kv_codes + slot * 256 + 64 * qq);
#pragma unroll
                        for (int i = 0; i < 4; i++) kc[i] = __ldg(src + i);
                        if (c.kv_format == CSA2_KV_FP4_E4M3)
                            ksc = __ldg(reinterpret_cast<const uint2 *>(c.kv_scales + slot * 32 + 8 * qq));
                        else
                            ksc.x = __ldg(reinterpret_cast<const uint32_t *>(c.kv_scales + slot * 16 + 4 * qq));
                        valid = true;
                    }
                }
            }
        }
    };
    // a window row (in ring order: any slot, the query's own included; otherwise
    // one other than the query's own token's)
    auto load_window_row = [&]() {
        if (ring_order) {
            // the staged ring (load_ring, waited for by the caller)
            kscale = ring_sc[key];
            // the slot holds the latest token u <= t with u = key (mod 128): t - u below
            valid = ((t - key) & (AC_KEYS - 1)) <= t - lo;
        } else if (lo + key <= t && key != kn) {
            const int64_t off = (int64_t)b * swa.rows + (lo + key) % swa.rows;
            const uint4 *src = reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM + 128 * qq);
#pragma unroll
            for (int i = 0; i < 8; i++) kc[i] = __ldg(src + i);
            kscale = swa.scales[off];
            valid = true;
        }
    };
    // dequantise the loaded key into row `key` of the key tile (zeros if none)
    auto store_key = [&]() {
        if (valid) {
            if (ring_order) stage_window_key(S.k, S.u.q, key, qq, (uint32_t)lane);
            else if (window) store_window_key(S.k, key, kc, qq);
            else if (c.kv_format == CSA2_KV_FP4_E4M3) store_main_key<true>(S.k, key, kc, ksc, qq, S.e2m1_pair, (uint32_t)lane);
            else store_main_key<false>(S.k, key, kc, ksc, qq, S.e2m1_pair, (uint32_t)lane);
        } else {
            zero_key(S.k, key, qq);
        }
        if (qq == 0) S.kscale[key] = valid ? kscale : -1.0f;
    };

    // Everything before the wait touches only this CTA's own state, except with
    // `early`, where the caller has guaranteed that the index array, the selected
    // entries and the window rows other than the query's own token were written
    // before the previous kernel's predecessors (a Reuse layer after another
    // layer call): those keys are then loaded and dequantised while that kernel
    // finishes.
    bool stored = tread;                           // a carried tile holds every key of the chunk
    uint32_t ring_word = 0;                        // the new token's window row, stored at the end
    int64_t ring_idx = -1, ring_scale_idx = -1;
    bool rfail = false;                            // the staged ring's copy timed out
    if (early && !tread) {
        if (ring_order) {
            __syncthreads();                       // the barrier's initialisation is visible
            load_ring();
            rfail = __syncthreads_or(!tc::mbar_wait(&S.tbar, 0, polls));
        }
        if (window) load_window_row();
        else load_selected();
        __syncthreads();                           // the pair table is ready
        if (!window || key != kn || ring_order) {  // (a new row for slot kn overwrites it below)
            store_key();
            stored = true;
        }
        if (ring_order) __syncthreads();           // every staged row read before the queries land
    }
    pdl_wait();
    if (tread && tile_mode == 2) load_tile();

    // ---- the decode token's new window row (issued first: its quantisation is the
    //      window chunk's longest chain), then the row's queries, all 64 heads and
    //      512 dims (coalesced 16-byte loads), stored as they arrive
    const bool newrow = window && kn >= 0 && kn < AC_KEYS && swa.new_rows && (warp & 3) == (kn >> 5);
    float4 nv[4];
    if (newrow) {
        const float4 *nr = reinterpret_cast<const float4 *>(swa.new_rows + r * CSA2_HEAD_DIM);
#pragma unroll
        for (int c4 = 0; c4 < 4; c4++) nv[c4] = __ldg(nr + c4 * 32 + lane);
    }
    constexpr int QCH = CSA2_HEAD_DIM / 8;         // 16-byte chunks per head
    constexpr int QV = CSA2_HEADS * QCH / AC_THREADS;
    {
        uint4 qv[QV];
        const uint4 *src = reinterpret_cast<const uint4 *>(qr);
#pragma unroll
        for (int i = 0; i < QV; i++) qv[i] = __ldg(src + tid + AC_THREADS * i);
        // keys not loaded before the wait: their lookups overlap the queries' loads
        // (a staged ring is dequantised out of the query buffer before the queries
        // are stored into it)
        if (!early && !tread) {
            if (ring_order) {
                __syncthreads();                   // the barrier's initialisation is visible
                load_ring();
                rfail = __syncthreads_or(!tc::mbar_wait(&S.tbar, 0, polls));
                load_window_row();
                if (key != kn || !swa.new_rows) {
                    store_key();
                    stored = true;
                }
                __syncthreads();                   // every staged row read before the queries land
            } else if (window) {
                load_window_row();
            } else {
                load_selected();
            }
        }
#pragma unroll
        for (int i = 0; i < QV; i++) {
            const int e = tid + AC_THREADS * i;
            *reinterpret_cast<uint4 *>(S.u.q + tc::sw128_offset(e / QCH, 8 * (e % QCH), CSA2_HEADS)) = qv[i];
        }
    }
    if (newrow) {
        // this warp holds quarter qq of the new token's key (lane kn % 32): the warp
        // takes the row's largest magnitude; each lane quantises the four dims
        // 128 qq + 4 lane .. exactly as the FP8 quantiser would and puts them,
        // widened exactly to bf16, into the key tile's row kn; the ring row is
        // stored at the end of the kernel
        float amax = 0.0f;
#pragma unroll
        for (int c4 = 0; c4 < 4; c4++)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(nv[c4].x), fabsf(nv[c4].y)), fmaxf(fabsf(nv[c4].z), fabsf(nv[c4].w))));
#pragma unroll
        for (int o2 = 16; o2; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
        const float sc = fp8_row_scale(amax);
        const float4 x = qq == 0 ? nv[0] : qq == 1 ? nv[1] : qq == 2 ? nv[2] : nv[3];
        const uint32_t wd = f32x2_to_e4m3x2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc)) |
                            (f32x2_to_e4m3x2(__fdiv_rn(x.z, sc), __fdiv_rn(x.w, sc)) << 16);
        const uint2 kb = make_uint2(e4m3x2_to_bf16x2(__byte_perm(wd, 0, 0x4140)),
                                    e4m3x2_to_bf16x2(__byte_perm(wd, 0, 0x4342)));
        *reinterpret_cast<uint2 *>(S.k + tc::sw128_offset((uint32_t)kn, 128 * qq + 4 * lane, AC_KEYS)) = kb;
        if (d == 0) {                              // one CTA of the chunk writes the ring
            ring_word = wd;
            ring_idx = (b * (int64_t)swa.rows + t % swa.rows) * (CSA2_HEAD_DIM / 4) + 32 * qq + lane;
        }
        if (key == kn) {
            if (d == 0 && qq == 0) ring_scale_idx = (int64_t)b * swa.rows + t % swa.rows;
            kscale = sc;
            valid = true;
            stored = true;                         // its row of the key tile is written above
            if (qq == 0) S.kscale[key] = sc;
        }
    } else if (window && !ring_order && kn >= 0 && kn < AC_KEYS && !swa.new_rows && key == kn) {
        // the own token's row, written before this call
        const int64_t off = (int64_t)b * swa.rows + t % swa.rows;
        const uint4 *src = reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM + 128 * qq);
#pragma unroll
        for (int i = 0; i < 8; i++) kc[i] = __ldg(src + i);
        kscale = swa.scales[off];
        valid = true;
    }

    __syncthreads();                               // the pair table is ready
    if (!stored) store_key();
    // a carried tile: every thread waits for its bytes (async proxy, acquired
    // through the barrier; the tensor core reads them through the same proxy)
    const bool tfail = tread && __syncthreads_or(!tc::mbar_wait(&S.tbar, 0, polls));
    if (tfail && tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);

    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    // a selecting layer leaves the chunk's dequantised tile for the Reuse layers:
    // each CTA of the chunk stores the slabs of its half of the dims, half 0 the
    // key scales (bulk stores, read from shared memory while the products run)
    if (twrite && tid == 0) {
#pragma unroll
        for (int sl = AC_SLABS / AC_HALVES * d; sl < AC_SLABS / AC_HALVES * (d + 1); sl++)
            tc::bulk_store(tile_g + sl * (AC_KEYS * 128), S.k + sl * (AC_KEYS * 128), AC_KEYS * 128);
        if (d == 0) tc::bulk_store(tile_g + AC_TILE_BYTES, S.kscale, AC_KEYS * 4);
        tc::bulk_commit();
    }

    // ---- S^T = K Q^T over all 512 dims (16 per K step)
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k), q0 = tc::smem_u32(S.u.q);
#pragma unroll
        for (int kk = 0; kk < CSA2_HEAD_DIM / 16; kk++) {
            const uint32_t off = (uint32_t)(kk >> 2) * (AC_KEYS * 128) + (uint32_t)(kk & 3) * 32u;
            const uint32_t offq = (uint32_t)(kk >> 2) * (CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
            tc::mma_f16(tmem + AC_S_COL, tc::smem_desc(k0 + off, 16, 1024, tc::kSwizzle128B),
                        tc::smem_desc(q0 + offq, 16, 1024, tc::kSwizzle128B), AC_IDESC_S, kk > 0);
        }
        tc::mma_commit(&S.mbar);
    }
    // the next kernel on the stream may be scheduled now (it waits for this grid
    // before reading anything this one writes)
    pdl_launch_dependents();
    // A CTA whose product timed out writes no partial output and flags the
    // status word; it still reaches the cluster barrier below.
    const bool fail = __syncthreads_or(!tc::mbar_wait(&S.mbar, 0, polls));
    tc::tc_fence_after();
    if (!fail) {
        // warp w: keys of its lane quarter, heads 16 (w >> 2) .. + 15, into the
        // logits [head][key] (Q is no longer read)
        const uint32_t col = 16u * (uint32_t)(warp >> 2);
        uint32_t acc[16];
        tc::tmem_ld16(tmem + lane_base + AC_S_COL + col, acc);
        tc::tmem_ld_wait();
        const int kr = (warp & 3) * 32 + lane;
#pragma unroll
        for (int j = 0; j < 16; j++) S.u.sp.s[col + j][kr] = __uint_as_float(acc[j]);
    } else if (tid == 0) {
        flag(c.status, CSA2_DEV_TIMEOUT);
    }
    __syncthreads();

    // ---- softmax of the chunk: eight threads per head; thread `part` takes keys
    //      32 i + 4 part .. + 3 (i < 4), so that a head's threads read 128
    //      contiguous bytes of logits and key scales (no bank conflicts)
    if (!fail) {
        const int h = tid >> 3, part = tid & 7;
        float lg[16], ksv[16];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float4 v = *reinterpret_cast<const float4 *>(&S.u.sp.s[h][32 * i + 4 * part]);
            const float4 ks = *reinterpret_cast<const float4 *>(&S.kscale[32 * i + 4 * part]);
            const float sv[4] = {v.x, v.y, v.z, v.w};
            ksv[4 * i] = ks.x;
            ksv[4 * i + 1] = ks.y;
            ksv[4 * i + 2] = ks.z;
            ksv[4 * i + 3] = ks.w;
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                const float kv = ksv[4 * i + jj];                         // -1: no key
                lg[4 * i + jj] = kv >= 0.0f ? sv[jj] * (sm_scale * kv) : -INFINITY;
                mx = fmaxf(mx, lg[4 * i + jj]);
            }
        }
#pragma unroll
        for (int o2 = 1; o2 < 8; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        float l = 0.0f;
        uint32_t hi2[8], lo2[8];                   // bf16 pairs of keys (32 i + 4 part + 2 u, + 1)
#pragma unroll
        for (int jj = 0; jj < 16; jj += 2) {
            const float e0 = mx != -INFINITY && lg[jj] != -INFINITY ? __expf(lg[jj] - mx) : 0.0f;
            const float e1 = mx != -INFINITY && lg[jj + 1] != -INFINITY ? __expf(lg[jj + 1] - mx) : 0.0f;
            l += e0 + e1;
            const float p0 = e0 * fmaxf(ksv[jj], 0.0f), p1 = e1 * fmaxf(ksv[jj + 1], 0.0f);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
            const float2 hf2 = __bfloat1622float2(hi);
            const __nv_bfloat162 lw = __floats2bfloat162_rn(p0 - hf2.x, p1 - hf2.y);
            hi2[jj >> 1] = *reinterpret_cast<const uint32_t *>(&hi);
            lo2[jj >> 1] = *reinterpret_cast<const uint32_t *>(&lw);
        }
#pragma unroll
        for (int o2 = 1; o2 < 8; o2 <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o2);
        // 8 consecutive keys 32 i + 8 (part / 2) .. make one 16-byte chunk of a row of
        // the probability operand: the even thread of a pair writes it to the hi row h,
        // the odd one to the lo row 64 + h, each after one shuffle with its neighbour
        const bool even = (part & 1) == 0;
        const uint32_t row = even ? (uint32_t)h : (uint32_t)(CSA2_HEADS + h);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t s0 = even ? lo2[2 * i] : hi2[2 * i], s1 = even ? lo2[2 * i + 1] : hi2[2 * i + 1];
            const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1), r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
            const uint4 w = even ? make_uint4(hi2[2 * i], hi2[2 * i + 1], r0, r1)
                                 : make_uint4(r0, r1, lo2[2 * i], lo2[2 * i + 1]);
            const uint32_t c16 = (uint32_t)(4 * (i & 1) + (part >> 1));   // chunk of the 64-key slab i / 2
            const uint32_t off = (uint32_t)(i >> 1) * (2 * CSA2_HEADS * 128) + row * 128u + ((c16 ^ (row & 7u)) << 4);
            *reinterpret_cast<uint4 *>(S.u.sp.p + off) = w;
        }
        // each half keeps its own copy of (m, l) (the two are equal): its cluster's
        // barrier orders only its own CTAs' writes
        if (part == 0) *reinterpret_cast<float2 *>(part_ml + ((base + h) * AC_HALVES + d) * 2) = make_float2(mx, l);
    }
    // the probability rows, written through the generic proxy, are read by the tensor core
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- [O_hi | O_lo]^T = V_d^T [P_hi | P_lo]^T: M-tiles of 128 of this CTA's dims,
    //      K = 128 keys, N = 128; tile mt in columns 128 mt .. 128 mt + 127
    if (tid == 0 && !fail) {
        const uint32_t k0 = tc::smem_u32(S.k), p0 = tc::smem_u32(S.u.sp.p);
#pragma unroll
        for (int mt = 0; mt < AC_MT; mt++) {
            const uint32_t slab = (uint32_t)(AC_DH / 64 * d + 2 * mt);     // first 64-dim slab of the tile
#pragma unroll
            for (int kk = 0; kk < AC_KEYS / 16; kk++) {   // 16 keys per step
                const uint64_t ad = tc::smem_desc(k0 + slab * (AC_KEYS * 128) + (uint32_t)kk * 2048u,
                                                  AC_KEYS * 128, 1024, tc::kSwizzle128B);
                const uint32_t boff = (uint32_t)(kk >> 2) * (2 * CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                tc::mma_f16(tmem + 128u * (uint32_t)mt, ad, tc::smem_desc(p0 + boff, 16, 1024, tc::kSwizzle128B),
                            AC_IDESC_O, kk > 0);
            }
        }
        tc::mma_commit(&S.mbar);
    }
    bool fail2 = fail;
    if (!fail) {
        fail2 = __syncthreads_or(!tc::mbar_wait(&S.mbar, 1, polls));
        tc::tc_fence_after();
        if (!fail2) {
            // ---- partial output: warp w takes M-tile (w >> 2) & 1, lane quarter w & 3
            //      (lane = dim) and heads 32 (w >> 3) .. + 31; hi + lo
            const int mt = (warp >> 2) & 1, hh = warp >> 3;
            uint32_t ahi[32], alo[32];
            const uint32_t colo = 128u * (uint32_t)mt + 32u * (uint32_t)hh;
            tc::tmem_ld32(tmem + lane_base + colo, ahi);
            tc::tmem_ld32(tmem + lane_base + colo + CSA2_HEADS, alo);
            tc::tmem_ld_wait();
            float *po = part_o + (base + 32 * hh) * CSA2_HEAD_DIM + AC_DH * d + 128 * mt + (warp & 3) * 32 + lane;
#pragma unroll
            for (int j = 0; j < 32; j++)
                po[(int64_t)j * CSA2_HEAD_DIM] = __uint_as_float(ahi[j]) + __uint_as_float(alo[j]);
        } else if (tid == 0) {
            flag(c.status, CSA2_DEV_TIMEOUT);
        }
    }
    // the new token's FP8 window row (codes and scale) into the ring
    if (ring_idx >= 0) reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(swa.codes))[ring_idx] = ring_word;
    if (ring_scale_idx >= 0) const_cast<float *>(swa.scales)[ring_scale_idx] = kscale;

    // ---- tensor memory back: a product that timed out may still be running, so
    //      its commit is awaited (long limit) before the columns are freed; so is
    //      a tile copy that timed out (it writes into this CTA's shared memory)
    if (tid == 0 && (tfail || rfail)) tc::mbar_wait(&S.tbar, 0, 1u << 26);
    if (rfail && tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);
    if (tid == 0 && fail) tc::mbar_wait(&S.mbar, 0, 1u << 26);
    if (tid == 0 && fail2 && !fail) tc::mbar_wait(&S.mbar, 1, 1u << 26);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, AC_TMEM_COLS);

    // ---- every chunk of this half has written its partials (release / acquire
    //      at cluster scope orders those global writes before the reads below)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");

    // ---- merge: item (head, lane j) of this half, one per thread of the cluster:
    //      the float4s of dims 4 j .. and 128 + 4 j .. of the half (each warp load
    //      is 512 contiguous bytes), every load of an item issued at once; with
    //      the output rotation (half 1), lanes 16..23 hold dims 448 + .. and
    //      lanes 24..31 their RoPE partners 32 dims on, exchanged by one shuffle
    const bool rot = rope && d == AC_HALVES - 1;
    const int cr = (int)cluster_rank();
    for (int it0 = cr * AC_THREADS; it0 < CSA2_HEADS * 32; it0 += nchunks * AC_THREADS) {
        const int it = it0 + tid;                  // warps run whole heads: it / 32 is warp-uniform
        if (it >= CSA2_HEADS * 32) break;
        const int h = it >> 5, jl = it & 31;
        const int64_t rb = r * AC_MAX_CHUNKS * CSA2_HEADS + h;     // (row, chunk 0, head)
        const int dim0 = AC_DH * d + 4 * jl;
        float mc[AC_MAX_CHUNKS], lc[AC_MAX_CHUNKS];
        float4 v[AC_MAX_CHUNKS][2];
        float M = -INFINITY;
#pragma unroll
        for (int ch = 0; ch < AC_MAX_CHUNKS; ch++) {
            mc[ch] = -INFINITY;
            lc[ch] = 0.0f;
            v[ch][0] = v[ch][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ch < nchunks) {
                // written by other CTAs of the cluster in this launch: read at L2 (.cg)
                const int64_t e = rb + (int64_t)ch * CSA2_HEADS;
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(part_ml + (e * AC_HALVES + d) * 2));
                const float4 *src = reinterpret_cast<const float4 *>(part_o + e * CSA2_HEAD_DIM + dim0);
                mc[ch] = ml.x;
                lc[ch] = ml.y;
                v[ch][0] = __ldcg(src);
                v[ch][1] = __ldcg(src + 32);
                M = fmaxf(M, ml.x);
            }
        }
        float L = 0.0f;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (M != -INFINITY) {
#pragma unroll
            for (int ch = 0; ch < AC_MAX_CHUNKS; ch++) {
                if (mc[ch] == -INFINITY) continue;
                const float wgt = expf(mc[ch] - M);
                L = fmaf(wgt, lc[ch], L);
                const float x[8] = {v[ch][0].x, v[ch][0].y, v[ch][0].z, v[ch][0].w,
                                    v[ch][1].x, v[ch][1].y, v[ch][1].z, v[ch][1].w};
#pragma unroll
                for (int i = 0; i < 8; i++) a[i] = fmaf(wgt, x[i], a[i]);
            }
        }
        const float z = swa.sink ? swa.sink[h] : -INFINITY;
        if (z != -INFINITY) {
            if (M == -INFINITY || z > M) {          // the sink sets the reference maximum
                const float f = M == -INFINITY ? 0.0f : expf(M - z);
                L = fmaf(L, f, 1.0f);
#pragma unroll
                for (int i = 0; i < 8; i++) a[i] *= f;
                M = z;
            } else {
                L += expf(z - M);
            }
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) a[i] *= inv;
        if (rot) {
            // pair i (dims 448 + i, 480 + i), rotated by -t theta_i: lane 16 + i / 4 holds
            // the first in its second float4, lane 24 + i / 4 the second
            float oth[4];
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) oth[c4] = __shfl_xor_sync(0xffffffffu, a[4 + c4], 8);
            if (jl >= 16) {
                const bool first = jl < 24;
                const int64_t tq = bt.q_pos[r];
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    float sn, cs;
                    rope_sincos(tq, turns.phi[4 * ((jl - 16) & 7) + c4], &sn, &cs);
                    // (x, y) -> (x cos + y sin, -x sin + y cos); this lane holds x (first) or y
                    a[4 + c4] = first ? fmaf(a[4 + c4], cs, oth[c4] * sn) : fmaf(a[4 + c4], cs, -oth[c4] * sn);
                }
            }
        }
        float *orow = o + (r * CSA2_HEADS + h) * CSA2_HEAD_DIM + dim0;
        *reinterpret_cast<float4 *>(orow) = make_float4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<float4 *>(orow + 128) = make_float4(a[4], a[5], a[6], a[7]);
        if (d == 0 && jl == 0) lse[r * CSA2_HEADS + h] = L > 0.0f ? M + logf(L) : -INFINITY;
    }
    // the tile's bulk stores have completed before the CTA's shared memory is released
    if (twrite && tid == 0) tc::bulk_wait_all();
}

size_t attn_workspace_bytes(int64_t rows)
{
    const size_t po = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4;
    const size_t ml = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * AC_HALVES * 2 * 4;
    return ((po + 255) & ~(size_t)255) + ml;
}

size_t attn_tile_bytes(int64_t rows) { return (size_t)rows * (AC_MAX_CHUNKS - 1) * AC_TILE_STRIDE; }

int launch_attn(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale, const int32_t *idx,
                int k, const csa2_swa &swa, float *o, float *lse, void *ws, size_t ws_bytes, cudaStream_t st,
                bool early, uint8_t *tiles, int tile_mode)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    if (ws_bytes < attn_workspace_bytes(rows) || !ws) return CSA2_ERR_WORKSPACE;
    if (rows > 65535) return CSA2_ERR_SHAPE;       // rows run along the grid's y dimension
    const size_t po_bytes = ((size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4 + 255) & ~(size_t)255;
    float *part_o = static_cast<float *>(ws);
    float *part_ml = reinterpret_cast<float *>(static_cast<char *>(ws) + po_bytes);
    const int nchunks = (k + AC_KEYS - 1) / AC_KEYS + 1;
    if (tiles && (k != CSA2_TOPK || !aligned(tiles, 16))) return CSA2_ERR_UNSUPPORTED;
    const size_t smem = sizeof(AcSmem) + 1024;
    if (const int s = kernel_smem_limit((const void *)k_attn_tc, smem, 100)) return s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;  // the chunks of one (row, half of the dims)
    at[0].val.clusterDim.x = (unsigned)nchunks;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(AC_HALVES * nchunks), (unsigned)rows);
    cfg.blockDim = dim3(AC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_attn_tc, c, bt, q, sm_scale, idx, k, swa,
                                             swa.rope_base > 0.0f ? 1 : 0, rope_turns(swa.rope_base), part_o,
                                             part_ml, o, lse, nchunks, (int)early, tile_mode ? tiles : nullptr,
                                             tiles ? tile_mode : 0, wait_polls());
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace csa2
