// Sparse MQA + sliding-window attention on the tcgen05 tensor cores.
//
// Every key is its own value ("DeepSeek-V4 report explainer" §4.3) and one
// softmax covers the selected entries and the window ("DeepSeek-V4.1-Flash
// 架构详解" §1 table, §3; explainer §3.3).
//
// Work unit (row, chunk): 128 keys -- chunks 0..3 the selected entries
// idx[128c .. 128c+127], the last chunk the window rows -- and all 64 heads.
// A cluster of two CTAs takes one unit, CTA d the dims 256 d .. 256 d + 255
// (the cluster size is a compile-time constant; four CTAs of 128 dims also
// work but leave some SMs with two CTAs of one launch on an 8-row decode):
//   1. dequantise its slice of the keys into a 128 x 256 bf16 tile: MXFP4
//      bytes through a 256-entry table (byte -> two bf16 magnitudes with
//      signs) and one bf16x2 multiply by 2^X per block; window codes e4m3 by
//      placing their bits in a bf16 and one multiply by 2^120 -- both exact;
//      the window's fp32 row scale is applied to the logit and to the
//      probability instead;
//   2. partial S^T[128 keys x 64 heads] = K_d Q_d^T over its dims (M = keys,
//      N = heads), read out of tensor memory into shared memory; the 32-head
//      slice each other CTA owns goes to it by one bulk shared-to-shared copy
//      that completes on that CTA's mbarrier (no cluster-wide barrier, no
//      cluster-scope proxy fence);
//   3. CTA d sums the partials of heads 32 d .. 32 d + 31 (in rank order, so
//      every run gives the same logits), takes their max m_c and sum l_c over
//      the chunk, writes P = exp(S - m_c) as bf16 hi + lo (P = hi + lo to
//      2^-17) into its own probability operand and bulk-copies those rows to
//      the other CTA in the same way;
//   4. [O_hi | O_lo]_d^T = V_d^T [P_hi | P_lo]^T, reading the same key tile
//      as an MN-major operand (V = K; M-tiles of 128 dims, K = 128 keys,
//      N = 128); the epilogue adds the two halves;
//   5. the unnormalised partial O_c (this CTA's dims) and (m_c, l_c) go to the
//      workspace.
// A second kernel merges the chunks of each row: O = sum_c e^(m_c-M) O_c / L.
// 512 threads: four per key (64 dims each) for the loads and dequantisation,
// sixteen per owned head for the softmax, one TMEM lane each in the epilogues.
#include <algorithm>

#include "csa2_attn_common.cuh"

namespace csa2 {

struct AcSmem {
    uint8_t k[AC_SLABS * AC_KEYS * 128];           // [slab of 64 dims][128 keys][128 B]
    union {
        uint8_t q[AC_SLABS * CSA2_HEADS * 128];    // [slab][64 heads][128 B] 32 KB
        float pout[CSA2_HEADS][AC_KEYS];           // this CTA's partial logits [head][key], written
    } u;                                           // once the first product is done with Q
    uint8_t p[2 * 2 * CSA2_HEADS * 128];           // [slab of 64 keys][hi 64 | lo 64 rows][128 B] 32 KB:
                                                   // this CTA's heads written here, the others' rows
                                                   // copied in by their owners
    float ps[AC_CL][AC_OWN][AC_KEYS];              // [source CTA][owned head][key]: the other CTAs'
                                                   // partial logits of this CTA's heads (copied in)
    uint32_t e2m1_pair[256][32];                   // byte -> bf16x2 of its two E2M1 codes, one
                                                   // copy per lane (bank = lane: no conflicts)  32 KB
    float kscale[AC_KEYS];                         // window row scale (1 for entries), -1: no key
    float2 mlv[AC_OWN];                            // (m_c, l_c) of the owned heads, held until the
                                                   // workspace may be written (early = 2)
    uint64_t mbar;                                 // the products' commits
    uint64_t sbar;                                 // the other CTAs' partial logits have landed
    uint64_t pbar;                                 // the other CTAs' probability rows have landed
    uint32_t tmem;
};


__global__ void __cluster_dims__(AC_CL, 1, 1) __launch_bounds__(AC_THREADS, AC_CL == 4 ? 2 : 1)
    k_attn_tc(csa2_cache c, csa2_batch bt, const uint16_t *__restrict__ q, float sm_scale,
              const int32_t *__restrict__ idx, int k, csa2_swa swa, float *__restrict__ part_o,
              float *__restrict__ part_ml, int nchunks, int early, uint32_t polls)
{
    extern __shared__ uint8_t smem_raw[];
    AcSmem &S = *reinterpret_cast<AcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int key = tid & (AC_KEYS - 1), hf = tid >> 7;          // key row; 64-dim slab of this CTA
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16; // TMEM lane quarter of this warp
    const uint32_t dq = cluster_rank();                           // dims AC_DIMS dq .. + AC_DIMS - 1
    const int chunk = blockIdx.x / AC_CL;
    const int64_t r = blockIdx.y;
    const int b = (int)(r / bt.nq);
    const bool window = chunk == nchunks - 1;
    const int64_t base = (r * AC_MAX_CHUNKS + chunk) * (int64_t)CSA2_HEADS;

    if (tid == 0) {
        tc::mbar_init(&S.mbar, 1);
        tc::mbar_init(&S.sbar, 1);
        tc::mbar_init(&S.pbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem, AC_TMEM_COLS);
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&S.sbar, AC_S_IN_BYTES);    // the other CTAs' partial logits
        tc::mbar_arrive_expect_tx(&S.pbar, AC_P_IN_BYTES);    // and probability rows
    }
    // first half of a cluster barrier: this CTA's mbarriers are initialised; the
    // matching wait comes before the first copy into another CTA
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    // E2M1 pair table: 2048 16-byte chunks of four copies each, consecutive per lane
#pragma unroll
    for (int ch = tid; ch < 256 * 32 / 4; ch += AC_THREADS) {
        const uint32_t v = e2m1x2_to_bf16x2((uint32_t)ch >> 3);
        reinterpret_cast<uint4 *>(&S.e2m1_pair[0][0])[ch] = make_uint4(v, v, v, v);
    }
    // ---- this thread's key: locate it and load its 64 dims
    float kscale = 1.0f;          // multiplies the logit and the probability (window rows)
    bool valid = false;
    uint4 kc[4];
    uint32_t ksc = 0;
    int64_t t = 0, lo = 0;
    int kn = -1;                  // the query's own token in the window chunk (when in it)
    if (window) {
        t = bt.q_pos[r];
        const int64_t s0 = swa.start ? swa.start[b] : 0;
        lo = t - (CSA2_SWA_WINDOW - 1);
        lo = lo < s0 ? s0 : lo;
        lo = lo < 0 ? 0 : lo;
        kn = (int)(t - lo);
    }
    // the selected entry of this thread's key (main KV)
    auto load_selected = [&]() {
        const int64_t vis = visible_entries(bt, r);   // issued alongside the index load
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
                    if (hf == 0 && dq == 0) flag(c.status, CSA2_DEV_BAD_INDEX);
                } else {
                    const int64_t slot = entry_slot(c, b, p);
                    if (slot >= 0) {
                        const uint4 *src =
                            reinterpret_cast<const uint4 *>(c.kv_codes + slot * 256 + AC_DIMS / 2 * dq) + 2 * hf;
                        kc[0] = __ldg(src);
                        kc[1] = __ldg(src + 1);
                        ksc = c.kv_format == CSA2_KV_FP4_E4M3
                                  ? __ldg(reinterpret_cast<const uint32_t *>(c.kv_scales + slot * 32 + AC_DIMS / 16 * dq) +
                                          hf)
                                  : __ldg(reinterpret_cast<const uint16_t *>(c.kv_scales + slot * 16 + AC_DIMS / 32 * dq) +
                                          hf);
                        valid = true;
                    }
                }
            }
        }
    };
    // a window row other than the query's own token's
    auto load_window_row = [&]() {
        if (lo + key <= t && key != kn) {
            const int64_t off = (int64_t)b * swa.rows + (lo + key) % swa.rows;
            const uint4 *src =
                reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM + AC_DIMS * dq) + 4 * hf;
#pragma unroll
            for (int i = 0; i < 4; i++) kc[i] = __ldg(src + i);
            kscale = swa.scales[off];
            valid = true;
        }
    };
    // dequantise the loaded key into row `key` of the key tile (zeros if none)
    auto store_key = [&]() {
        if (valid) {
            if (window) store_window_key(S.k, key, kc, hf);
            else if (c.kv_format == CSA2_KV_FP4_E4M3) store_main_key<true>(S.k, key, kc, ksc, hf, S.e2m1_pair, (uint32_t)lane);
            else store_main_key<false>(S.k, key, kc, ksc, hf, S.e2m1_pair, (uint32_t)lane);
        } else {
            zero_key(S.k, key, hf);
        }
        if (hf == 0) S.kscale[key] = valid ? kscale : -1.0f;
    };

    // Launched as a programmatic dependent of the previous kernel on the stream:
    // everything before the wait touches only this CTA's own state, except with
    // `early`, where the caller has guaranteed that the index array, the selected
    // entries and the window rows other than the query's own token were written
    // before that kernel's predecessors (a Reuse layer after another layer call):
    // those keys are then loaded and dequantised while that kernel finishes.  With
    // early = 2 the caller has also written q and new_rows before then and given
    // this call a workspace of its own: the whole computation runs before the
    // wait, which comes only before the workspace is written (the previous merge
    // may still be reading its own).
    bool stored = false;
    uint32_t ring_word = 0;                        // the new token's window row, stored at the end
    int64_t ring_idx = -1, ring_scale_idx = -1;
    // this CTA's slice of the queries (64 heads x AC_DIMS dims: one 128-byte line
    // per thread) and the decode token's new window row into L2 while the previous
    // kernel finishes: a prefetch carries no data into this CTA, so it may run
    // before the wait
    if (tid < CSA2_HEADS * AC_DIMS * 2 / 128) {
        constexpr int LPH = AC_DIMS * 2 / 128;     // lines per head
        prefetch_l2(q + (r * CSA2_HEADS + tid / LPH) * CSA2_HEAD_DIM + AC_DIMS * dq + 64 * (tid % LPH));
    } else if (window && swa.new_rows && tid - CSA2_HEADS * AC_DIMS * 2 / 128 < CSA2_HEAD_DIM * 4 / 128) {
        prefetch_l2(swa.new_rows + r * CSA2_HEAD_DIM + 32 * (tid - CSA2_HEADS * AC_DIMS * 2 / 128));
    }
    if (early) {
        if (window) load_window_row();
        else load_selected();
        __syncthreads();                           // the pair table is ready
        if (!window || key != kn) {
            store_key();
            stored = true;
        }
    }
    if (early < 2) pdl_wait();

    // ---- this CTA's dims of the 64 queries (coalesced 16-byte loads)
    constexpr int QCH = AC_DIMS / 8;               // 16-byte chunks per head
    uint4 qv[4];
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(q + r * CSA2_HEADS * CSA2_HEAD_DIM + AC_DIMS * dq);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int e = tid + AC_THREADS * i;
            qv[i] = __ldg(src + (e / QCH) * (CSA2_HEAD_DIM / 8) + (e % QCH));
        }
    }
    if (!early) {
        if (window) load_window_row();
        else load_selected();
    }
    if (window && kn >= 0 && kn < AC_KEYS) {
        if (swa.new_rows) {
            if ((warp & 3) == (kn >> 5)) {
                // this warp holds the new token's key in lane kn % 32: the whole warp takes
                // the row's largest magnitude; the 16 lanes that loaded this thread-slab's
                // dims (float4 chunks base .. base + 15 of the row) each quantise four of
                // them exactly as the FP8 quantiser would and store them to the ring; the
                // key's lane collects the 16 words
                const float4 *nr = reinterpret_cast<const float4 *>(swa.new_rows + r * CSA2_HEAD_DIM);
                float4 v[4];
                float amax = 0.0f;
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    v[c4] = __ldg(nr + c4 * 32 + lane);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[c4].x), fabsf(v[c4].y)), fmaxf(fabsf(v[c4].z), fabsf(v[c4].w))));
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sc = fp8_row_scale(amax);
                const int base = (AC_DIMS * (int)dq + 64 * hf) / 4;          // first float4 of the slab
                const int cb = base >> 5, lb = base & 31;                     // its register and lane
                const float4 x = cb == 0 ? v[0] : cb == 1 ? v[1] : cb == 2 ? v[2] : v[3];
                const uint32_t wd = f32x2_to_e4m3x2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc)) |
                                    (f32x2_to_e4m3x2(__fdiv_rn(x.z, sc), __fdiv_rn(x.w, sc)) << 16);
                // each of the 16 lanes puts its four codes, widened exactly to bf16, into
                // the key tile's row kn itself (no gathering into the key's lane); the
                // ring row is stored at the end of the kernel
                if (lane >= lb && lane < lb + 16) {
                    ring_word = wd;
                    ring_idx = (int64_t)((b * (int64_t)swa.rows + t % swa.rows) * (CSA2_HEAD_DIM / 4)) + base + (lane - lb);
                    const uint2 kb = make_uint2(e4m3x2_to_bf16x2(__byte_perm(wd, 0, 0x4140)),
                                                e4m3x2_to_bf16x2(__byte_perm(wd, 0, 0x4342)));
                    *reinterpret_cast<uint2 *>(S.k + tc::sw128_offset((uint32_t)kn, 64 * hf + 4 * (lane - lb), AC_KEYS)) = kb;
                }
                if (key == kn) {
                    if (dq == 0 && hf == 0) ring_scale_idx = (int64_t)b * swa.rows + t % swa.rows;
                    kscale = sc;
                    valid = true;
                    stored = true;                 // its row of the key tile is written above
                    if (hf == 0) S.kscale[key] = sc;
                }
            }
        } else if (key == kn) {                    // the own token's row, written before this call
            const int64_t off = (int64_t)b * swa.rows + t % swa.rows;
            const uint4 *src =
                reinterpret_cast<const uint4 *>(swa.codes + off * CSA2_HEAD_DIM + AC_DIMS * dq) + 4 * hf;
#pragma unroll
            for (int i = 0; i < 4; i++) kc[i] = __ldg(src + i);
            kscale = swa.scales[off];
            valid = true;
        }
    }

    // ---- the queries' slice arrives while the key lookups run
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int e = tid + AC_THREADS * i;
        *reinterpret_cast<uint4 *>(S.u.q + tc::sw128_offset(e / QCH, 8 * (e % QCH), CSA2_HEADS)) = qv[i];
    }
    __syncthreads();                               // the pair table is ready
    if (!stored) store_key();

    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;

    // ---- partial S^T = K_d Q_d^T over this CTA's dims
    if (tid == 0) {
        const uint32_t k0 = tc::smem_u32(S.k), q0 = tc::smem_u32(S.u.q);
#pragma unroll
        for (int kk = 0; kk < AC_DIMS / 16; kk++) {   // 16 dims per step
            const uint32_t off = (uint32_t)(kk >> 2) * (AC_KEYS * 128) + (uint32_t)(kk & 3) * 32u;
            const uint32_t offq = (uint32_t)(kk >> 2) * (CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
            tc::mma_f16(tmem, tc::smem_desc(k0 + off, 16, 1024, tc::kSwizzle128B),
                        tc::smem_desc(q0 + offq, 16, 1024, tc::kSwizzle128B), AC_IDESC_S, kk > 0);
        }
        tc::mma_commit(&S.mbar);
    }
    // A CTA whose product timed out still sends its (meaningless) partials and
    // probabilities, so that the other CTAs' bounded waits complete, but writes
    // no output; the status word says why.
    const bool fail = __syncthreads_or(!tc::mbar_wait(&S.mbar, 0, polls));
    tc::tc_fence_after();
    if (!fail) {
        // this warp: keys of its lane quarter, heads col .. col + 64 / AC_SLABS - 1,
        // into this CTA's partial logits [head][key] (Q is no longer read)
        constexpr int NG = 4 / AC_SLABS;           // groups of 16 heads per warp
        const uint32_t col = 64u / AC_SLABS * (uint32_t)(warp >> 2);
        uint32_t acc[NG][16];
#pragma unroll
        for (int g = 0; g < NG; g++) tc::tmem_ld16(tmem + lane_base + col + 16u * g, acc[g]);
        tc::tmem_ld_wait();
        const int kr = (warp & 3) * 32 + lane;
#pragma unroll
        for (int g = 0; g < NG; g++)
#pragma unroll
            for (int j = 0; j < 16; j++) S.u.pout[col + 16 * g + j][kr] = __uint_as_float(acc[g][j]);
    } else if (tid == 0) {
        flag(c.status, CSA2_DEV_TIMEOUT);
    }
    // the partials of each other CTA's heads go to that CTA by one bulk copy (async
    // proxy): generic writes fenced, then issued once every thread has written
    tc::fence_proxy_async_smem();
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // the others' mbarriers exist
    if (tid == 0) {
        const uint32_t sb = tc::smem_u32(&S.sbar);
#pragma unroll
        for (int dst = 0; dst < AC_CL; dst++) {
            if (dst == (int)dq) continue;
            bulk_to_peer(cluster_map(tc::smem_u32(&S.ps[dq][0][0]), (uint32_t)dst),
                         tc::smem_u32(&S.u.pout[AC_OWN * dst][0]), AC_S_BYTES, cluster_map(sb, (uint32_t)dst));
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    // the other CTAs' partials of this CTA's heads have landed
    const bool s_fail = __syncthreads_or(!tc::mbar_wait(&S.sbar, 0, polls));
    if (s_fail && tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);

    // ---- owned heads AC_OWN dq .. : sixteen threads per head, eight
    //      consecutive keys per thread
    {
        const int hl = tid >> 4, h = AC_OWN * (int)dq + hl, part = tid & 15;
        float4 v[AC_CL][2];
#pragma unroll
        for (int src = 0; src < AC_CL; src++) {     // rank order: the same sum in every run
            const float *row = src == (int)dq ? &S.u.pout[h][0] : &S.ps[src][hl][0];
            v[src][0] = *reinterpret_cast<const float4 *>(row + 8 * part);
            v[src][1] = *reinterpret_cast<const float4 *>(row + 8 * part + 4);
        }
        const float4 ks0 = *reinterpret_cast<const float4 *>(&S.kscale[8 * part]);
        const float4 ks1 = *reinterpret_cast<const float4 *>(&S.kscale[8 * part + 4]);
        const float ks[8] = {ks0.x, ks0.y, ks0.z, ks0.w, ks1.x, ks1.y, ks1.z, ks1.w};   // -1: no key
        float lg[8];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float sum = 0.0f;
#pragma unroll
            for (int src = 0; src < AC_CL; src++) {
                const float4 &w = v[src][j >> 2];
                sum += (j & 3) == 0 ? w.x : (j & 3) == 1 ? w.y : (j & 3) == 2 ? w.z : w.w;
            }
            lg[j] = ks[j] >= 0.0f ? sum * (sm_scale * ks[j]) : -INFINITY;
            mx = fmaxf(mx, lg[j]);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float e[8], l = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            e[j] = mx != -INFINITY && lg[j] != -INFINITY ? __expf(lg[j] - mx) : 0.0f;
            l += e[j];
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        uint32_t hi2[4], lo2[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const float p0 = e[j] * fmaxf(ks[j], 0.0f), p1 = e[j + 1] * fmaxf(ks[j + 1], 0.0f);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
            const float2 hf2 = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf2.x, p1 - hf2.y);
            hi2[j >> 1] = *reinterpret_cast<const uint32_t *>(&hi);
            lo2[j >> 1] = *reinterpret_cast<const uint32_t *>(&lo);
        }
        // row h (hi) and 64 + h (lo) of the probability operand, keys 8 part .. +7
        const uint32_t chunk16 = (uint32_t)((part & 7) ^ (h & 7)) << 4;
        const uint32_t off_hi = (uint32_t)(part >> 3) * (2 * CSA2_HEADS * 128) + (uint32_t)h * 128u + chunk16;
        const uint32_t off_lo = off_hi + CSA2_HEADS * 128;
        *reinterpret_cast<uint4 *>(S.p + off_hi) = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
        *reinterpret_cast<uint4 *>(S.p + off_lo) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
        if (part == 0 && !fail && !s_fail) {
            if (early == 2) {
                S.mlv[hl] = make_float2(mx, l);
            } else {
                part_ml[(base + h) * 2] = mx;
                part_ml[(base + h) * 2 + 1] = l;
            }
        }
    }
    // this CTA's rows of P, written through the generic proxy, are read by the
    // tensor core here and by the bulk copies to the other CTAs (async proxy)
    tc::fence_proxy_async_smem();
    __syncthreads();
    bool p_ok = true;
    if (tid == 0) {
        // rows AC_OWN dq .. of each half (hi, lo) of each 64-key slab to every other CTA,
        // completing on that CTA's pbar
        const uint32_t p0 = tc::smem_u32(S.p), pb = tc::smem_u32(&S.pbar);
#pragma unroll
        for (int dst = 0; dst < AC_CL; dst++) {
            if (dst == (int)dq) continue;
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {       // (slab, half) = (q4 >> 1, q4 & 1)
                const uint32_t off = (uint32_t)(q4 >> 1) * (2 * CSA2_HEADS * 128) +
                                     ((uint32_t)(q4 & 1) * CSA2_HEADS + AC_OWN * dq) * 128u;
                bulk_to_peer(cluster_map(p0 + off, (uint32_t)dst), p0 + off, AC_P_ROWS_BYTES,
                             cluster_map(pb, (uint32_t)dst));
            }
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        p_ok = tc::mbar_wait(&S.pbar, 0, polls);   // the other CTAs' rows have landed here
    }
    const bool p_fail = __syncthreads_or(!p_ok);
    tc::tc_fence_after();
    pdl_launch_dependents();                       // let the merge kernel be scheduled

    // ---- [O_hi | O_lo]_d^T = V_d^T [P_hi | P_lo]^T: M-tiles of 128 dims, K = 128 keys,
    //      N = 128; tile mt in columns 128 mt .. +127 (S has been read out)
    if (tid == 0 && !fail && !s_fail && !p_fail) {
        const uint32_t k0 = tc::smem_u32(S.k), p0 = tc::smem_u32(S.p);
#pragma unroll
        for (int mt = 0; mt < AC_MT; mt++) {
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {       // 16 keys per step
                const uint64_t ad = tc::smem_desc(k0 + (uint32_t)(2 * mt) * (AC_KEYS * 128) + (uint32_t)kk * 2048u,
                                                  AC_KEYS * 128, 1024, tc::kSwizzle128B);
                const uint32_t boff = (uint32_t)(kk >> 2) * (2 * CSA2_HEADS * 128) + (uint32_t)(kk & 3) * 32u;
                tc::mma_f16(tmem + 128u * (uint32_t)mt, ad, tc::smem_desc(p0 + boff, 16, 1024, tc::kSwizzle128B),
                            AC_IDESC_O, kk > 0);
            }
        }
        tc::mma_commit(&S.mbar);
    }
    if (early == 2) {
        pdl_wait();                                // the previous merge is done with its workspace
        if (tid < AC_OWN && !fail && !s_fail)
            *reinterpret_cast<float2 *>(part_ml + (base + AC_OWN * (int64_t)dq + tid) * 2) = S.mlv[tid];
    }
    if (p_fail && tid == 0) flag(c.status, CSA2_DEV_TIMEOUT);
    bool fail2 = false;
    if (!fail && !s_fail && !p_fail) {
        fail2 = __syncthreads_or(!tc::mbar_wait(&S.mbar, 1, polls));
        tc::tc_fence_after();
        if (!fail2) {
            // ---- partial output: M-tile mt, 32 heads per warp, lane = dim; hi + lo
            const int u = warp >> 2, mt = u >> 1, hh = u & 1;
            uint32_t ahi[32], alo[32];
            const uint32_t colo = 128u * (uint32_t)mt + 32u * (uint32_t)hh;
            tc::tmem_ld32(tmem + lane_base + colo, ahi);
            tc::tmem_ld32(tmem + lane_base + colo + 64u, alo);
            tc::tmem_ld_wait();
            float *po = part_o + (base + 32 * hh) * CSA2_HEAD_DIM + AC_DIMS * dq + 128 * mt + (warp & 3) * 32 + lane;
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
    // after a timeout, what is still in flight into this CTA's memory -- its own
    // products and the other CTAs' copies (every CTA sends both rounds on every
    // path) -- is awaited with a long limit before that memory is released
    if (tid == 0) {
        constexpr uint32_t kLong = 1u << 22;
        if (fail) tc::mbar_wait(&S.mbar, 0, kLong);
        if (fail2) tc::mbar_wait(&S.mbar, 1, kLong);
        if (s_fail) tc::mbar_wait(&S.sbar, 0, kLong);
        if (p_fail) tc::mbar_wait(&S.pbar, 0, kLong);
    }
    // the bulk copies out of this CTA's shared memory have finished reading it
    if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, AC_TMEM_COLS);
}

// o = sum_c e^(m_c - M) O_c / (sum_c e^(m_c - M) l_c + e^(z_h - M)), lse = M +
// log of that denominator (z_h the head's sink logit, -inf without one); one
// CTA per (row, 2 or 8 heads), thread = 4 consecutive dims (float4) of one head,
// all chunk loads in flight.  With rope_base > 0 the RoPE dims 448+i and
// 480+i of the output are rotated back by -t * rope_base^(-i/32) (angles
// reduced exactly in integer turns: t reaches 2^20).  Launched as a programmatic dependent of
// the attention kernel: it is scheduled early and waits for that grid here.
__global__ void __launch_bounds__(1024) k_attn_combine(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_ml, int nchunks,
                                                      const float *__restrict__ sink, int rope, RopeTurns turns,
                                                      const int64_t *__restrict__ q_pos,
                                                      float *__restrict__ o, float *__restrict__ lse)
{
    // the next kernel on the stream may be scheduled now; it waits for this grid
    pdl_launch_dependents();
    pdl_wait();
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x & 127;
    const int h = blockIdx.y * (int)(blockDim.x >> 7) + (threadIdx.x >> 7);   // 128 threads per head
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
    const float z = sink ? sink[h] : -INFINITY;
    if (z != -INFINITY) {
        if (M == -INFINITY || z > M) {              // the sink sets the reference maximum
            const float f = M == -INFINITY ? 0.0f : expf(M - z);
            L = fmaf(L, f, 1.0f);
            acc = make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
            M = z;
        } else {
            L += expf(z - M);
        }
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    float4 out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (rope && tid >= 96) {                        // the warp holding dims 384..511
        // dims 448+i (threads 112..119) pair with 480+i (threads 120..127), 8 lanes apart
        const float4 other = make_float4(__shfl_xor_sync(0xffffffffu, out.x, 8), __shfl_xor_sync(0xffffffffu, out.y, 8),
                                         __shfl_xor_sync(0xffffffffu, out.z, 8), __shfl_xor_sync(0xffffffffu, out.w, 8));
        if (tid >= 112) {
            const bool first = tid < 120;
            const int i0 = 4 * (tid - (first ? 112 : 120));
            const int64_t t = q_pos[r];
            float rot[4];
            const float mine[4] = {out.x, out.y, out.z, out.w}, oth[4] = {other.x, other.y, other.z, other.w};
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                float sn, cs;
                rope_sincos(t, turns.phi[i0 + c4], &sn, &cs);
                // (a, b) -> (a cos + b sin, -a sin + b cos); this thread holds a (first) or b
                rot[c4] = first ? fmaf(mine[c4], cs, oth[c4] * sn) : fmaf(mine[c4], cs, -oth[c4] * sn);
            }
            out = make_float4(rot[0], rot[1], rot[2], rot[3]);
        }
    }
    *reinterpret_cast<float4 *>(o + (r * CSA2_HEADS + h) * CSA2_HEAD_DIM + 4 * tid) = out;
    if (tid == 0) lse[r * CSA2_HEADS + h] = L > 0.0f ? M + logf(L) : -INFINITY;
}

size_t attn_workspace_bytes(int64_t rows)
{
    const size_t po = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4;
    const size_t ml = (size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * 2 * 4;
    return ((po + 255) & ~(size_t)255) + ml;
}

// Many rows: persistent clusters over whole rows (no merge, no partials).
bool attn_by_rows(int64_t rows, const csa2_swa &swa)
{
    if (swa.flags & CSA2_ATTN_SCHEDULE_ROWS) return true;
    if (swa.flags & CSA2_ATTN_SCHEDULE_CHUNKS) return false;
    return rows >= 40;
}

int launch_attn_rows(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale,
                     const int32_t *idx, int k, const csa2_swa &swa, float *o, float *lse, cudaStream_t st);

int launch_attn(const csa2_cache &c, const csa2_batch &bt, const uint16_t *q, float sm_scale, const int32_t *idx,
                int k, const csa2_swa &swa, float *o, float *lse, void *ws, size_t ws_bytes, cudaStream_t st,
                int early)
{
    const int64_t rows = (int64_t)bt.batch * bt.nq;
    if (rows == 0) return CSA2_OK;
    if (ws_bytes < attn_workspace_bytes(rows) || !ws) return CSA2_ERR_WORKSPACE;
    if (attn_by_rows(rows, swa)) return launch_attn_rows(c, bt, q, sm_scale, idx, k, swa, o, lse, st);
    const size_t po_bytes = ((size_t)rows * AC_MAX_CHUNKS * CSA2_HEADS * CSA2_HEAD_DIM * 4 + 255) & ~(size_t)255;
    float *part_o = static_cast<float *>(ws);
    float *part_ml = reinterpret_cast<float *>(static_cast<char *>(ws) + po_bytes);
    const int nchunks = (k + AC_KEYS - 1) / AC_KEYS + 1;
    const size_t smem = sizeof(AcSmem) + 1024;
    if (rows > 65535) return CSA2_ERR_SHAPE;       // rows run along the grid's y dimension
    if (const int s = kernel_smem_limit((const void *)k_attn_tc, smem, 100)) return s;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t ac = {};
        ac.gridDim = dim3((unsigned)(AC_CL * nchunks), (unsigned)rows);
        ac.blockDim = dim3(AC_THREADS);
        ac.dynamicSmemBytes = smem;
        ac.stream = st;
        ac.attrs = pdl;
        ac.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&ac, k_attn_tc, c, bt, q, sm_scale, idx, k, swa, part_o, part_ml,
                                                 nchunks, early, wait_polls());
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return CSA2_ERR_CUDA;
        }
    }
    int s = launch_status();
    if (s) return s;
    cudaLaunchConfig_t cfg = {};
    // decode (few rows): eight heads per CTA, few CTAs to schedule after the
    // wait; many rows: two heads per CTA, more CTAs resident per SM
    const int heads_per_cta = rows <= 256 ? 8 : 2;
    cfg.gridDim = dim3((unsigned)rows, CSA2_HEADS / heads_per_cta);
    cfg.blockDim = dim3(heads_per_cta * 128);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_attn_combine, (const float *)part_o, (const float *)part_ml,
                                             nchunks, swa.sink, swa.rope_base > 0.0f ? 1 : 0,
                                             rope_turns(swa.rope_base), bt.q_pos, o, lse);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace csa2
