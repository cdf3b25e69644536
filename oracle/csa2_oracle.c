/*
 * CPU oracle for the CSA2 (Compressed Sparse Attention 2) attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA kernels.
 *
 * Plain loops, double-precision accumulation, no blocking, no fusion.  Each
 * function cites the passage of the source pages it writes out:
 *   [P1] "DeepSeek-V4.1-Flash" research note (vibe-research.pages.dev)
 *   [P2] "DeepSeek-V4.1-Flash 架构详解：CED、CSA2 与 890 字节 KV Cache" (gentlecold.top)
 *   [P3] DeepSeek-V4 report explainer (mlqm.cn)
 * plus the OCP Microscaling (MX) and OCP FP8 format definitions, which the
 * pages name ("OCP MXFP4", "E2M1", "FP8") but do not spell out.
 *
 * Where the pages leave a choice open this file takes the reading listed in
 * the design notes (scale of the MX block, sign of zero, tie-breaking, ...).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math: the
 * two fp32 operations of the FP8 quantiser must be single IEEE roundings).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> exact value. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E2M1 (OCP FP4) code -> value.  Bit 3 sign, bits 2:1 exponent (bias 1),
 * bit 0 mantissa; exponent field 0 is subnormal (0 or 0.5).
 * [P2] §4: main KV is stored as MXFP4 with E2M1 elements. */
double or_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int mbit = code & 1;
    double mag = (e == 0) ? 0.5 * mbit : ldexp(1.0 + 0.5 * mbit, e - 1);
    return sign ? -mag : mag;
}

/* Round a scaled value to the nearest E2M1 magnitude, ties to the code with
 * an even mantissa bit, magnitudes beyond the largest value (6) saturating to
 * it; the sign bit copies the sign of the input (so -0.1 -> 0x8). */
uint8_t or_e2m1_encode(double v)
{
    double a = fabs(v);
    if (a > 6.0)                        /* saturation: beyond 6 every distance is */
        a = 6.0;                        /* the same in double precision for huge a */
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 8; c++) {
        double d = fabs(a - or_e2m1_value((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 8 : 0));
}

/* E4M3 (OCP FP8, "fn" variant: no infinities, S.1111.111 is NaN) -> value. */
double or_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int man = code & 7;
    if (e == 15 && man == 7)
        return NAN;
    double mag = (e == 0) ? ldexp(man / 8.0, -6) : ldexp(1.0 + man / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round to the nearest E4M3 value, ties to even (code LSB 0), saturating to
 * the largest finite value 448; the sign bit copies the input's sign.  The
 * positive codes 0..126 are increasing in value, so a binary search finds the
 * two neighbours. */
uint8_t or_e4m3_encode(float x)
{
    double a = fabs((double)x);
    int lo = 0, hi = 126;               /* largest code with value <= a */
    if (a >= or_e4m3_value(126)) {
        lo = 126;
    } else {
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (or_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
        }
    }
    int c = lo;
    if (lo < 126) {
        double dlo = a - or_e4m3_value((uint8_t)lo);
        double dhi = or_e4m3_value((uint8_t)(lo + 1)) - a;
        if (dhi < dlo || (dhi == dlo && ((lo + 1) & 1) == 0))
            c = lo + 1;
    }
    return (uint8_t)(c | (signbit(x) ? 0x80 : 0));
}

/* ------------------------------------------------------------------------ */
/* MXFP4 quantisation of main-KV entries                                    */
/* ------------------------------------------------------------------------ */

/* OCP MX shared scale of one 32-element block: X = floor(log2(amax)) - 2,
 * 2 being the largest exponent of E2M1 (6 = 1.5 * 2^2); stored as the E8M0
 * byte X + 127, X clamped to [-127, 127].  amax == 0 gives X = 0.
 * [P2] §4 ("OCP MXFP4 ... no global scale"); block 32 / E8M0 per the OCP MX
 * definition of MXFP4. */
int or_mx_exponent(float amax)
{
    if (amax == 0.0f)
        return 0;
    int e;
    frexp((double)amax, &e);            /* amax = f * 2^e, f in [0.5, 1) */
    int x = (e - 1) - 2;
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

/* Quantise n entries of 512 fp32 values.  codes: [n][256] bytes, element 2i
 * in the low nibble of byte i, 2i+1 in the high nibble; scales: [n][16] E8M0. */
void or_quant_mxfp4(const float *x, int64_t n, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        const float *row = x + r * 512;
        for (int b = 0; b < 16; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = fabsf(row[b * 32 + i]);
                if (a > amax) amax = a;
            }
            int X = or_mx_exponent(amax);
            scales[r * 16 + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; i += 2) {
                uint8_t c0 = or_e2m1_encode(ldexp((double)row[b * 32 + i], -X));
                uint8_t c1 = or_e2m1_encode(ldexp((double)row[b * 32 + i + 1], -X));
                codes[r * 256 + (b * 32 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}

/* Exact decode of n MXFP4 entries to doubles [n][512]. */
void or_dequant_mxfp4(const uint8_t *codes, const uint8_t *scales, int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++)
        for (int d = 0; d < 512; d++) {
            uint8_t byte = codes[r * 256 + d / 2];
            uint8_t c = (d & 1) ? (byte >> 4) : (byte & 15);
            int X = (int)scales[r * 16 + d / 32] - 127;
            out[r * 512 + d] = ldexp(or_e2m1_value(c), X);
        }
}

/* FP4 main KV with one E4M3 scale per 16 elements: the block size and scale
 * type that [P2] §4 and [P4] give for the FP4 cache ("16 channels share one
 * E4M3 scale").  For a block with largest magnitude amax:
 *   s  = e4m3(amax / 6)      one fp32 IEEE division, then the FP8 rounding
 *                            (to nearest, ties to even, saturating at 448);
 *   c_i = e2m1(x_i / s)      one fp32 IEEE division, then the E2M1 rounding
 *                            (to nearest, ties to the even code, saturating
 *                            at 6, sign bit kept);
 * a block whose scale rounds to zero keeps only the elements' sign bits.
 * codes: [n][256] in the MXFP4 nibble order; scales: [n][32] E4M3 bytes. */
void or_quant_fp4_e4m3(const float *x, int64_t n, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        const float *row = x + r * 512;
        for (int b = 0; b < 32; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 16; i++) {
                float a = fabsf(row[b * 16 + i]);
                if (a > amax) amax = a;
            }
            volatile float q = amax / 6.0f;           /* one fp32 rounding */
            uint8_t sb = or_e4m3_encode(q);
            scales[r * 32 + b] = sb;
            float sv = (float)or_e4m3_value(sb);
            for (int i = 0; i < 16; i += 2) {
                uint8_t c[2];
                for (int t = 0; t < 2; t++) {
                    float v = row[b * 16 + i + t];
                    if (sv == 0.0f) {
                        c[t] = (uint8_t)(signbit(v) ? 8 : 0);
                    } else {
                        volatile float y = v / sv;    /* one fp32 rounding */
                        c[t] = or_e2m1_encode((double)y);
                    }
                }
                codes[r * 256 + (b * 16 + i) / 2] = (uint8_t)(c[0] | (c[1] << 4));
            }
        }
    }
}

/* Exact decode of n entries of that format to doubles [n][512]. */
void or_dequant_fp4_e4m3(const uint8_t *codes, const uint8_t *scales, int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++)
        for (int d = 0; d < 512; d++) {
            uint8_t byte = codes[r * 256 + d / 2];
            uint8_t c = (d & 1) ? (byte >> 4) : (byte & 15);
            out[r * 512 + d] = or_e2m1_value(c) * or_e4m3_value(scales[r * 32 + d / 16]);
        }
}

/* ------------------------------------------------------------------------ */
/* FP8 quantisation with a per-row fp32 scale (SWA KV, indexer keys)        */
/* ------------------------------------------------------------------------ */

/* s = amax / 448 (one fp32 IEEE division; amax == 0 gives s = 1), then each
 * element code = e4m3(x / s) with x / s one fp32 IEEE division.
 * [P1] §3.3 / [P2] §4: SWA KV stays FP8; per-token fp32 scale is the
 * stated reading for both the SWA rows and the indexer keys. */
void or_quant_fp8(const float *x, int64_t n, int dim, uint8_t *codes, float *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        const float *row = x + r * dim;
        float amax = 0.0f;
        for (int i = 0; i < dim; i++) {
            float a = fabsf(row[i]);
            if (a > amax) amax = a;
        }
        volatile float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scales[r] = s;
        for (int i = 0; i < dim; i++) {
            volatile float y = row[i] / s;
            codes[r * dim + i] = or_e4m3_encode(y);
        }
    }
}

void or_dequant_fp8(const uint8_t *codes, const float *scales, int64_t n, int dim, double *out)
{
    for (int64_t r = 0; r < n; r++)
        for (int i = 0; i < dim; i++)
            out[r * dim + i] = or_e4m3_value(codes[r * dim + i]) * (double)scales[r];
}

/* ------------------------------------------------------------------------ */
/* CSA compressor                                                            */
/* ------------------------------------------------------------------------ */

/* e_j[d] = sum_i softmax_i(Z_{jm+i}[d] + B_i[d]) * C_{jm+i}[d], i < m.
 * [P3] §3.1: m consecutive tokens fold into one entry through softmax
 * weights from content scores plus a learned bias; [P2] §2: C and Z are the
 * per-layer KV and score projections; [P2] §3.1: m = 2 encoder, 1 decoder.
 * C, Z: [n_tok][512] bf16 patterns; bias: [m][512]; out: [n_tok/m][512]. */
void or_compress(const uint16_t *C, const uint16_t *Z, const float *bias, int m,
                 int64_t n_tok, float *out)
{
    int64_t n_ent = n_tok / m;
    for (int64_t j = 0; j < n_ent; j++)
        for (int d = 0; d < 512; d++) {
            double zmax = -INFINITY;
            for (int i = 0; i < m; i++) {
                double z = bf16_value(Z[(j * m + i) * 512 + d]) + (double)bias[i * 512 + d];
                if (z > zmax) zmax = z;
            }
            double den = 0.0, num = 0.0;
            for (int i = 0; i < m; i++) {
                double z = bf16_value(Z[(j * m + i) * 512 + d]) + (double)bias[i * 512 + d];
                double p = exp(z - zmax);
                den += p;
                num += p * bf16_value(C[(j * m + i) * 512 + d]);
            }
            out[j * 512 + d] = (float)(num / den);
        }
}

/* ------------------------------------------------------------------------ */
/* lightning-indexer score                                                   */
/* ------------------------------------------------------------------------ */

/* score = sum_h w_h * ReLU(q_h . k), k = e4m3(code) * scale, 32 heads x 128.
 * [P3] §3.2 (query projected to a low dimension, matched against the
 * compressed index keys); [P2] §1 table (32 indexer heads, dim 128); the
 * ReLU-weighted head sum is the stated reading. */
double or_index_score(const uint16_t *qi, const float *w, const uint8_t *code, float scale)
{
    double k[128];
    for (int d = 0; d < 128; d++)
        k[d] = or_e4m3_value(code[d]) * (double)scale;      /* dequantised key */
    double s = 0.0;
    for (int h = 0; h < 32; h++) {
        double dot = 0.0;
        for (int d = 0; d < 128; d++)
            dot += bf16_value(qi[h * 128 + d]) * k[d];
        s += (double)w[h] * (dot > 0.0 ? dot : 0.0);
    }
    return s;
}

/* Scores of entries pos[0..n) (rows of codes/scales addressed by position). */
void or_index_scores(const uint16_t *qi, const float *w, const uint8_t *codes,
                     const float *scales, const int32_t *pos, int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        int64_t p = pos ? pos[i] : i;
        out[i] = or_index_score(qi, w, codes + p * 128, scales[p]);
    }
}

/* ------------------------------------------------------------------------ */
/* selection                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    double score;
    int64_t pos;
} or_item;

/* higher score first; equal scores: lower position first */
static int or_item_cmp(const void *pa, const void *pb)
{
    const or_item *a = (const or_item *)pa, *b = (const or_item *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->pos > b->pos) - (a->pos < b->pos);
}

static int or_i32_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Top-k positions among candidates (score[i], pos[i]) ordered by score
 * descending then position ascending; the chosen positions are written in
 * ascending order, the rest of out[0..k) is -1.  Returns the count chosen. */
int or_topk(const double *score, const int32_t *pos, int64_t n, int k, int32_t *out)
{
    or_item *it = (or_item *)malloc(sizeof(or_item) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; i++) {
        it[i].score = score[i];
        it[i].pos = pos ? pos[i] : i;
    }
    qsort(it, (size_t)n, sizeof(or_item), or_item_cmp);
    int kk = (int)(n < k ? n : k);
    for (int i = 0; i < kk; i++) out[i] = (int32_t)it[i].pos;
    qsort(out, (size_t)kk, sizeof(int32_t), or_i32_cmp);
    for (int i = kk; i < k; i++) out[i] = -1;
    free(it);
    return kk;
}

/* Hierarchical candidate pool of a Full layer.  block b covers positions
 * [blk*b, blk*b+blk) of the n visible ones; its score is the maximum over
 * those positions; the top pmax blocks (score descending, index ascending)
 * are kept and all their visible positions form the pool, ascending.
 * [P1] §3.2 and [P2] §3.2: the Full layer aggregates index scores per block
 * of 8 and keeps at most 2,048 blocks, i.e. at most 16,384 candidates.
 * Returns the pool size. */
int64_t or_block_pool(const double *score, int64_t n, int blk, int pmax, int32_t *pool)
{
    int64_t nb = (n + blk - 1) / blk;
    or_item *it = (or_item *)malloc(sizeof(or_item) * (size_t)(nb > 0 ? nb : 1));
    for (int64_t b = 0; b < nb; b++) {
        double mx = -INFINITY;
        for (int64_t p = b * blk; p < n && p < (b + 1) * blk; p++)
            if (score[p] > mx) mx = score[p];
        it[b].score = mx;
        it[b].pos = b;
    }
    qsort(it, (size_t)nb, sizeof(or_item), or_item_cmp);
    int64_t keep = nb < pmax ? nb : pmax;
    int32_t *blocks = (int32_t *)malloc(sizeof(int32_t) * (size_t)(keep > 0 ? keep : 1));
    for (int64_t i = 0; i < keep; i++) blocks[i] = (int32_t)it[i].pos;
    qsort(blocks, (size_t)keep, sizeof(int32_t), or_i32_cmp);
    int64_t np = 0;
    for (int64_t i = 0; i < keep; i++)
        for (int64_t p = (int64_t)blocks[i] * blk; p < n && p < ((int64_t)blocks[i] + 1) * blk; p++)
            pool[np++] = (int32_t)p;
    free(blocks);
    free(it);
    return np;
}

/* ------------------------------------------------------------------------ */
/* sparse MQA attention over selected entries plus the SWA window            */
/* ------------------------------------------------------------------------ */

/* One query: 64 heads x 512 dims against nk keys shared by all heads, each
 * key serving as its own value.  logits l[h][j] = sm_scale * q_h . k_j;
 * o_h = sum_j softmax_j(l[h]) k_j; lse_h = log sum_j exp(l[h][j]).
 * nk == 0 gives o = 0 and lse = -inf.
 * [P2] §1 table (64 query heads x 512, top-k 512, SWA 128); [P3] §3.3 (the
 * window branch beside the compressed branch) and §4.3 (the compressed
 * entry serves as both key and value); one softmax over both branches.
 *
 * Options around it ([P3] §4.3 names a learnable attention sink and partial
 * RoPE on the last 64 dims with the output rotated back):
 *  - sink (NULL for none): per head a logit z_h that joins the softmax's
 *    denominator without a value: o_h = sum_j e^l_j k_j / (e^z_h + sum_j e^l_j),
 *    lse_h = log(e^z_h + sum_j e^l_j); z_h = -inf is no sink;
 *  - rope_base > 0: the output's dims 448 + i and 480 + i (i < 32) are rotated
 *    by -t * rope_base^(-i/32), t the query's token position:
 *    (a, b) -> (a cos + b sin, -a sin + b cos). */
void or_attention(const uint16_t *q, double sm_scale, const double *keys, int64_t nk,
                  const double *sink, double rope_base, int64_t t, float *o, float *lse)
{
#pragma omp parallel for schedule(static)
    for (int h = 0; h < 64; h++) {
        const double z = sink ? sink[h] : -INFINITY;
        double *l = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        double mx = z;
        for (int64_t j = 0; j < nk; j++) {
            double dot = 0.0;
            for (int d = 0; d < 512; d++)
                dot += bf16_value(q[h * 512 + d]) * keys[j * 512 + d];
            l[j] = sm_scale * dot;
            if (l[j] > mx) mx = l[j];
        }
        double out[512];
        if (mx == -INFINITY) {               /* no key and no sink */
            for (int d = 0; d < 512; d++) out[d] = 0.0;
            lse[h] = -INFINITY;
        } else {
            double den = (z == -INFINITY) ? 0.0 : exp(z - mx);
            for (int64_t j = 0; j < nk; j++) den += exp(l[j] - mx);
            for (int d = 0; d < 512; d++) {
                double acc = 0.0;
                for (int64_t j = 0; j < nk; j++) acc += exp(l[j] - mx) * keys[j * 512 + d];
                out[d] = acc / den;
            }
            lse[h] = (float)(mx + log(den));
        }
        if (rope_base > 0.0) {
            for (int i = 0; i < 32; i++) {
                const double th = (double)t * pow(rope_base, -(double)i / 32.0);
                const double c = cos(th), sn = sin(th);
                const double a = out[448 + i], b = out[480 + i];
                out[448 + i] = a * c + b * sn;
                out[480 + i] = -a * sn + b * c;
            }
        }
        for (int d = 0; d < 512; d++) o[h * 512 + d] = (float)out[d];
        free(l);
    }
}

/* RMSNorm and forward partial RoPE of nvec 512-dim vectors, vecs of them per
 * row sharing the row's token position pos[row] ([P3] §4.3: queries and
 * compressed KV are RMS-normalised before the core attention; RoPE acts on the
 * last 64 dims only):
 *   y_d = x_d / sqrt((1/512) sum_e x_e^2 + eps) * gamma_d   (gamma NULL: 1);
 *   rope_base > 0: for i < 32 the pair (y[448 + i], y[480 + i]) turns by the
 *   angle +t * rope_base^(-i/32), t = pos[row]:
 *     (a, b) -> (a cos - b sin, a sin + b cos),
 *   the inverse of the output rotation in or_attention. */
void or_norm_rope(const double *x, int64_t nvec, int vecs, const double *gamma, double eps,
                  const int64_t *pos, double rope_base, double *out)
{
    for (int64_t v = 0; v < nvec; v++) {
        const double *xv = x + v * 512;
        double *y = out + v * 512;
        double ms = 0.0;
        for (int d = 0; d < 512; d++) ms += xv[d] * xv[d];
        ms /= 512.0;
        const double rms = sqrt(ms + eps);
        for (int d = 0; d < 512; d++) y[d] = xv[d] / rms * (gamma ? gamma[d] : 1.0);
        if (rope_base > 0.0) {
            const double t = (double)pos[v / vecs];
            for (int i = 0; i < 32; i++) {
                const double th = t * pow(rope_base, -(double)i / 32.0);
                const double c = cos(th), sn = sin(th);
                const double a = y[448 + i], b = y[480 + i];
                y[448 + i] = a * c - b * sn;
                y[480 + i] = a * sn + b * c;
            }
        }
    }
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
