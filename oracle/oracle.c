/*
 * oracle.c -- plain, slow, single-threaded CPU restatement of the decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file.  It exists so that tests/, the smoke check and the bench's CPU
 * baseline can compare the CUDA library against an implementation that a reader
 * can check against the source pages by eye.  It shares no code, header, table or
 * constant with weight_streaming_warp_gb300/csrc: it has its own IEEE-754 half
 * conversion, its own bf16 decode and its own loops.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "vulkan : dequant q8_0 KV once in coopmat1" (llama.cpp PR), Overview and
 *        the discussion of the tensor strides ne = [128, 256, 4], nb = [2, 1024, 256]
 *        and the per-head-contiguous scratch.
 *   [P2] "ggml-cuda: pad matmul weight rows to avoid cache-set aliasing", Overview
 *        (row stride nb[1] larger than the packed row; pad bytes are never read as
 *        data) and Tuning.
 *   [P3] "QuantizeQ8KK is thread-per-superblock: 95.5us/call ...", Cause (the amax
 *        scan over one 256-element superblock) and Scope (quantize, then the
 *        quantized mat-vec; the MoE path quantizes m = T x top_k rows).
 *   [P4] "perf(vulkan): decode GEMV reads four elements per load, and the row lever
 *        is dead", opening paragraph (y = W.x over bf16 weights streamed once per
 *        token) and "What did NOT work" (results must not depend on rows per
 *        workgroup).
 *   [P5] "cuda: prefetch the next PTQ1_0 mat-vec's weights into L2 from the last
 *        CTAs", Overview (a chain of dependent mat-vecs; values never change).
 *
 * The q8_0 rule used throughout: a block of B consecutive values (B = 32 for q8_0,
 * B = 256 for the superblock) gets amax = max |x|, d = amax / 127 and
 * q = round(x / d).  Readings where the pages are silent:
 *   - "round" is round-half-away-from-zero (C roundf);
 *   - x / d divides by the fp32 d (the stored fp16 copy of d is only storage);
 *   - both divisions are IEEE fp32 divisions (no reciprocal multiply);
 *   - an all-zero block stores d = +0 and q = 0, and so does a block whose
 *     d = amax / 127 rounds to +0 (amax of a few subnormal steps);
 *   - q is clamped to [-127, 127] (a no-op for finite inputs);
 *   - the superblock keeps an fp32 positive scale from amax; the signed "mx" value
 *     that the [P3] excerpt also tracks is not used by any result here;
 *   - non-finite inputs are outside the contract.
 * Mat-vec results are returned in fp64.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fPIC -shared (see oracle/build.py).
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * IEEE-754 binary16 / bfloat16 helpers, written from the format definitions.
 * ------------------------------------------------------------------------- */

/* binary32 -> binary16, round to nearest, ties to even, with subnormals and
 * overflow to infinity.  NaN stays NaN (quiet). */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t bexp = (u >> 23) & 0xffu;
    uint32_t man = u & 0x7fffffu;
    if (bexp == 0xffu) /* inf or nan */
        return (uint16_t)(sign | 0x7c00u | (man ? 0x0200u : 0u));
    if (bexp == 0u) /* binary32 zero or subnormal: far below half's range */
        return (uint16_t)sign;
    int e = (int)bexp - 127;         /* value = 1.man * 2^e */
    uint32_t sig = man | 0x800000u;  /* 24-bit significand, value = sig * 2^(e-23) */
    if (e >= -14) {
        /* normal half candidate: keep 11 significant bits */
        uint32_t keep = sig >> 13;
        uint32_t rem = sig & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (keep & 1u)))
            keep++;
        int he = e + 15;
        if (keep == 0x800u) { /* rounding carried into a new binade */
            keep = 0x400u;
            he++;
        }
        if (he >= 31)
            return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | ((uint32_t)he << 10) | (keep & 0x3ffu));
    }
    /* half subnormal: value in units of 2^-24 is sig * 2^(e+1) */
    int shift = -(e + 1); /* >= 14 */
    if (shift > 24)
        return (uint16_t)sign; /* below half of the smallest subnormal */
    uint32_t keep = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (keep & 1u)))
        keep++;
    /* keep == 0x400 encodes the smallest normal, which is the right answer */
    return (uint16_t)(sign | keep);
}

/* binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t he = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t man = (uint32_t)h & 0x3ffu;
    float mag;
    if (he == 0u) {
        mag = ldexpf((float)man, -24);
    } else if (he == 31u) {
        uint32_t u = 0x7f800000u | (man << 13);
        memcpy(&mag, &u, 4);
    } else {
        mag = ldexpf((float)(man | 0x400u), (int)he - 25);
    }
    uint32_t u;
    memcpy(&u, &mag, 4);
    u |= sign;
    memcpy(&mag, &u, 4);
    return mag;
}

/* bfloat16 -> double (exact: bf16 is the top half of a binary32). */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * quantize_q8  ([P3] Cause and Scope; the q8_0 rule above)
 *
 * x: fp32, `rows` rows of `n` values, row stride ldx (elements).
 * q: int8 [rows][n], packed.
 * scales: block 32 -> binary16 bit patterns [rows][n/32];
 *         block 256 -> fp32 [rows][n/256].
 * Returns 0, or -1 for arguments outside the contract.
 * ------------------------------------------------------------------------- */
int orc_quantize_q8(const float *x, int64_t rows, int64_t n, int64_t ldx, int block,
                    int8_t *q, void *scales)
{
    if (block != 32 && block != 256)
        return -1;
    if (rows < 0 || n < 0 || n % block != 0 || ldx < n)
        return -1;
    int64_t nb = n / block;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + r * ldx + b * block;
            int8_t *qb = q + r * n + b * block;
            /* one pass, one load per element: amax = max |x| (exact in fp32) */
            float amax = 0.0f;
            for (int i = 0; i < block; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f; /* IEEE fp32 division */
            for (int i = 0; i < block; ++i) {
                int v = 0;
                /* d == 0: an all-zero block, or one whose amax is so small (at most
                 * 63.5 binary32 subnormal steps) that amax / 127 rounds to +0; x / d
                 * is then undefined and the block is stored as zero. */
                if (d != 0.0f) {
                    float t = roundf(xb[i] / d); /* fp32 division, half away from zero */
                    if (t > 127.0f)
                        t = 127.0f;
                    if (t < -127.0f)
                        t = -127.0f;
                    v = (int)t;
                }
                qb[i] = (int8_t)v;
            }
            if (block == 32)
                ((uint16_t *)scales)[r * nb + b] = orc_f32_to_f16(d);
            else
                ((float *)scales)[r * nb + b] = d;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * gemv_bf16  ([P4] opening paragraph; [P2] Overview for the row stride)
 *
 * y[r] = alpha * sum_k W[r*ld + k] * x[k], evaluated in fp64.
 * W: bf16 bit patterns, M rows of K values, row stride ld >= K (the elements
 * between K and ld are padding and are never read).
 * x: fp64 [K] (an fp32 activation converts to fp64 exactly).
 * ------------------------------------------------------------------------- */
void orc_gemv_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const double *x,
                   double alpha, double *y)
{
    for (int64_t r = 0; r < M; ++r) {
        const uint16_t *w = W + r * ld;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += bf16_to_f64(w[k]) * x[k];
        y[r] = alpha * acc;
    }
}

/* ---------------------------------------------------------------------------
 * gemv_q8_0  ([P3] Scope: the quantized mat-vec that follows the quantizer)
 *
 * y[r] = sum_b Wd[r][b] * xd[b] * (sum_{i<32} Wq[r][32b+i] * xq[32b+i]), fp64.
 * Wq: int8, M rows, row stride ldq (elements, multiple of 32);
 * Wd: binary16 [M][K/32] packed; xq: int8 [K]; xd: binary16 [K/32].
 * The integer block sum is exact; Wd*xd*isum is exact in fp64 (22 + 19 bits);
 * only the sum over blocks rounds.
 * ------------------------------------------------------------------------- */
void orc_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t M, int64_t K, int64_t ldq,
                   const int8_t *xq, const uint16_t *xd, double *y)
{
    int64_t nb = K / 32;
    for (int64_t r = 0; r < M; ++r) {
        double acc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            int64_t isum = 0;
            for (int i = 0; i < 32; ++i)
                isum += (int64_t)Wq[r * ldq + 32 * b + i] * (int64_t)xq[32 * b + i];
            double dw = (double)orc_f16_to_f32(Wd[r * nb + b]);
            double dx = (double)orc_f16_to_f32(xd[b]);
            acc += dw * dx * (double)isum;
        }
        y[r] = acc;
    }
}

/* ---------------------------------------------------------------------------
 * moe_gemv_q8_0  ([P3] Cause/Scope: the grouped MoE path quantizes m = T x top_k
 * rows and multiplies each row by its expert's weights)
 *
 * For each row m: y[m][:] = gemv_q8_0(W_{ids[m]}, x_m).
 * Wq: int8 [E][Mo][K]; Wd: binary16 [E][Mo][K/32]; xq: int8 [R][K];
 * xd: binary16 [R][K/32]; ids: int32 [R]; y: fp64 [R][Mo].
 * A row whose id lies outside [0, E) is skipped (its y row is left untouched);
 * the return value counts such rows.
 * ------------------------------------------------------------------------- */
int64_t orc_moe_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                          const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                          double *y)
{
    int64_t bad = 0;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < R; ++m) {
        int32_t e = ids[m];
        if (e < 0 || (int64_t)e >= E) {
            bad++;
            continue;
        }
        orc_gemv_q8_0(Wq + (int64_t)e * Mo * K, Wd + (int64_t)e * Mo * nb, Mo, K, K,
                      xq + m * K, xd + m * nb, y + m * Mo);
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * gemm_bf16  ([P2] Results: small-batch prefill, where a short run of output rows
 * streams the whole weight matrix; the row stride may carry one extra cache line)
 *
 * Y[n][r] = sum_k W[r*ld + k] * X[n*ldx + k], fp64.  Y row stride = M.
 * ------------------------------------------------------------------------- */
void orc_gemm_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const uint16_t *X,
                   int64_t N, int64_t ldx, double *Y)
{
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t r = 0; r < M; ++r) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(W[r * ld + k]) * bf16_to_f64(X[n * ldx + k]);
            Y[n * M + r] = acc;
        }
    }
}

/* ---------------------------------------------------------------------------
 * dequant_q8_0_kv  ([P1] Overview and the stride discussion)
 *
 * Input cache, position-major with the heads interleaved (the page's
 * ne = [head_dim, KV, n_head_kv] walk with nb[1] = head_dim * n_head_kv * elem):
 *   q: int8 [depth][heads][head_dim]; d: binary16 [depth][heads][head_dim/32].
 * Output, per-head contiguous: out[h][p][i] = f16_rn(f32(d) * f32(q)).
 * The fp32 product is exact (11 x 8 significant bits); one rounding to half.
 * ------------------------------------------------------------------------- */
void orc_dequant_q8_0_kv(const int8_t *q, const uint16_t *d, int64_t depth, int64_t heads,
                         int64_t head_dim, uint16_t *out)
{
    int64_t nb = head_dim / 32;
    for (int64_t h = 0; h < heads; ++h) {
        for (int64_t p = 0; p < depth; ++p) {
            for (int64_t i = 0; i < head_dim; ++i) {
                float s = orc_f16_to_f32(d[(p * heads + h) * nb + i / 32]);
                float v = (float)q[(p * heads + h) * head_dim + i];
                out[(h * depth + p) * head_dim + i] = orc_f32_to_f16(s * v);
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * attn_decode  ([P1] Overview: the flash-attention pass reads the dequantized
 * binary16 K and V of every cached position; the stride discussion gives the two
 * layouts it can read them in)
 *
 * One decoding step of scaled dot-product attention over `depth` cached positions,
 * for `heads` KV heads with `group` query heads each (grouped-query attention):
 *   s_p          = scale * sum_i q[h][g][i] * K(h, p)[i]
 *   out[h][g][i] = sum_p exp(s_p - m) * V(h, p)[i] / sum_p exp(s_p - m),
 *                  m = max_p s_p
 * (subtracting m changes nothing mathematically; it keeps exp finite).  K(h, p) is
 * the binary16 row that starts k_head_stride * h + k_pos_stride * p elements into k:
 * the per-head-contiguous scratch has (k_pos_stride, k_head_stride) =
 * (head_dim, depth * head_dim), the position-major cache (head_dim * heads,
 * head_dim).  V likewise.  q is fp32 [heads][group][head_dim]; out is fp64
 * [heads][group][head_dim].  All arithmetic in fp64, exp from libm.
 * ------------------------------------------------------------------------- */
void orc_attn_decode(const float *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                     int64_t heads, int64_t group, int64_t head_dim, int64_t k_pos_stride,
                     int64_t k_head_stride, int64_t v_pos_stride, int64_t v_head_stride,
                     double scale, double *out)
{
    double *s = (double *)malloc((size_t)(depth > 0 ? depth : 1) * sizeof(double));
    for (int64_t h = 0; h < heads; ++h) {
        for (int64_t g = 0; g < group; ++g) {
            const float *qv = q + (h * group + g) * head_dim;
            double *o = out + (h * group + g) * head_dim;
            double m = -HUGE_VAL;
            for (int64_t p = 0; p < depth; ++p) {
                const uint16_t *kr = k + h * k_head_stride + p * k_pos_stride;
                double dot = 0.0;
                for (int64_t i = 0; i < head_dim; ++i)
                    dot += (double)qv[i] * (double)orc_f16_to_f32(kr[i]);
                s[p] = scale * dot;
                if (s[p] > m) m = s[p];
            }
            double den = 0.0;
            for (int64_t i = 0; i < head_dim; ++i) o[i] = 0.0;
            for (int64_t p = 0; p < depth; ++p) {
                const uint16_t *vr = v + h * v_head_stride + p * v_pos_stride;
                double w = exp(s[p] - m);
                den += w;
                for (int64_t i = 0; i < head_dim; ++i) o[i] += w * (double)orc_f16_to_f32(vr[i]);
            }
            for (int64_t i = 0; i < head_dim; ++i) o[i] /= den;
        }
    }
    free(s);
}

/* ---------------------------------------------------------------------------
 * attn_prefill  ([P1] Overview: the prefill flash-attention pass, pp512, reads the
 * binary16 K and V of one layer; the stride discussion gives the two layouts)
 *
 * A batch of nq query positions at the end of a cache of `depth` positions: query i
 * (0 <= i < nq) sits at position depth - nq + i and attends to positions
 * 0 .. depth - nq + i (causal; the batch's own keys are the last nq positions).
 *   s_p          = scale * sum_d q[h][g][i][d] * K(h, p)[d]
 *   out[h][g][i] = sum_p exp(s_p - m) V(h, p) / sum_p exp(s_p - m),  m = max_p s_p
 * in fp64 over the visible positions.  q is binary16 [heads][group][nq][head_dim];
 * K(h, p) is the row of head_dim binary16 values at k + h * k_head_stride +
 * p * k_pos_stride (elements), V likewise; out is fp64 [heads][group][nq][head_dim].
 * Returns 0, or -1 for arguments outside the contract (nq < 1 or nq > depth).
 * ------------------------------------------------------------------------- */
int orc_attn_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                     int64_t heads, int64_t group, int64_t nq, int64_t head_dim,
                     int64_t k_pos_stride, int64_t k_head_stride, int64_t v_pos_stride,
                     int64_t v_head_stride, double scale, double *out)
{
    if (nq < 1 || nq > depth || heads < 0 || group < 1 || head_dim < 1)
        return -1;
    double *s = (double *)malloc((size_t)depth * sizeof(double));
    double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
    for (int64_t h = 0; h < heads; ++h) {
        for (int64_t g = 0; g < group; ++g) {
            for (int64_t i = 0; i < nq; ++i) {
                const uint16_t *qv = q + ((h * group + g) * nq + i) * head_dim;
                double *o = out + ((h * group + g) * nq + i) * head_dim;
                const int64_t visible = depth - nq + i + 1; /* positions 0 .. depth - nq + i */
                for (int64_t d = 0; d < head_dim; ++d)
                    qd[d] = (double)orc_f16_to_f32(qv[d]);
                double m = -HUGE_VAL;
                for (int64_t p = 0; p < visible; ++p) {
                    const uint16_t *kr = k + h * k_head_stride + p * k_pos_stride;
                    double dot = 0.0;
                    for (int64_t d = 0; d < head_dim; ++d)
                        dot += qd[d] * (double)orc_f16_to_f32(kr[d]);
                    s[p] = scale * dot;
                    if (s[p] > m)
                        m = s[p];
                }
                double den = 0.0;
                for (int64_t d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                for (int64_t p = 0; p < visible; ++p) {
                    const uint16_t *vr = v + h * v_head_stride + p * v_pos_stride;
                    double w = exp(s[p] - m);
                    den += w;
                    for (int64_t d = 0; d < head_dim; ++d)
                        o[d] += w * (double)orc_f16_to_f32(vr[d]);
                }
                for (int64_t d = 0; d < head_dim; ++d)
                    o[d] /= den;
            }
        }
    }
    free(qd);
    free(s);
    return 0;
}

