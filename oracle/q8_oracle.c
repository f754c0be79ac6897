/*
 * q8_oracle.c -- plain, slow, obviously-correct CPU oracle for the int8
 * quantized projection path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  It shares no source,
 * header, constant or table with the CUDA path, and the CUDA path never calls
 * it.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -fPIC -shared
 * (no SIMD intrinsics; OpenMP only splits independent outputs across cores,
 * it never reorders the arithmetic of one output).
 *
 * Sources (web pages; cited by title and section):
 *   [L05]  "Part 4 - Lecture 05 - Fusion and the Activation-Quantization
 *          Discipline" (jared-hpc.com): sec. 2.1 (the 34-byte BlockQ8_0:
 *          f16 scale, then 32 int8), sec. 2.2 (int8 dot products).
 *   [R51]  "54 - r51 - producer-fused A-quantize mode 1" (yusiwen.cn/minfer):
 *          sec. 2.1 (q8_0 activation block: f16 d = amax/127, int8 q, int16
 *          ssum = sum of q, d and ssum packed in 4 bytes), sec. 3.1 (padded
 *          token rows are zero-filled), sec. 3.2 (rms_norm_quant_f32_t:
 *          ss -> rsqrt(ss/d + eps), y = x*scale*w; quantize body: dsc =
 *          am/127, q = rint(e*di), clamp; swiglu: g/(1+exp(-g))*u).
 *   [R56]  "12 - r5-r6 re-ranking + structural rewrite spec"
 *          (yusiwen.cn/minfer): sec. 2 / 3.1 (q8_0 activation x Q8_0-style
 *          weight blocks contracted with per-block scales; the q4_K weight
 *          value d*s*nib - dmin*m, whose min term the plane's ssum serves).
 *
 * Readings where the pages are silent or disagree:
 *   - di = 1/d computed in f32 (the page multiplies by di); di = 0 when d = 0.
 *   - clamp to [-127, 127]: for finite inputs |x*di| < 127.5, so the page's
 *     [-128, 127] clamp and the +-127 clamp give identical codes.
 *   - rint rounds half to even (default IEEE rounding mode).
 *   - the stored d is the f32 d rounded to f16 (round to nearest even).
 *   - ds word = f16 bits of d in bits 0..15, int16 ssum in bits 16..31.
 *   - RMSNorm, SwiGLU and the contraction are evaluated in fp64 ("truth"),
 *     not as models of any GPU instruction.
 *   - asymmetric 4-bit blocks: one f16 scale and one f16 min per 32 elements
 *     (the q4_K super-block packing is left out), nibble j < 16 in the low
 *     half of byte j, nibble j >= 16 in the high half of byte j - 16.
 *
 * Parity pins (tests/test_oracle_pins.py): exhaustive f32->f16 against numpy,
 * half-even ties, the round-trip bound |x - q*d| <= d/2 (+ f32 slack), the
 * ssum invariant, closed forms for RMSNorm/SwiGLU, Python-int brute force of
 * the block dot products, the all-scales-one integer matmul, and the pages'
 * byte accounts.  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32          /* elements per q8_0 block            [L05 sec. 2.1] */
#define WBLK_BYTES 34  /* f16 d + 32 x int8                  [L05 sec. 2.1] */

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary32 <-> binary16, written from the format definitions.      */
/* ------------------------------------------------------------------------ */

/* binary32 -> binary16, round to nearest, ties to even; overflow -> inf.   */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ebits = (x >> 23) & 0xffu;
    uint32_t frac = x & 0x7fffffu;

    if (ebits == 0xffu)                       /* inf or NaN */
        return (uint16_t)(sign | 0x7c00u | (frac ? 0x0200u : 0u));
    if (ebits == 0u)                          /* f32 zero/subnormal: < 2^-126 */
        return sign;                          /* far below half the f16 quantum */

    int e = (int)ebits - 127;                 /* value = sig * 2^(e-23) */
    uint32_t sig = frac | 0x800000u;          /* 24-bit significand */
    if (e > 15)                               /* >= 2^16: beyond f16 max */
        return (uint16_t)(sign | 0x7c00u);

    /* Quantum of the target: 2^(e-10) for normals (e >= -14), else 2^-24.   */
    int shift = (e >= -14) ? 13 : (-1 - e);   /* sig >> shift = quanta count */
    if (shift > 24)                           /* value < 2^-25: rounds to 0 */
        return sign;
    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1u;

    uint32_t bits;
    if (e >= -14)
        bits = ((uint32_t)(e + 15) << 10) + (q - 1024u); /* carry -> exponent */
    else
        bits = q;                                        /* subnormal (or 2^-14) */
    if (bits >= 0x7c00u)
        bits = 0x7c00u;                                  /* rounded up to inf */
    return (uint16_t)(sign | bits);
}

/* binary16 -> binary32 (exact). */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (h & 0x8000u) ? 1u : 0u;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t m = h & 0x3ffu;
    double v;
    if (e == 0u)
        v = ldexp((double)m, -24);
    else if (e == 31u)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024u), (int)e - 25);
    return (float)(sign ? -v : v);
}

void oracle_f32_to_f16_array(const float *in, uint16_t *out, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f16_to_f32_array(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_f16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* q8_0 activation quantization of one 32-element block            [R51 3.2] */
/* ------------------------------------------------------------------------ */

/* Steps, in the page's order: amax over the block; d = amax/127 in f32;
 * di = 1/d; q = rint(x*di) clamped; ssum = sum of q; d stored as f16.     */
static void quantize_block(const float *x, uint16_t *d16, int8_t *q, int16_t *ssum)
{
    float amax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    float di = (d != 0.0f) ? 1.0f / d : 0.0f;
    int s = 0;
    for (int j = 0; j < QK; j++) {
        float r = rintf(x[j] * di);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[j] = (int8_t)r;
        s += q[j];
    }
    *d16 = oracle_f32_to_f16(d);
    *ssum = (int16_t)s;
}

/* Diagnostic, not part of the path: how many elements would get a different
 * code under the other reading of the quantize step, q = rint(x/d) (one f32
 * division) instead of the adopted q = rint(x * (1/d)) (a rounded reciprocal,
 * then a rounded product), both clamped to +-127 with d = amax/127 in f32.
 * [R51 3.2] prints the product form; the other form is the plain definition
 * q = rint(x/d).  Returns the count over rows x k elements.                 */
int64_t oracle_div_reading_diff(const float *x, int64_t rows, int64_t k)
{
    int64_t nb = k / QK, count = 0;
#pragma omp parallel for schedule(static) reduction(+ : count)
    for (int64_t t = 0; t < rows; t++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *xb = x + t * k + b * QK;
            float amax = 0.0f;
            for (int j = 0; j < QK; j++) {
                float a = fabsf(xb[j]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f;
            if (d == 0.0f)
                continue; /* both readings give 0 */
            float di = 1.0f / d;
            for (int j = 0; j < QK; j++) {
                float r_mul = rintf(xb[j] * di);
                float r_div = rintf(xb[j] / d);
                if (r_mul > 127.0f) r_mul = 127.0f;
                if (r_mul < -127.0f) r_mul = -127.0f;
                if (r_div > 127.0f) r_div = 127.0f;
                if (r_div < -127.0f) r_div = -127.0f;
                if (r_mul != r_div)
                    count++;
            }
        }
    }
    return count;
}

/* The f32 d of a block (before f16 storage), exported for round-trip pins. */
float oracle_block_d32(const float *x)
{
    float amax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax)
            amax = a;
    }
    return amax / 127.0f;
}

/* Plane layout: qs int8 [rows_pad][k]; ds uint32 [rows_pad][k/32] with the
 * f16 bits of d in bits 0..15 and ssum (int16) in bits 16..31.  Rows
 * rows..rows_pad-1 are all zero (padded token rows)               [R51 3.1] */
void oracle_quantize(const float *x, int64_t rows, int64_t k,
                     int8_t *qs, uint32_t *ds, int64_t rows_pad)
{
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows_pad; t++) {
        for (int64_t b = 0; b < nb; b++) {
            int8_t *qo = qs + t * k + b * QK;
            uint32_t *dso = ds + t * nb + b;
            if (t >= rows) {
                memset(qo, 0, QK);
                *dso = 0u;
                continue;
            }
            uint16_t d16;
            int16_t ssum;
            quantize_block(x + t * k + b * QK, &d16, qo, &ssum);
            *dso = (uint32_t)d16 | ((uint32_t)(uint16_t)ssum << 16);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm (producer of the gate/up and q/k/v activations)          [R51 3.2] */
/* ------------------------------------------------------------------------ */

/* y = (x * scale) * w with scale = 1/sqrt(mean(x^2) + eps), all in fp64.   */
void oracle_rmsnorm(const float *x, const float *w, float eps,
                    int64_t rows, int64_t d, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows; t++) {
        const float *xr = x + t * d;
        double ss = 0.0;
        for (int64_t i = 0; i < d; i++)
            ss += (double)xr[i] * (double)xr[i];
        double scale = 1.0 / sqrt(ss / (double)d + (double)eps);
        for (int64_t i = 0; i < d; i++)
            y[t * d + i] = ((double)xr[i] * scale) * (double)w[i];
    }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU (producer of the down-projection activation)              [R51 3.2] */
/* ------------------------------------------------------------------------ */

/* y = g / (1 + exp(-g)) * u in fp64. */
void oracle_swiglu(const float *g, const float *u, int64_t n, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        double gv = (double)g[i];
        y[i] = gv / (1.0 + exp(-gv)) * (double)u[i];
    }
}

/* ------------------------------------------------------------------------ */
/* Q8_0 weights x q8_0 activations                    [L05 2.1-2.2, R56 2]  */
/* ------------------------------------------------------------------------ */

/* Weight row n is nb consecutive 34-byte blocks: little-endian f16 d at +0,
 * int8 qs[32] at +2.                                            [L05 2.1] */
static inline float wblock_d(const uint8_t *blk)
{
    uint16_t h = (uint16_t)(blk[0] | ((uint16_t)blk[1] << 8));
    return oracle_f16_to_f32(h);
}

static inline float plane_d(uint32_t w)
{
    return oracle_f16_to_f32((uint16_t)(w & 0xffffu));
}

/* Integer dot product of weight block b of row n with activation block b of
 * token t: exact in int32 (|sum| <= 32*127*127).                          */
static inline int32_t block_dot(const uint8_t *wblk, const int8_t *qa)
{
    const int8_t *qw = (const int8_t *)(wblk + 2);
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
        s += (int32_t)qw[j] * (int32_t)qa[j];
    return s;
}

/* y[i][j] = sum_b d_w(n_j, b) * d_a(t_i, b) * isum_b   for the sampled
 * tokens t_idx[0..nt) and rows n_idx[0..nn).  Each term is exact in fp64
 * (11 + 11 + 20 significant bits); the sum over b is in fp64.  absum gets
 * sum_b |term_b|, the scale of the summation used by the tolerance.       */
void oracle_gemm(const uint8_t *w, int64_t n, int64_t k,
                 const int8_t *qs, const uint32_t *ds,
                 const int64_t *t_idx, int64_t nt,
                 const int64_t *n_idx, int64_t nn,
                 double *y, double *absum)
{
    int64_t nb = k / QK;
    int64_t pitch = nb * WBLK_BYTES;
    (void)n;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nt; i++) {
        int64_t t = t_idx[i];
        for (int64_t j = 0; j < nn; j++) {
            const uint8_t *wr = w + n_idx[j] * pitch;
            double acc = 0.0, aacc = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *wblk = wr + b * WBLK_BYTES;
                int32_t isum = block_dot(wblk, qs + t * k + b * QK);
                double term = (double)wblock_d(wblk) * (double)plane_d(ds[t * nb + b]) * (double)isum;
                acc += term;
                aacc += fabs(term);
            }
            y[i * nn + j] = acc;
            absum[i * nn + j] = aacc;
        }
    }
}

/* isum[i][j][b] for tiny shapes (pinned by Python-int brute force). */
void oracle_block_dots(const uint8_t *w, int64_t n, int64_t k,
                       const int8_t *qs, int64_t t, int32_t *isum)
{
    int64_t nb = k / QK;
    int64_t pitch = nb * WBLK_BYTES;
    for (int64_t i = 0; i < t; i++)
        for (int64_t j = 0; j < n; j++)
            for (int64_t b = 0; b < nb; b++)
                isum[(i * n + j) * nb + b] =
                    block_dot(w + j * pitch + b * WBLK_BYTES, qs + i * k + b * QK);
}

/* ------------------------------------------------------------------------ */
/* Asymmetric 4-bit weight blocks x q8_0 activations: the consumer of ssum    */
/*                                          [R51 2.1; R56 sec. 2, q4_K value] */
/* ------------------------------------------------------------------------ */

/* A 32-element asymmetric weight block, 20 bytes: little-endian f16 d at +0,
 * f16 m at +2, 16 bytes of unsigned nibbles at +4.  Element j (0..31) is
 * nib_j = low nibble of byte j for j < 16, high nibble of byte j - 16 for
 * j >= 16, and its value is d * nib_j - m: the pages' q4_K value form
 * d*s*nib - dmin*m with the two-level (super-block, sub-block) scales folded
 * into one f16 scale and one f16 min per 32-element block.                 */
#define A4BLK_BYTES 20

static inline int a4_nib(const uint8_t *blk, int j)
{
    const uint8_t b = blk[4 + (j & 15)];
    return j < 16 ? (b & 15) : (b >> 4);
}

static inline float a4_half(const uint8_t *p)
{
    return oracle_f16_to_f32((uint16_t)(p[0] | ((uint16_t)p[1] << 8)));
}

/* y[i][j] = sum_b sum_e (d*nib_e - m) * (d_a*q_e) for weight row n_idx[j] and
 * token t_idx[i].  Per block, as the pages' min-term correction does:
 *     d * d_a * sum_e nib_e*q_e  -  m * d_a * ssum,
 * with ssum = sum_e q_e taken from the plane (its int16 field) instead of a
 * second dot product.  Both terms are exact in fp64 (11+11+16 and 11+11+13
 * significant bits); absum gets the sum of their magnitudes.              */
void oracle_q4a_gemm(const uint8_t *w, int64_t n, int64_t k,
                     const int8_t *qs, const uint32_t *ds,
                     const int64_t *t_idx, int64_t nt,
                     const int64_t *n_idx, int64_t nn,
                     double *y, double *absum)
{
    int64_t nb = k / QK;
    int64_t pitch = nb * A4BLK_BYTES;
    (void)n;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nt; i++) {
        int64_t t = t_idx[i];
        for (int64_t j = 0; j < nn; j++) {
            const uint8_t *wr = w + n_idx[j] * pitch;
            double acc = 0.0, aacc = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *blk = wr + b * A4BLK_BYTES;
                const int8_t *qa = qs + t * k + b * QK;
                int32_t isum = 0;
                for (int e = 0; e < QK; e++)
                    isum += (int32_t)a4_nib(blk, e) * (int32_t)qa[e];
                uint32_t dsw = ds[t * nb + b];
                int16_t ssum = (int16_t)(uint16_t)(dsw >> 16);
                double da = (double)plane_d(dsw);
                double t1 = (double)a4_half(blk) * da * (double)isum;
                double t2 = (double)a4_half(blk + 2) * da * (double)ssum;
                acc += t1;
                acc -= t2;
                aacc += fabs(t1) + fabs(t2);
            }
            y[i * nn + j] = acc;
            absum[i * nn + j] = aacc;
        }
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
