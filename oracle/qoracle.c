/*
 * qoracle.c -- plain, slow, single-threaded CPU oracle for weight-only,
 * group-wise, low-bit quantization and the linear layer y = x . dequant(W)^T.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA
 * library (no headers, tables or helpers); the two meet only through the
 * seeded inputs the tests hand to both.
 *
 * What it computes, and where each step comes from:
 *
 *  - Affine asymmetric quantizer: scale = (max - min) / (qmax - qmin),
 *    zero_point = qmin - round(min / scale), q = round(x / scale) + zero_point,
 *    x_hat = (q - zero_point) * scale  ("Inference acceleration guide" page, section 1.1).
 *  - Per-group statistics over groups of consecutive weights along K, with the
 *    top 0.1 % of weights by magnitude excluded and kept as FP16 outliers that
 *    are added back after the matrix product ("70B on one GPU" page,
 *    section 2, steps 1-3; group size 128).
 *  - 2-bit layers use a 4-entry non-uniform codebook found by k-means
 *    ("Mixed-width quantization" page, sections 2.1 table and 4.1).
 *  - Packing: b-bit codes stored LSB-first in a little-endian bit stream;
 *    the pages' unpack routines read 3-bit units of 8 values in 3 bytes with
 *    shifts 0,3,...,21, 6-bit units of 4 values in 3 bytes with shifts
 *    0,6,12,18, 5-bit units of 8 values in 5 bytes with shifts 5i ("Mixed-width quantization"
 *    page, sections 3.1-3.2), the 4-bit value pair as the low/high half of a
 *    byte (section 2.1 table).
 *  - Group sizes 32, 64 and 128; at 32 the scale may be stored as an 8-bit
 *    float, groups outside its range keeping an fp16 scale ("Mixed-width
 *    quantization" page, section 2.3; see orc_quantize_fp8).
 *  - The product accumulates in fp64 here (the pages require at least fp32
 *    accumulation, "Mixed-width quantization" page, section 4.2).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  round = round-half-to-even; q clamped to [0, 2^b - 1]; the group range is
 *  widened to include 0; the fp16 scale is rounded toward +infinity from the
 *  fp32 quotient; zero-point stored as one byte per group; "top 0.1 %" =
 *  the floor(frac*N*K) largest |w| of the whole matrix (ties by lower linear
 *  index); the dense code at an outlier contributes 0 (affine) or the
 *  codebook entry nearest to 0 with the residual stored (2-bit); the codebook
 *  is 16 Lloyd iterations from a uniform 4-level start with ties to the lower
 *  entry.  All fp32 arithmetic below is IEEE single precision, round to
 *  nearest even, evaluated in the order written (build with
 *  -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ENOMEM -2
#define ORC_ENONFINITE -3

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16, written from the format definitions */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

float orc_f16_to_f32(uint16_t h) { return (float)orc_f16_to_f64(h); }

/* Round a float to binary16.  mode 0: nearest, ties to even.  mode 1: toward
 * +infinity.  The value is split as q * ulp with ulp the spacing of binary16
 * numbers in the value's binade (2^-24 below the normal range); q is then
 * rounded to an integer, which is exactly the rounding of the significand. */
static uint16_t f32_to_f16(float f, int mode)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return (uint16_t)(sign | 0x7E00);
    if (isinf(f)) return (uint16_t)(sign | 0x7C00);
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);                 /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    if (E < -14) E = -14;
    double ulp = ldexp(1.0, E - 10);
    double q = a / ulp;            /* exact: power-of-two scaling */
    double qi;
    if (mode == 0)
        qi = nearbyint(q);         /* default environment: ties to even */
    else
        qi = sign ? floor(q) : ceil(q);   /* toward +inf on the signed value */
    double r = qi * ulp;
    if (r >= 65536.0) return (uint16_t)(sign | 0x7C00);   /* overflow */
    if (r < ldexp(1.0, -14))                            /* subnormal or 0 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    frexp(r, &e2);
    int Er = e2 - 1;
    uint16_t m = (uint16_t)(r / ldexp(1.0, Er - 10) - 1024.0);
    return (uint16_t)(sign | ((Er + 15) << 10) | m);
}

uint16_t orc_f32_to_f16_rn(float f) { return f32_to_f16(f, 0); }
uint16_t orc_f32_to_f16_ru(float f) { return f32_to_f16(f, 1); }

/* bfloat16 is the upper half of a binary32. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

void orc_f16_to_f32_array(const uint16_t *in, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_f16_to_f32(in[i]);
}

void orc_f32_to_f16_array(const float *in, int64_t n, int mode, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = f32_to_f16(in[i], mode);
}

/* ------------------------------------------------------------------ */
/* sizes                                                                */
/* ------------------------------------------------------------------ */

/* Number of outliers: floor(frac * N * K) evaluated in double. */
int64_t orc_nnz(int64_t N, int64_t K, float frac)
{
    if (frac <= 0.0f) return 0;
    return (int64_t)floor((double)frac * (double)N * (double)K);
}

static int valid_shape(int64_t N, int64_t K, int bits, int group)
{
    if (N <= 0 || K <= 0) return 0;
    if ((bits < 2 || bits > 6) && bits != 8) return 0;
    if (group != 32 && group != 64 && group != 128) return 0;
    if (K % group) return 0;
    return 1;
}

/* Bytes of each buffer of a quantized matrix (packed codes, fp16 scales,
 * one-byte zero-points, fp16 codebooks, outlier CSR).  out[0..7] =
 * packed, scale, zp, codebook, nnz, row_ptr, col, val. */
int orc_sizes(int64_t N, int64_t K, int bits, int group, float frac, int64_t *out)
{
    if (!valid_shape(N, K, bits, group) || frac < 0.0f || frac >= 1.0f) return ORC_EINVAL;
    int64_t ng = K / group;
    int64_t nnz = orc_nnz(N, K, frac);
    out[0] = N * K * bits / 8;
    out[1] = bits == 2 ? 0 : N * ng * 2;
    out[2] = bits == 2 ? 0 : N * ng;
    out[3] = bits == 2 ? N * ng * 4 * 2 : 0;
    out[4] = nnz;
    out[5] = (N + 1) * 4;
    out[6] = nnz * 4;
    out[7] = nnz * 2;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* bit packing: code i occupies stream bits [b*i, b*i + b), bit j of the  */
/* code at stream bit b*i + j; stream bit t is bit (t mod 8) of byte t/8. */
/* ------------------------------------------------------------------ */
void orc_pack(const uint8_t *codes, int64_t n, int bits, uint8_t *out)
{
    int64_t nbytes = (n * bits + 7) / 8;
    memset(out, 0, (size_t)nbytes);
    for (int64_t i = 0; i < n; i++)
        for (int j = 0; j < bits; j++)
            if ((codes[i] >> j) & 1u) {
                int64_t t = i * bits + j;
                out[t / 8] |= (uint8_t)(1u << (t % 8));
            }
}

void orc_unpack(const uint8_t *in, int64_t n, int bits, uint8_t *codes)
{
    for (int64_t i = 0; i < n; i++) {
        unsigned c = 0;
        for (int j = 0; j < bits; j++) {
            int64_t t = i * bits + j;
            c |= ((in[t / 8] >> (t % 8)) & 1u) << j;
        }
        codes[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------ */
/* outlier selection                                                    */
/* ------------------------------------------------------------------ */
typedef struct {
    uint16_t mag;   /* |w| as the binary16 bit pattern without sign */
    uint32_t idx;   /* linear index n*K + k */
} okey;

static int okey_cmp(const void *pa, const void *pb)
{
    const okey *a = (const okey *)pa, *b = (const okey *)pb;
    if (a->mag != b->mag) return a->mag > b->mag ? -1 : 1;   /* larger |w| first */
    return a->idx < b->idx ? -1 : (a->idx > b->idx);        /* then lower index */
}

static int finite16(uint16_t h) { return ((h >> 10) & 0x1F) != 31; }

/* Mark the floor(frac*N*K) largest-|w| elements.  mask[n*K+k] = 1 for an
 * outlier.  Returns nnz or a negative error. */
static int64_t select_outliers(const uint16_t *W, int64_t N, int64_t K, float frac, uint8_t *mask)
{
    int64_t total = N * K, nnz = orc_nnz(N, K, frac);
    memset(mask, 0, (size_t)total);
    if (nnz == 0) return 0;
    if (total > 0xFFFFFFFFll) return ORC_EINVAL;
    okey *keys = (okey *)malloc(sizeof(okey) * (size_t)total);
    if (!keys) return ORC_ENOMEM;
    for (int64_t i = 0; i < total; i++) {
        keys[i].mag = (uint16_t)(W[i] & 0x7FFF);
        keys[i].idx = (uint32_t)i;
    }
    qsort(keys, (size_t)total, sizeof(okey), okey_cmp);
    for (int64_t r = 0; r < nnz; r++) mask[keys[r].idx] = 1;
    free(keys);
    return nnz;
}

/* CSR of the outlier positions, columns ascending within a row. */
int64_t orc_select_outliers(const uint16_t *W, int64_t N, int64_t K, float frac,
                            int32_t *row_ptr, int32_t *col)
{
    uint8_t *mask = (uint8_t *)malloc((size_t)(N * K));
    if (!mask) return ORC_ENOMEM;
    int64_t nnz = select_outliers(W, N, K, frac, mask);
    if (nnz >= 0) {
        int64_t p = 0;
        for (int64_t n = 0; n < N; n++) {
            row_ptr[n] = (int32_t)p;
            for (int64_t k = 0; k < K; k++)
                if (mask[n * K + k]) col[p++] = (int32_t)k;
        }
        row_ptr[N] = (int32_t)p;
    }
    free(mask);
    return nnz;
}

/* ------------------------------------------------------------------ */
/* group quantizers                                                     */
/* ------------------------------------------------------------------ */

/* Range of a group's non-outlier elements, widened to contain 0. */
static void group_range(const uint16_t *w, const uint8_t *is_out, int g, float *mn_out, float *mx_out)
{
    float mn = 0.0f, mx = 0.0f;
    for (int i = 0; i < g; i++) {
        if (is_out[i]) continue;
        float v = orc_f16_to_f32(w[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    *mn_out = mn;
    *mx_out = mx;
}

/* Affine scale: (max - min) / (qmax - qmin) in fp32, rounded up to fp16
 * (1.0 when max == min). */
static uint16_t affine_scale16(float mn, float mx, int bits)
{
    const int qmin = 0, qmax = (1 << bits) - 1;
    if (mx == mn) return 0x3C00; /* 1.0 */
    float range = mx - mn;
    float s32 = range / (float)(qmax - qmin);
    return f32_to_f16(s32, 1);
}

/* Codes of an affine group for the fp16 scale s16: zp = clamp(qmin -
 * round(min / scale)), q = clamp(round(w / scale) + zp); q = zp at outliers.
 * Returns zp. */
static uint8_t affine_encode(const uint16_t *w, const uint8_t *is_out, int g, int bits, float mn, uint16_t s16,
                             uint8_t *codes)
{
    const int qmin = 0, qmax = (1 << bits) - 1;
    float s = orc_f16_to_f32(s16);
    float r = rintf(mn / s);
    int zp = qmin - (int)r;
    if (zp < qmin) zp = qmin;
    if (zp > qmax) zp = qmax;
    for (int i = 0; i < g; i++) {
        int q;
        if (is_out[i]) {
            q = zp;     /* dense part contributes (zp - zp) * s = 0 */
        } else {
            float v = orc_f16_to_f32(w[i]);
            q = (int)rintf(v / s) + zp;
            if (q < qmin) q = qmin;
            if (q > qmax) q = qmax;
        }
        codes[i] = (uint8_t)q;
    }
    return (uint8_t)zp;
}

/* Affine asymmetric quantizer of one group (b in 2..8).
 * w: g fp16 values, out: g codes.  Writes the fp16 scale and the u8 zp. */
static void quant_group_affine(const uint16_t *w, const uint8_t *is_out, int g, int bits,
                               uint8_t *codes, uint16_t *scale16, uint8_t *zp_out)
{
    float mn, mx;
    group_range(w, is_out, g, &mn, &mx);
    uint16_t s16 = affine_scale16(mn, mx, bits);
    *zp_out = affine_encode(w, is_out, g, bits, mn, s16, codes);
    *scale16 = s16;
}

/* Symmetric quantizer of one group, stored in the affine format ("Mixed-
 * width quantization" page, section 2.3: no zero point for the narrow
 * widths, the scale absorbs the offset; the integer range follows the
 * symmetric INT8 example of the inference-acceleration guide page, section
 * 1.1, [-(2^(b-1) - 1), 2^(b-1) - 1]).  With qs = 2^(b-1) - 1 and amax the
 * largest |w| over the non-outliers: scale = fp16 rounded up of amax / qs
 * (1.0 if amax is 0), q = clamp(round(w / scale), -qs, qs), stored as
 * q + 2^(b-1) with the zero point byte fixed at 2^(b-1); q = 0 at outliers. */
static uint16_t symmetric_scale16(const uint16_t *w, const uint8_t *is_out, int g, int bits)
{
    const int qs = (1 << (bits - 1)) - 1;
    float amax = 0.0f;
    for (int i = 0; i < g; i++) {
        if (is_out[i]) continue;
        float a = fabsf(orc_f16_to_f32(w[i]));
        if (a > amax) amax = a;
    }
    return amax == 0.0f ? 0x3C00 : f32_to_f16(amax / (float)qs, 1);
}

static uint8_t symmetric_encode(const uint16_t *w, const uint8_t *is_out, int g, int bits, uint16_t s16,
                                uint8_t *codes)
{
    const int qs = (1 << (bits - 1)) - 1, zp = 1 << (bits - 1);
    float s = orc_f16_to_f32(s16);
    for (int i = 0; i < g; i++) {
        int q = 0;
        if (!is_out[i]) {
            q = (int)rintf(orc_f16_to_f32(w[i]) / s);
            if (q < -qs) q = -qs;
            if (q > qs) q = qs;
        }
        codes[i] = (uint8_t)(q + zp);
    }
    return (uint8_t)zp;
}

static void quant_group_symmetric(const uint16_t *w, const uint8_t *is_out, int g, int bits,
                                  uint8_t *codes, uint16_t *scale16, uint8_t *zp_out)
{
    uint16_t s16 = symmetric_scale16(w, is_out, g, bits);
    *zp_out = symmetric_encode(w, is_out, g, bits, s16, codes);
    *scale16 = s16;
}

/* 2-bit groups on a uniform grid, stored as the four constants a code
 * selects ("Mixed-width quantization" page, section 4.2: a linear 2-bit grid
 * maps each code to one of four constants picked by a select instruction,
 * not a k-means codebook).  mode 1 (symmetric): the symmetric rule above at
 * b = 2 (qs = 1, levels -s, 0, s; the fourth constant repeats s), codes
 * q + 1.  mode 2 (linear): the affine quantizer at b = 2 (range widened to
 * contain 0, scale = fp16 rounded up of (max - min) / 3, zp = clamp(-round(
 * min / scale), 0, 3), q = clamp(round(w / scale) + zp, 0, 3)), constants
 * fp16((i - zp) * scale) for i = 0..3.  Either way the constant of the zero
 * code is exactly 0, so an outlier takes that code and keeps fp16(w) as its
 * stored value. */
static void quant_group_uniform2(const uint16_t *w, const uint8_t *is_out, int g, int mode,
                                 uint8_t *codes, uint16_t cb16[4], uint16_t *resid)
{
    if (mode == 1) {
        float amax = 0.0f;
        for (int i = 0; i < g; i++) {
            if (is_out[i]) continue;
            float a = fabsf(orc_f16_to_f32(w[i]));
            if (a > amax) amax = a;
        }
        uint16_t s16 = amax == 0.0f ? 0x3C00 : f32_to_f16(amax, 1);
        float s = orc_f16_to_f32(s16);
        for (int i = 0; i < g; i++) {
            int q = 0;
            if (!is_out[i]) {
                q = (int)rintf(orc_f16_to_f32(w[i]) / s);
                if (q < -1) q = -1;
                if (q > 1) q = 1;
            }
            codes[i] = (uint8_t)(q + 1);
            if (is_out[i]) resid[i] = w[i];
        }
        cb16[0] = (uint16_t)(s16 | 0x8000);
        cb16[1] = 0;
        cb16[2] = s16;
        cb16[3] = s16;
        return;
    }
    uint16_t s16;
    uint8_t zp;
    quant_group_affine(w, is_out, g, 2, codes, &s16, &zp);
    float s = orc_f16_to_f32(s16);
    for (int i = 0; i < 4; i++) cb16[i] = f32_to_f16((float)(i - (int)zp) * s, 0);
    for (int i = 0; i < g; i++)
        if (is_out[i]) resid[i] = w[i];
}

/* Index of the entry nearest to v; ties go to the lower index. */
static int nearest4(float v, const float c[4])
{
    int best = 0;
    float bd = fabsf(v - c[0]);
    for (int i = 1; i < 4; i++) {
        float d = fabsf(v - c[i]);
        if (d < bd) {
            bd = d;
            best = i;
        }
    }
    return best;
}

#define LLOYD_ITERS 16

/* 2-bit non-uniform codebook of one group: 1-D k-means (Lloyd) with four
 * centroids, started from four evenly spaced levels over the group range.
 * Writes 4 fp16 entries (ascending) and the codes.  For an outlier the code
 * is the entry nearest to 0 and *resid receives fp16(w - entry). */
static void quant_group_codebook(const uint16_t *w, const uint8_t *is_out, int g,
                                 uint8_t *codes, uint16_t cb16[4], uint16_t *resid)
{
    float mn = 0.0f, mx = 0.0f;
    for (int i = 0; i < g; i++) {
        if (is_out[i]) continue;
        float v = orc_f16_to_f32(w[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float c[4];
    float step = (mx - mn) / 3.0f;
    for (int i = 0; i < 4; i++) c[i] = mn + (float)i * step;

    for (int it = 0; it < LLOYD_ITERS; it++) {
        float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int cnt[4] = {0, 0, 0, 0};
        for (int i = 0; i < g; i++) {      /* ascending k */
            if (is_out[i]) continue;
            float v = orc_f16_to_f32(w[i]);
            int j = nearest4(v, c);
            sum[j] = sum[j] + v;
            cnt[j] += 1;
        }
        for (int j = 0; j < 4; j++)
            if (cnt[j] > 0) c[j] = sum[j] / (float)cnt[j];   /* empty: keep */
    }

    /* fp16 entries, then a stable ascending sort */
    uint16_t e[4];
    for (int i = 0; i < 4; i++) e[i] = f32_to_f16(c[i], 0);
    for (int i = 1; i < 4; i++) {
        uint16_t x = e[i];
        float xv = orc_f16_to_f32(x);
        int j = i - 1;
        while (j >= 0 && orc_f16_to_f32(e[j]) > xv) {
            e[j + 1] = e[j];
            j--;
        }
        e[j + 1] = x;
    }
    float ef[4];
    for (int i = 0; i < 4; i++) ef[i] = orc_f16_to_f32(e[i]);
    int zero_code = nearest4(0.0f, ef);
    for (int i = 0; i < g; i++) {
        if (is_out[i]) {
            codes[i] = (uint8_t)zero_code;
            float v = orc_f16_to_f32(w[i]);
            resid[i] = f32_to_f16(v - ef[zero_code], 0);
        } else {
            codes[i] = (uint8_t)nearest4(orc_f16_to_f32(w[i]), ef);
        }
    }
    for (int i = 0; i < 4; i++) cb16[i] = e[i];
}

/* Quantize and pack a whole matrix W [N, K] (fp16 bit patterns).
 * Outputs (caller-allocated, sizes from orc_sizes): packed [N, K*bits/8],
 * scale fp16 [N, K/group] and zp u8 [N, K/group] for bits != 2,
 * cb fp16 [N, K/group, 4] for bits == 2, outlier CSR row_ptr [N+1],
 * col [nnz], val fp16 [nnz].  Unused outputs may be NULL. */
int orc_quantize_mode(const uint16_t *W, int64_t N, int64_t K, int bits, int group, float frac, int mode,
                      uint8_t *packed, uint16_t *scale, uint8_t *zp, uint16_t *cb,
                      int32_t *row_ptr, int32_t *col, uint16_t *val)
{
    if (!valid_shape(N, K, bits, group) || frac < 0.0f || frac >= 1.0f) return ORC_EINVAL;
    if (mode < 0 || mode > 2 || (mode == 2 && bits != 2)) return ORC_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (!finite16(W[i])) return ORC_ENONFINITE;
    int64_t ng = K / group;
    uint8_t *mask = (uint8_t *)malloc((size_t)(N * K));
    uint8_t *codes = (uint8_t *)malloc((size_t)K);
    uint16_t *resid = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K);
    if (!mask || !codes || !resid) {
        free(mask); free(codes); free(resid);
        return ORC_ENOMEM;
    }
    int64_t nnz = select_outliers(W, N, K, frac, mask);
    if (nnz < 0) {
        free(mask); free(codes); free(resid);
        return (int)nnz;
    }
    int64_t p = 0;
    for (int64_t n = 0; n < N; n++) {
        const uint16_t *wr = W + n * K;
        const uint8_t *mr = mask + n * K;
        for (int64_t j = 0; j < ng; j++) {
            int64_t k0 = j * group;
            if (bits == 2 && mode == 0)
                quant_group_codebook(wr + k0, mr + k0, group, codes + k0, cb + (n * ng + j) * 4,
                                     resid + k0);
            else if (bits == 2)
                quant_group_uniform2(wr + k0, mr + k0, group, mode, codes + k0, cb + (n * ng + j) * 4,
                                     resid + k0);
            else if (mode == 1)
                quant_group_symmetric(wr + k0, mr + k0, group, bits, codes + k0, scale + n * ng + j,
                                      zp + n * ng + j);
            else
                quant_group_affine(wr + k0, mr + k0, group, bits, codes + k0, scale + n * ng + j,
                                   zp + n * ng + j);
        }
        orc_pack(codes, K, bits, packed + n * (K * bits / 8));
        row_ptr[n] = (int32_t)p;
        for (int64_t k = 0; k < K; k++)
            if (mr[k]) {
                col[p] = (int32_t)k;
                val[p] = bits == 2 ? resid[k] : wr[k];
                p++;
            }
    }
    row_ptr[N] = (int32_t)p;
    free(mask); free(codes); free(resid);
    return ORC_OK;
}

/* The default quantizer: asymmetric affine at 3..6 bits, k-means codebook at 2. */
int orc_quantize(const uint16_t *W, int64_t N, int64_t K, int bits, int group, float frac,
                 uint8_t *packed, uint16_t *scale, uint8_t *zp, uint16_t *cb,
                 int32_t *row_ptr, int32_t *col, uint16_t *val)
{
    return orc_quantize_mode(W, N, K, bits, group, frac, 0, packed, scale, zp, cb, row_ptr, col, val);
}

/* ------------------------------------------------------------------ */
/* 8-bit float (E4M3) group scales with an fp16 fallback                */
/* ------------------------------------------------------------------ */
/* "Mixed-width quantization" page, section 2.3: the group scale itself may
 * be stored as an 8-bit float.  Its range is narrower than fp16's, so the
 * scales of all groups are surveyed first; the groups whose scale falls
 * outside what the 8-bit format can hold keep an fp16 scale, all others
 * store 8 bits.  Readings (the page names neither the format nor the
 * window):
 *  - the format is E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 fraction
 *    bits, no infinities, S.1111.111 is NaN, largest finite value 448;
 *  - one power of two per matrix, 2^E, places the format's range over the
 *    scales: E is the lower median of floor(log2 s16) over all groups of
 *    the matrix (the survey), so the typical scale sits near 1 in the
 *    format's terms and only groups far from it fall out;
 *  - a group's code is the least normal E4M3 value >= s16 * 2^-E (rounded up,
 *    like the fp16 scale, so the grid still spans the group's range);
 *  - the group falls back to fp16 when s16 * 2^-E is below the normal range
 *    (2^-6), when the rounded value would exceed 448, or when (the rounded
 *    value) * 2^E is not a normal fp16 number; a fallback group stores code
 *    0x7F and keeps s16 in a per-row list (row_ptr [N+1], group index,
 *    fp16 scale), groups ascending;
 *  - the codes and the zero point are then those of the quantizer above
 *    with the group's stored scale (the E4M3 value times 2^E, which is an
 *    fp16 number, or the fallback s16).
 * 2-bit groups have no single scale (codebooks) and are not covered. */

/* Value of an E4M3 code, written from the format definition. */
double orc_e4m3_to_f64(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m * 2^-9 */
    else
        v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* The least positive normal E4M3 code whose value is >= t, by scanning the
 * normal codes in ascending order; -1 if t < 2^-6 or t > 448. */
int orc_e4m3_ceil_normal(double t)
{
    if (!(t >= ldexp(1.0, -6))) return -1;
    for (int c = 0x08; c <= 0x7E; c++)
        if (orc_e4m3_to_f64((uint8_t)c) >= t) return c;
    return -1;
}

/* floor(log2 v) of a positive finite double. */
static int floor_log2(double v)
{
    int e2;
    frexp(v, &e2);   /* v in [2^(e2-1), 2^e2) */
    return e2 - 1;
}

/* Matrix exponent E: the lower median (element (n-1)/2 in ascending order)
 * of floor(log2 s16) over the n fp16 scales. */
int orc_fp8_matrix_exponent(const uint16_t *s16, int64_t n)
{
    /* fp16 scales lie in [2^-24, 65504]: floor(log2) in [-24, 15] */
    int64_t hist[40] = {0};
    for (int64_t i = 0; i < n; i++) hist[floor_log2(orc_f16_to_f64(s16[i])) + 24]++;
    int64_t want = (n - 1) / 2, seen = 0;
    for (int b = 0; b < 40; b++) {
        seen += hist[b];
        if (seen > want) return b - 24;
    }
    return 0;
}

/* The stored scale of a group with fp16 scale s16 under exponent E: returns
 * the E4M3 code and sets *eff to the fp16 value code * 2^E, or returns 0x7F
 * and sets *eff = s16 (fallback). */
static uint8_t fp8_store(uint16_t s16, int E, uint16_t *eff)
{
    double t = ldexp(orc_f16_to_f64(s16), -E);
    int c = orc_e4m3_ceil_normal(t);
    if (c >= 0) {
        double v = ldexp(orc_e4m3_to_f64((uint8_t)c), E);
        if (v >= ldexp(1.0, -14) && v <= 65504.0) {
            *eff = f32_to_f16((float)v, 0);   /* exact: 4 significant bits */
            return (uint8_t)c;
        }
    }
    *eff = s16;
    return 0x7F;
}

/* Quantize with E4M3 scales (bits 3..8; mode 0 asymmetric, 1 symmetric).
 * Outputs as orc_quantize_mode, with scale8 u8 [N, K/group] in place of the
 * fp16 scales, *exp_out = E, and the fallback list fb_row_ptr [N+1],
 * fb_col [fb_cap] (group index within the row), fb_val fp16 [fb_cap].
 * Returns the number of fallback groups, or a negative ORC_ error
 * (ORC_ENOMEM also when more than fb_cap groups fall back). */
int64_t orc_quantize_fp8(const uint16_t *W, int64_t N, int64_t K, int bits, int group, float frac, int mode,
                         uint8_t *packed, uint8_t *scale8, uint8_t *zp, int32_t *row_ptr, int32_t *col,
                         uint16_t *val, int32_t *exp_out, int32_t *fb_row_ptr, int32_t *fb_col,
                         uint16_t *fb_val, int64_t fb_cap)
{
    if (!valid_shape(N, K, bits, group) || bits == 2 || frac < 0.0f || frac >= 1.0f) return ORC_EINVAL;
    if (mode != 0 && mode != 1) return ORC_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (!finite16(W[i])) return ORC_ENONFINITE;
    int64_t ng = K / group;
    uint8_t *mask = (uint8_t *)malloc((size_t)(N * K));
    uint8_t *codes = (uint8_t *)malloc((size_t)K);
    uint16_t *s16 = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(N * ng));
    if (!mask || !codes || !s16) {
        free(mask); free(codes); free(s16);
        return ORC_ENOMEM;
    }
    int64_t nnz = select_outliers(W, N, K, frac, mask);
    if (nnz < 0) {
        free(mask); free(codes); free(s16);
        return nnz;
    }
    /* 1. the fp16 scale of every group, as the fp16 quantizer finds it */
    for (int64_t n = 0; n < N; n++)
        for (int64_t j = 0; j < ng; j++) {
            const uint16_t *wg = W + n * K + j * group;
            const uint8_t *mg = mask + n * K + j * group;
            if (mode == 1) {
                s16[n * ng + j] = symmetric_scale16(wg, mg, group, bits);
            } else {
                float mn, mx;
                group_range(wg, mg, group, &mn, &mx);
                s16[n * ng + j] = affine_scale16(mn, mx, bits);
            }
        }
    /* 2. the matrix exponent from all groups' scales */
    int E = orc_fp8_matrix_exponent(s16, N * ng);
    /* 3. stored scales, codes with the stored scale, fallback list, outliers */
    int64_t p = 0, f = 0;
    for (int64_t n = 0; n < N; n++) {
        const uint16_t *wr = W + n * K;
        const uint8_t *mr = mask + n * K;
        fb_row_ptr[n] = (int32_t)f;
        for (int64_t j = 0; j < ng; j++) {
            int64_t k0 = j * group;
            uint16_t eff;
            uint8_t c = fp8_store(s16[n * ng + j], E, &eff);
            scale8[n * ng + j] = c;
            if (c == 0x7F) {
                if (f >= fb_cap) {
                    free(mask); free(codes); free(s16);
                    return ORC_ENOMEM;
                }
                fb_col[f] = (int32_t)j;
                fb_val[f] = eff;
                f++;
            }
            if (mode == 1) {
                zp[n * ng + j] = symmetric_encode(wr + k0, mr + k0, group, bits, eff, codes + k0);
            } else {
                float mn, mx;
                group_range(wr + k0, mr + k0, group, &mn, &mx);
                zp[n * ng + j] = affine_encode(wr + k0, mr + k0, group, bits, mn, eff, codes + k0);
            }
        }
        orc_pack(codes, K, bits, packed + n * (K * bits / 8));
        row_ptr[n] = (int32_t)p;
        for (int64_t k = 0; k < K; k++)
            if (mr[k]) {
                col[p] = (int32_t)k;
                val[p] = wr[k];
                p++;
            }
    }
    row_ptr[N] = (int32_t)p;
    fb_row_ptr[N] = (int32_t)f;
    *exp_out = E;
    free(mask); free(codes); free(s16);
    return f;
}

/* The fp16 scale every group stores, from its E4M3 code and the matrix
 * exponent, or from the row's fallback list for code 0x7F.  Returns
 * ORC_EINVAL for a code that is not a positive normal E4M3 value, a scale
 * that is not a normal fp16 number, or a 0x7F group missing from the list. */
int orc_fp8_expand(const uint8_t *scale8, int32_t E, int64_t N, int64_t ng, const int32_t *fb_row_ptr,
                   const int32_t *fb_col, const uint16_t *fb_val, uint16_t *s16_out)
{
    for (int64_t n = 0; n < N; n++)
        for (int64_t j = 0; j < ng; j++) {
            uint8_t c = scale8[n * ng + j];
            if (c == 0x7F) {
                int found = 0;
                for (int32_t q = fb_row_ptr[n]; q < fb_row_ptr[n + 1]; q++)
                    if (fb_col[q] == j) {
                        s16_out[n * ng + j] = fb_val[q];
                        found = 1;
                        break;
                    }
                if (!found) return ORC_EINVAL;
                continue;
            }
            if (c < 0x08 || c > 0x7E) return ORC_EINVAL;
            double v = ldexp(orc_e4m3_to_f64(c), E);
            if (!(v >= ldexp(1.0, -14) && v <= 65504.0)) return ORC_EINVAL;
            s16_out[n * ng + j] = f32_to_f16((float)v, 0);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* dequantization and the linear layer (fp64)                           */
/* ------------------------------------------------------------------ */
typedef struct {
    int64_t N, K;
    int32_t bits, group;
    const uint8_t *packed;
    const uint16_t *scale;
    const uint8_t *zp;
    const uint16_t *cb;
    int64_t nnz;
    const int32_t *row_ptr;
    const int32_t *col;
    const uint16_t *val;
} orc_qweight;

/* Row n of x_hat + S in fp64: x_hat = (q - zp) * scale, or cb[q] for 2-bit;
 * S holds the fp16 outlier values at their positions. */
static void dequant_row(const orc_qweight *w, int64_t n, uint8_t *codes, double *out)
{
    int64_t K = w->K, ng = K / w->group;
    orc_unpack(w->packed + n * (K * w->bits / 8), K, w->bits, codes);
    for (int64_t k = 0; k < K; k++) {
        int64_t j = k / w->group;
        if (w->bits == 2) {
            out[k] = orc_f16_to_f64(w->cb[(n * ng + j) * 4 + codes[k]]);
        } else {
            double s = orc_f16_to_f64(w->scale[n * ng + j]);
            out[k] = ((double)codes[k] - (double)w->zp[n * ng + j]) * s;
        }
    }
    if (w->nnz > 0)
        for (int32_t p = w->row_ptr[n]; p < w->row_ptr[n + 1]; p++)
            out[w->col[p]] += orc_f16_to_f64(w->val[p]);
}

int orc_dequant_rows(const orc_qweight *w, int64_t n0, int64_t n1, double *out)
{
    if (n0 < 0 || n1 > w->N || n0 > n1) return ORC_EINVAL;
    uint8_t *codes = (uint8_t *)malloc((size_t)w->K);
    if (!codes) return ORC_ENOMEM;
    for (int64_t n = n0; n < n1; n++) dequant_row(w, n, codes, out + (n - n0) * w->K);
    free(codes);
    return ORC_OK;
}

/* y[m, n - n0] = sum_k x[m, k] * (x_hat[n, k] + S[n, k]) for n in [n0, n1),
 * x bf16 [M, K] with row stride ldx, accumulated in fp64 in ascending k. */
int orc_linear_rows(const uint16_t *x, int64_t M, int64_t ldx, const orc_qweight *w,
                    int64_t n0, int64_t n1, double *y)
{
    if (n0 < 0 || n1 > w->N || n0 > n1 || ldx < w->K) return ORC_EINVAL;
    int64_t K = w->K, nn = n1 - n0;
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K));
    uint8_t *codes = (uint8_t *)malloc((size_t)K);
    if (!row || !xd || !codes) {
        free(row); free(xd); free(codes);
        return ORC_ENOMEM;
    }
    for (int64_t m = 0; m < M; m++)
        for (int64_t k = 0; k < K; k++) xd[m * K + k] = orc_bf16_to_f64(x[m * ldx + k]);
    for (int64_t n = n0; n < n1; n++) {
        dequant_row(w, n, codes, row);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) acc += xd[m * K + k] * row[k];
            y[m * nn + (n - n0)] = acc;
        }
    }
    free(row); free(xd); free(codes);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* per-layer quantization diagnostics                                   */
/* ------------------------------------------------------------------ */

/* Diagnostics of one quantized layer ("Mixed-width quantization" page,
 * section 6.1: unpack the quantized weights and compare them element by
 * element with the original fp16 weights -- maximum absolute error, root
 * mean square error, cosine similarity; section 6.2: the "dynamic range
 * ratio" of a block, its largest value over its second largest, flags
 * blocks that hold one extreme value).
 *   e[n,k] = w[n,k] - (x_hat[n,k] + S[n,k]) over all N*K elements (the
 *   layer's effective weight includes the FP16 outliers added back);
 *   out[0] = max |e|, out[1] = sqrt(sum e^2 / (N*K)),
 *   out[2] = sum w*v / (|w| |v|) with v = x_hat + S (1 if both norms are 0,
 *   0 if only one is), out[3] = largest group ratio,
 *   out[4] = number of groups whose ratio exceeds `threshold`.
 * ratio[n*ng + j] (may be NULL) = max |w| / second largest |w| over the
 * group's elements (magnitudes, counted with multiplicity): 1 for an
 * all-zero group, +infinity when exactly one element is nonzero.
 * Everything in fp64, in ascending element order. */
int orc_diagnostics(const uint16_t *W, const orc_qweight *q, double threshold, double *out, double *ratio)
{
    int64_t N = q->N, K = q->K, g = q->group, ng = K / g;
    double *v = (double *)malloc(sizeof(double) * (size_t)K);
    uint8_t *codes = (uint8_t *)malloc((size_t)K);
    if (!v || !codes) {
        free(v); free(codes);
        return ORC_ENOMEM;
    }
    double emax = 0.0, se = 0.0, sww = 0.0, svv = 0.0, swv = 0.0, rmax = 0.0, over = 0.0;
    for (int64_t n = 0; n < N; n++) {
        dequant_row(q, n, codes, v);
        for (int64_t j = 0; j < ng; j++) {
            double m1 = 0.0, m2 = 0.0;
            for (int64_t i = j * g; i < (j + 1) * g; i++) {
                double w = orc_f16_to_f64(W[n * K + i]);
                double e = w - v[i];
                if (fabs(e) > emax) emax = fabs(e);
                se += e * e;
                sww += w * w;
                svv += v[i] * v[i];
                swv += w * v[i];
                double a = fabs(w);
                if (a > m1) {
                    m2 = m1;
                    m1 = a;
                } else if (a > m2) {
                    m2 = a;
                }
            }
            double r = m1 == 0.0 ? 1.0 : (m2 == 0.0 ? INFINITY : m1 / m2);
            if (ratio) ratio[n * ng + j] = r;
            if (r > rmax) rmax = r;
            if (r > threshold) over += 1.0;
        }
    }
    out[0] = emax;
    out[1] = sqrt(se / (double)(N * K));
    out[2] = (sww == 0.0 && svv == 0.0) ? 1.0 : (sww == 0.0 || svv == 0.0) ? 0.0 : swv / (sqrt(sww) * sqrt(svv));
    out[3] = rmax;
    out[4] = over;
    free(v); free(codes);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* W8A8: int8 weights and int8 activations                              */
/* ------------------------------------------------------------------ */

/* Dynamic per-token activation quantizer ("Inference acceleration guide"
 * page, section 1.2: W8A8 quantizes the activations as well, dynamically
 * per token; section 1.1: the symmetric INT8 range [-127, 127]).  For token
 * m: s[m] = max_k |x[m,k]| / 127 in fp32 (1 if the maximum is 0),
 * q[m,k] = clamp(round(x[m,k] / s[m]), -127, 127), fp32 division, round half
 * to even. */
int orc_quantize_act_int8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int8_t *q, float *s)
{
    for (int64_t m = 0; m < M; m++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float a = fabsf((float)orc_bf16_to_f64(x[m * ldx + k]));
            if (a > amax) amax = a;
        }
        float sm = amax == 0.0f ? 1.0f : amax / 127.0f;
        for (int64_t k = 0; k < K; k++) {
            float v = rintf((float)orc_bf16_to_f64(x[m * ldx + k]) / sm);
            if (v < -127.0f) v = -127.0f;
            if (v > 127.0f) v = 127.0f;
            q[m * K + k] = (int8_t)v;
        }
        s[m] = sm;
    }
    return ORC_OK;
}

/* y[m, n - n0] = sum_k (q[m,k] * s[m]) * (x_hat[n,k] + S[n,k]) in fp64: the
 * product of the quantized activations with the layer's weight. */
int orc_linear_w8a8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const orc_qweight *w, int64_t n0,
                    int64_t n1, double *y)
{
    if (n0 < 0 || n1 > w->N || n0 > n1 || ldx < w->K || K != w->K) return ORC_EINVAL;
    int8_t *q = (int8_t *)malloc((size_t)(M * K));
    float *s = (float *)malloc(sizeof(float) * (size_t)M);
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    uint8_t *codes = (uint8_t *)malloc((size_t)K);
    if (!q || !s || !row || !codes) {
        free(q); free(s); free(row); free(codes);
        return ORC_ENOMEM;
    }
    orc_quantize_act_int8(x, M, K, ldx, q, s);
    int64_t nn = n1 - n0;
    for (int64_t n = n0; n < n1; n++) {
        dequant_row(w, n, codes, row);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) acc += ((double)q[m * K + k] * (double)s[m]) * row[k];
            y[m * nn + (n - n0)] = acc;
        }
    }
    free(q); free(s); free(row); free(codes);
    return ORC_OK;
}
