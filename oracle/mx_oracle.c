/*
 * mx_oracle.c -- plain, slow CPU oracle for block-scaled quantization and the
 * block-scaled matrix products that consume it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; every value here is derived from the format definitions.
 *
 * Arithmetic is done in double unless the method fixes FP32 (the NVFP4 and
 * DeepSeek scale recipes are FP32 by definition, so those steps use float,
 * in the literal order the pages write them, with IEEE division).
 *
 * Sources (cited by page title and section):
 *  [MX]   "MXFP8 on SM120: software support" (xuesongtap.github.io), sec 0.1
 *         (format table, E8M0, q = Q(x/s), 64-element example) and sec 0.3
 *         (block-scaled dot product y = sum_b sA_b sB_b sum_i qA qB).
 *  [DS]   "Why FP8 training is stable: scale granularity and accumulation
 *         precision" (magicnetworld.com, DeepSeek-V3 FP8), sec 4 (s = amax/MAX,
 *         x_hat = s Q(x/s)), sec 5 (1x128 activation tiles, 128x128 weight
 *         blocks), sec 5.1 (worked tile), sec 6.3 (FP32 promotion every 128).
 *  [NV]   "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 2.4 (E2M1
 *         values), sec 3.2 (0.7 -> 0.5), sec 5.4 (two-level scale recipe),
 *         sec 5.5 (MXFP4: E2M1 elements, 32-element blocks, one E8M0 scale),
 *         sec 5.6 (worked example), sec 7.1-7.4 (scale outside the sum, W4A4).
 *
 * Readings where the pages are silent:
 *  - E4M3 bias 7 / E5M2 bias 15 / E2M1 bias 1: the biases reproduce the
 *    printed max and min-subnormal values exactly.
 *  - Rounding is round-to-nearest, ties to the even code; results above the
 *    format maximum saturate to +-max ("satfinite"); +-Inf saturates; NaN maps
 *    to the positive NaN code 0x7F (E4M3 / E5M2).  E2M1 has no NaN code: the
 *    NVFP4 path is defined for finite inputs only.
 *  - The sign of zero is kept (-0 encodes as 0x80 / 0x8).
 *  - MX scale: k = floor(log2 amax) - emax, clamped to [-127, 127]; amax == 0
 *    gives k = -127.  A NaN or Inf anywhere in a block makes the block scale
 *    the E8M0 NaN code 0xFF and every code of that block 0x7F (E2M1 blocks of
 *    MXFP4: 0x7, the largest positive code; the NaN scale already marks the
 *    block, so these element codes are unpinned).
 *  - NVFP4: amax == 0 gives a global scale of 1.0; a block whose E4M3 scale
 *    code rounds to 0 gets all-zero element codes.  Element 2i is stored in the
 *    low nibble of byte i.
 *  - DeepSeek: amax == 0 gives s = 1.0.
 *
 * Parity pins: see tests/test_oracle_*.py (printed values from the pages,
 * brute-force nearest-code search, exhaustive decode, closed forms).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FMT_E4M3 0
#define FMT_E5M2 1
#define FMT_E2M1 2
#define FMT_E8M0 3

/* ---------------------------------------------------------------------- */
/* format parameters, written from the bit-field definitions              */
/* ---------------------------------------------------------------------- */
typedef struct {
    int exp_bits;   /* exponent field width */
    int man_bits;   /* mantissa field width */
    int bias;       /* exponent bias */
    double maxval;  /* largest finite magnitude */
} fmt_t;

static fmt_t fmt_of(int fmt) {
    fmt_t f;
    if (fmt == FMT_E4M3) {        /* 1-4-3, no Inf, S.1111.111 = NaN        */
        f.exp_bits = 4; f.man_bits = 3; f.bias = 7;  f.maxval = 448.0;
    } else if (fmt == FMT_E5M2) { /* 1-5-2, IEEE-style Inf/NaN              */
        f.exp_bits = 5; f.man_bits = 2; f.bias = 15; f.maxval = 57344.0;
    } else {                      /* E2M1: 1-2-1, no Inf/NaN                */
        f.exp_bits = 2; f.man_bits = 1; f.bias = 1;  f.maxval = 6.0;
    }
    return f;
}

int orc_emax(int fmt) {
    /* exponent of the largest finite value: 448 = 1.75*2^8, 57344 = 1.75*2^15,
       6 = 1.5*2^2 */
    fmt_t f = fmt_of(fmt);
    int e; frexp(f.maxval, &e);
    return e - 1;
}

/* decode one code to its exact value (NaN as NAN, Inf as INFINITY) */
double orc_decode(int fmt, uint32_t code) {
    if (fmt == FMT_E8M0) {
        code &= 0xFF;
        if (code == 0xFF) return NAN;
        return ldexp(1.0, (int)code - 127);
    }
    fmt_t f = fmt_of(fmt);
    int nbits = 1 + f.exp_bits + f.man_bits;
    code &= (1u << nbits) - 1;
    int sign = (code >> (nbits - 1)) & 1;
    int e = (code >> f.man_bits) & ((1 << f.exp_bits) - 1);
    int m = code & ((1 << f.man_bits) - 1);
    int emask = (1 << f.exp_bits) - 1;
    double v;
    if (fmt == FMT_E5M2 && e == emask) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (fmt == FMT_E4M3 && e == emask && m == (1 << f.man_bits) - 1) {
        v = NAN;
    } else if (e == 0) {
        /* subnormal: 0.m * 2^(1-bias) */
        v = ldexp((double)m, 1 - f.bias - f.man_bits);
    } else {
        v = ldexp((double)((1 << f.man_bits) + m), e - f.bias - f.man_bits);
    }
    return sign ? -v : v;
}

/* bits of an exactly representable non-negative magnitude a <= maxval */
static uint32_t magnitude_bits(fmt_t f, double a) {
    if (a == 0.0) return 0;
    double min_normal = ldexp(1.0, 1 - f.bias);
    if (a < min_normal) {
        /* subnormal: a = m * 2^(1-bias-man_bits) */
        double m = ldexp(a, -(1 - f.bias - f.man_bits));
        return (uint32_t)m;
    }
    int e2; double fr = frexp(a, &e2); /* a = fr * 2^e2, fr in [0.5,1) */
    int e = e2 - 1;                     /* a = (2fr) * 2^e, 2fr in [1,2) */
    double man = (2.0 * fr - 1.0) * (double)(1 << f.man_bits);
    return ((uint32_t)(e + f.bias) << f.man_bits) | (uint32_t)man;
}

/* round-half-even of a non-negative double n to an integer-valued double */
static double rne(double n) {
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5) return r + 1.0;
    if (frac < 0.5) return r;
    return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;
}

/* encode a real value: nearest representable, ties to even, satfinite */
uint32_t orc_encode(int fmt, double v) {
    fmt_t f = fmt_of(fmt);
    int nbits = 1 + f.exp_bits + f.man_bits;
    uint32_t sbit = 1u << (nbits - 1);
    if (isnan(v)) {
        if (fmt == FMT_E2M1) return 0x7; /* no NaN code: unpinned, saturate */
        return 0x7F;
    }
    uint32_t sign = signbit(v) ? sbit : 0;
    double a = fabs(v);
    if (a >= f.maxval) return sign | magnitude_bits(f, f.maxval); /* incl. Inf */
    /* quantum (spacing of representable values) at a's binade */
    double min_normal = ldexp(1.0, 1 - f.bias);
    double quantum;
    if (a < min_normal) {
        quantum = ldexp(1.0, 1 - f.bias - f.man_bits);
    } else {
        int e2; frexp(a, &e2);
        quantum = ldexp(1.0, (e2 - 1) - f.man_bits);
    }
    double n = a / quantum;       /* exact: quantum is a power of two */
    double r = rne(n) * quantum;  /* may step up into the next binade */
    if (r > f.maxval) r = f.maxval;
    return sign | magnitude_bits(f, r);
}

/* brute force: nearest code by scanning every finite code; ties -> even code.
   Used only to pin orc_encode. */
uint32_t orc_encode_bruteforce(int fmt, double v) {
    fmt_t f = fmt_of(fmt);
    int nbits = 1 + f.exp_bits + f.man_bits;
    uint32_t ncodes = 1u << nbits;
    uint32_t best = 0xFFFFFFFFu;
    double bestd = INFINITY;
    double a = fabs(v);
    int neg = signbit(v) ? 1 : 0;
    if (isnan(v)) return (fmt == FMT_E2M1) ? 0x7 : 0x7F;
    if (a > f.maxval) a = f.maxval; /* saturation */
    for (uint32_t c = 0; c < ncodes; ++c) {
        if ((c >> (nbits - 1)) & 1) continue;  /* magnitudes only */
        double d = orc_decode(fmt, c);
        if (!isfinite(d)) continue;
        double dist = fabs(d - a);
        if (dist < bestd || (dist == bestd && (c & 1) == 0)) { bestd = dist; best = c; }
    }
    return best | (neg ? (1u << (nbits - 1)) : 0);
}

/* bf16 bit pattern -> exact double */
double orc_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float fl; memcpy(&fl, &u, 4);
    return (double)fl;
}

static float bf16f(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float fl; memcpy(&fl, &u, 4);
    return fl;
}

/* ---------------------------------------------------------------------- */
/* MX (OCP) block quantization, [MX] sec 0.1                              */
/* ---------------------------------------------------------------------- */

/* shared exponent k for a block with maximum magnitude amax (finite) */
int orc_mx_scale_exp(double amax, int fmt) {
    if (amax == 0.0) return -127;
    int e2; frexp(amax, &e2);          /* amax in [2^(e2-1), 2^e2) */
    int k = (e2 - 1) - orc_emax(fmt);  /* floor(log2 amax) - emax */
    if (k < -127) k = -127;
    if (k > 127) k = 127;
    return k;
}

/* quantize one block of n values given as doubles (strided source) */
static void mx_block(const uint16_t* x, int64_t stride, int n, int fmt,
                     uint8_t* q, int64_t qstride, uint8_t* s) {
    double amax = 0.0; int bad = 0;
    for (int i = 0; i < n; ++i) {
        double v = orc_bf16(x[i * stride]);
        if (!isfinite(v)) bad = 1;
        else if (fabs(v) > amax) amax = fabs(v);
    }
    if (bad) {
        *s = 0xFF;
        for (int i = 0; i < n; ++i) q[i * qstride] = (fmt == FMT_E2M1) ? 0x7 : 0x7F;
        return;
    }
    int k = orc_mx_scale_exp(amax, fmt);
    *s = (uint8_t)(k + 127);
    for (int i = 0; i < n; ++i) {
        double v = orc_bf16(x[i * stride]);
        q[i * qstride] = (uint8_t)orc_encode(fmt, ldexp(v, -k)); /* x / 2^k exact */
    }
}

/* row-wise: 1x32 blocks along each row.
   x[rows][cols] bf16 -> q[rows][cols], s[rows][cols/32] (plain layout).
   fmt E4M3 / E5M2 is MXFP8, E2M1 is MXFP4 ([NV] sec 5.5); codes are returned
   one per byte (unpacked) for every format. */
void orc_mx_quantize_rowwise(const uint16_t* x, int64_t rows, int64_t cols, int fmt,
                             uint8_t* q, uint8_t* s) {
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            mx_block(x + r * cols + b * 32, 1, 32, fmt, q + r * cols + b * 32, 1,
                     s + r * nb + b);
}

/* column-wise: 32x1 blocks down each column, stored transposed.
   x[rows][cols] -> qT[cols][rows], sT[cols][rows/32] */
void orc_mx_quantize_colwise(const uint16_t* x, int64_t rows, int64_t cols, int fmt,
                             uint8_t* qT, uint8_t* sT) {
    int64_t nb = rows / 32;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c)
        for (int64_t b = 0; b < nb; ++b)
            mx_block(x + (b * 32) * cols + c, cols, 32, fmt, qT + c * rows + b * 32, 1,
                     sT + c * nb + b);
}

/* row-wise MX quantization of FP32 values (a GEMM's FP32 results quantized
   for the next product): the rule of mx_block on float input.
   x[rows][cols] float -> q[rows][cols], s[rows][cols/32] (plain layout) */
void orc_mx_quantize_rowwise_f32(const float* x, int64_t rows, int64_t cols, int fmt,
                                 uint8_t* q, uint8_t* s) {
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float* xb = x + r * cols + b * 32;
            double amax = 0.0; int bad = 0;
            for (int i = 0; i < 32; ++i) {
                double v = (double)xb[i];
                if (!isfinite(v)) bad = 1;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            if (bad) {
                s[r * nb + b] = 0xFF;
                for (int i = 0; i < 32; ++i) q[r * cols + b * 32 + i] = (uint8_t)((fmt == FMT_E2M1) ? 0x7 : 0x7F);
                continue;
            }
            int k = orc_mx_scale_exp(amax, fmt);
            s[r * nb + b] = (uint8_t)(k + 127);
            for (int i = 0; i < 32; ++i)
                q[r * cols + b * 32 + i] = (uint8_t)orc_encode(fmt, ldexp((double)xb[i], -k));
        }
}

/* ---------------------------------------------------------------------- */
/* DeepSeek fine-grained FP8 quantization, [DS] sec 4 and sec 5           */
/* s = fl32(amax / 448), q = E4M3(fl32(x / s))                             */
/* ---------------------------------------------------------------------- */
float orc_ds_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    volatile float s = amax / 448.0f;
    return s;
}

uint8_t orc_ds_encode(float x, float s) {
    volatile float y = x / s;
    return (uint8_t)orc_encode(FMT_E4M3, (double)y);
}

/* 1x128 tiles: x[rows][cols] -> q[rows][cols], s[rows][cols/128] (plain) */
void orc_ds_quantize_1x128(const uint16_t* x, int64_t rows, int64_t cols,
                           uint8_t* q, float* s) {
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16f(x[r * cols + b * 128 + i]));
                if (a > amax) amax = a;
            }
            float sc = orc_ds_scale(amax);
            s[r * nb + b] = sc;
            for (int i = 0; i < 128; ++i)
                q[r * cols + b * 128 + i] = orc_ds_encode(bf16f(x[r * cols + b * 128 + i]), sc);
        }
}

/* 128x128 blocks: x[rows][cols] -> q[rows][cols], s[rows/128][cols/128] */
void orc_ds_quantize_128x128(const uint16_t* x, int64_t rows, int64_t cols,
                             uint8_t* q, float* s) {
    int64_t nbr = rows / 128, nbc = cols / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t br = 0; br < nbr; ++br)
        for (int64_t bc = 0; bc < nbc; ++bc) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    float a = fabsf(bf16f(x[(br * 128 + i) * cols + bc * 128 + j]));
                    if (a > amax) amax = a;
                }
            float sc = orc_ds_scale(amax);
            s[br * nbc + bc] = sc;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t o = (br * 128 + i) * cols + bc * 128 + j;
                    q[o] = orc_ds_encode(bf16f(x[o]), sc);
                }
        }
}

/* ---------------------------------------------------------------------- */
/* Float8BlockScaling with power-of-two scales and its MX form, [MX] sec  */
/* 1.3: on Blackwell the 1x128 / 128x128 recipe's FP32 scales are powers   */
/* of two, so each converts to an E8M0 code; a 128-block's scale serves    */
/* its four 32-blocks unchanged and a 2-D block's scale is broadcast to    */
/* every row; the FP8 codes are reused as they are.                        */
/* Reading (the page does not give the rounding of the scale): s = 2^k,    */
/* k the smallest integer with 448 * 2^k >= amax (no element saturates),   */
/* clamped to [-127, 127]; amax == 0 gives s = 1.  q = E4M3(x / s), exact. */
/* ---------------------------------------------------------------------- */
int orc_pow2_scale_exp(double amax) {
    if (amax == 0.0) return 0;
    int k = -127;
    while (k < 127 && ldexp(448.0, k) < amax) ++k;   /* linear search, no shortcuts */
    return k;
}

/* 1x128 tiles with power-of-two scales: q[rows][cols], s[rows][cols/128] (plain) */
void orc_ds_quantize_1x128_pow2(const uint16_t* x, int64_t rows, int64_t cols,
                                uint8_t* q, float* s) {
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int i = 0; i < 128; ++i) {
                double a = fabs(orc_bf16(x[r * cols + b * 128 + i]));
                if (a > amax) amax = a;
            }
            int k = orc_pow2_scale_exp(amax);
            s[r * nb + b] = (float)ldexp(1.0, k);
            for (int i = 0; i < 128; ++i)
                q[r * cols + b * 128 + i] =
                    (uint8_t)orc_encode(FMT_E4M3, ldexp(orc_bf16(x[r * cols + b * 128 + i]), -k));
        }
}

/* 128x128 blocks with power-of-two scales: q[rows][cols], s[rows/128][cols/128] */
void orc_ds_quantize_128x128_pow2(const uint16_t* x, int64_t rows, int64_t cols,
                                  uint8_t* q, float* s) {
    int64_t nbr = rows / 128, nbc = cols / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t br = 0; br < nbr; ++br)
        for (int64_t bc = 0; bc < nbc; ++bc) {
            double amax = 0.0;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    double a = fabs(orc_bf16(x[(br * 128 + i) * cols + bc * 128 + j]));
                    if (a > amax) amax = a;
                }
            int k = orc_pow2_scale_exp(amax);
            s[br * nbc + bc] = (float)ldexp(1.0, k);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t o = (br * 128 + i) * cols + bc * 128 + j;
                    q[o] = (uint8_t)orc_encode(FMT_E4M3, ldexp(orc_bf16(x[o]), -k));
                }
        }
}

/* E8M0 code of an FP32 scale: k + 127 when the scale is exactly 2^k with
   -127 <= k <= 127, otherwise the E8M0 NaN code 0xFF */
uint8_t orc_e8m0_of_scale(float sc) {
    double v = (double)sc;
    if (!(v > 0.0) || isinf(v)) return 0xFF;
    int e; double m = frexp(v, &e);              /* v = m 2^e, m in [0.5, 1) */
    if (m != 0.5) return 0xFF;
    int k = e - 1;
    if (k < -127 || k > 127) return 0xFF;
    return (uint8_t)(k + 127);
}

/* Expand block scales into per-32 MX scales of the [rows][cols] code matrix:
   block_rows 1:   s[rows][cols/128] (1x128 tiles),
   block_rows 128: s[rows/128][cols/128] (128x128 blocks);
   out[rows][cols/32] E8M0 codes (plain layout). */
void orc_mx_scales_from_blocks(const float* s, int64_t rows, int64_t cols, int block_rows,
                               uint8_t* out) {
    int64_t nb = cols / 32, nbc = cols / 128;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            float sc = (block_rows == 1) ? s[r * nbc + b / 4] : s[(r / 128) * nbc + b / 4];
            out[r * nb + b] = orc_e8m0_of_scale(sc);
        }
}

/* 2-D 32x32 MX blocks ([MX] sec 1.3): one E8M0 scale per 32x32 block by the
   MX rule over the whole block; codes q[rows][cols]; scales s[rows/32][cols/32].
   The row-wise MX form uses s[r/32][b] for row r, block b; the column-wise
   (transposed) form is the transpose of q with s[b][c/32]. */
void orc_mx_quantize_2d32(const uint16_t* x, int64_t rows, int64_t cols, int fmt,
                          uint8_t* q, uint8_t* s) {
    int64_t nbr = rows / 32, nbc = cols / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t br = 0; br < nbr; ++br)
        for (int64_t bc = 0; bc < nbc; ++bc) {
            double amax = 0.0; int bad = 0;
            for (int i = 0; i < 32; ++i)
                for (int j = 0; j < 32; ++j) {
                    double v = orc_bf16(x[(br * 32 + i) * cols + bc * 32 + j]);
                    if (!isfinite(v)) bad = 1;
                    else if (fabs(v) > amax) amax = fabs(v);
                }
            int k = orc_mx_scale_exp(amax, fmt);
            s[br * nbc + bc] = bad ? 0xFF : (uint8_t)(k + 127);
            for (int i = 0; i < 32; ++i)
                for (int j = 0; j < 32; ++j) {
                    int64_t o = (br * 32 + i) * cols + bc * 32 + j;
                    q[o] = bad ? (uint8_t)((fmt == FMT_E2M1) ? 0x7 : 0x7F)
                               : (uint8_t)orc_encode(fmt, ldexp(orc_bf16(x[o]), -k));
                }
        }
}

/* ---------------------------------------------------------------------- */
/* NVFP4 two-level quantization, [NV] sec 5.4 and 5.6                     */
/* ---------------------------------------------------------------------- */
float orc_nv_global_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    volatile float sg = amax / (448.0f * 6.0f);  /* 448*6 = 2688 exactly */
    return sg;
}

/* block scale for one 16-element block with magnitude bamax:
   t = (bamax / 6) / s_g, code = E4M3(t) (positive), s_hat = dec(code) * s_g */
uint8_t orc_nv_block_scale(float sg, float bamax, float* s_hat) {
    volatile float t0 = bamax / 6.0f;
    volatile float t = t0 / sg;
    uint8_t code = (uint8_t)orc_encode(FMT_E4M3, (double)t);
    volatile float sh = (float)orc_decode(FMT_E4M3, code) * sg;
    *s_hat = sh;
    return code;
}

uint8_t orc_nv_encode(float x, float s_hat) {
    if (s_hat == 0.0f) return 0;
    volatile float y = x / s_hat;
    return (uint8_t)orc_encode(FMT_E2M1, (double)y);
}

float orc_nv_amax(const uint16_t* x, int64_t n) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16f(x[i]));
        if (a > amax) amax = a;
    }
    return amax;
}

/* x[rows][cols] -> qp[rows][cols/2] (element 2i low nibble), s[rows][cols/16]
   E4M3 codes (plain), *sg = global FP32 scale */
void orc_nv_quantize(const uint16_t* x, int64_t rows, int64_t cols,
                     uint8_t* qp, uint8_t* s, float* sg_out) {
    float sg = orc_nv_global_scale(orc_nv_amax(x, rows * cols));
    *sg_out = sg;
    int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* xb = x + r * cols + b * 16;
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(bf16f(xb[i]));
                if (a > bamax) bamax = a;
            }
            float sh;
            s[r * nb + b] = orc_nv_block_scale(sg, bamax, &sh);
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = orc_nv_encode(bf16f(xb[i]), sh);
                uint8_t hi = orc_nv_encode(bf16f(xb[i + 1]), sh);
                qp[r * (cols / 2) + b * 8 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
}

/* ---------------------------------------------------------------------- */
/* NVFP4 training options, [DS] sec 13 ("from FP8 to 4 bits": a 16x16     */
/* random Hadamard transform, stochastic rounding, 16x16 2-D weight       */
/* blocks) and [NV] sec 3.2 (stochastic rounding: round up or down with   */
/* probability set by the distance, E[Q(x) - x] = 0).                      */
/* Readings (the pages give no formulas beyond these):                     */
/*  - the transform acts on every 1x16 block along the reduction axis:     */
/*    v = 0.25 * H16 * (d .* x), d_i = -1 where bit i of a 16-bit sign     */
/*    mask is set, H16 the Sylvester Hadamard matrix; in FP32 with the    */
/*    butterfly order h = 1, 2, 4, 8 below (both sides use this order);    */
/*    the NVFP4 recipe then runs on v (global amax included);              */
/*  - stochastic rounding takes one random byte r per element (an input):  */
/*    for a = |fl32(v / s_hat)| below 6 with E2M1 neighbours lo <= a < hi, */
/*    round up iff r < floor(256 * (a - lo) / (hi - lo)); a >= 6 gives 6;  */
/*    so E[Q] - a lies in (-(hi - lo)/256, 0] and is 0 when 256 (a - lo)  */
/*    / (hi - lo) is an integer;                                           */
/*  - 2-D blocks: the block maximum runs over 16x16 elements; W and W^T    */
/*    then hold the same codes and scales.                                 */
/* ---------------------------------------------------------------------- */
void orc_fwht16_f32(float v[16], uint32_t signs) {
    for (int i = 0; i < 16; ++i)
        if ((signs >> i) & 1u) v[i] = -v[i];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int i = 0; i < 16; ++i) v[i] *= 0.25f;
}

/* E2M1 code of a by stochastic rounding with random byte r (sign from y) */
uint8_t orc_e2m1_stochastic(float y, uint8_t r) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(y) ? 0x8 : 0x0;
    double a = fabs((double)y);
    int lo = 0;
    if (a >= 6.0) return (uint8_t)(sign | 7);
    while (lo < 6 && grid[lo + 1] <= a) ++lo;        /* grid[lo] <= a < grid[lo + 1] */
    double frac = (a - grid[lo]) / (grid[lo + 1] - grid[lo]);
    int up = (double)r < floor(256.0 * frac);
    return (uint8_t)(sign | (lo + up));
}

/* NVFP4 quantization with the options above on x[rows][cols]:
   rht != 0 applies the transform to every 1x16 block first; rbits != NULL
   switches the element codes to stochastic rounding (rbits[rows][cols]).
   Codes unpacked q[rows][cols] (4-bit values), block scales s[rows][cols/16]
   (E4M3 codes), the global scale in *sg_out. */
void orc_nv_quantize_ex(const uint16_t* x, int64_t rows, int64_t cols, int rht, uint32_t signs,
                        const uint8_t* rbits, uint8_t* q, uint8_t* s, float* sg_out) {
    int64_t nb = cols / 16;
    float* v = (float*)malloc(sizeof(float) * (size_t)(rows * cols));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            float blk[16];
            for (int i = 0; i < 16; ++i) blk[i] = bf16f(x[r * cols + b * 16 + i]);
            if (rht) orc_fwht16_f32(blk, signs);
            for (int i = 0; i < 16; ++i) v[r * cols + b * 16 + i] = blk[i];
        }
    float amax = 0.0f;
    for (int64_t i = 0; i < rows * cols; ++i)
        if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
    float sg = orc_nv_global_scale(amax);
    *sg_out = sg;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float* vb = v + r * cols + b * 16;
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i)
                if (fabsf(vb[i]) > bamax) bamax = fabsf(vb[i]);
            float sh;
            s[r * nb + b] = orc_nv_block_scale(sg, bamax, &sh);
            for (int i = 0; i < 16; ++i) {
                int64_t o = r * cols + b * 16 + i;
                if (!rbits) {
                    q[o] = orc_nv_encode(vb[i], sh);
                } else if (sh == 0.0f) {
                    q[o] = 0;
                } else {
                    volatile float y = vb[i] / sh;
                    q[o] = orc_e2m1_stochastic(y, rbits[o]);
                }
            }
        }
    free(v);
}

/* NVFP4 with 16x16 2-D blocks: codes q[rows][cols] (unpacked), block scales
   s[rows/16][cols/16] (E4M3 codes), global scale *sg_out */
void orc_nv_quantize_2d16(const uint16_t* x, int64_t rows, int64_t cols,
                          uint8_t* q, uint8_t* s, float* sg_out) {
    float sg = orc_nv_global_scale(orc_nv_amax(x, rows * cols));
    *sg_out = sg;
    int64_t nbr = rows / 16, nbc = cols / 16;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t br = 0; br < nbr; ++br)
        for (int64_t bc = 0; bc < nbc; ++bc) {
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float a = fabsf(bf16f(x[(br * 16 + i) * cols + bc * 16 + j]));
                    if (a > bamax) bamax = a;
                }
            float sh;
            s[br * nbc + bc] = orc_nv_block_scale(sg, bamax, &sh);
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    int64_t o = (br * 16 + i) * cols + bc * 16 + j;
                    q[o] = orc_nv_encode(bf16f(x[o]), sh);
                }
        }
}

/* ---------------------------------------------------------------------- */
/* Reference products in double.                                          */
/* C[m][n] = sum_k A[m][k] B[n][k]; both operands K-contiguous.            */
/* Each returns out[i][n] and absum[i][n] = sum_k |a_k b_k| for the rows   */
/* listed in rows_idx (nrows of them).                                     */
/* ---------------------------------------------------------------------- */

/* MX: y = sum_b sA_b sB_b sum_{i<32} qA qB   ([MX] sec 0.3); element formats
   E4M3, E5M2 or E2M1 (MXFP4), codes one per byte */
void orc_mx_gemm(const uint8_t* qa, const uint8_t* sa, int fa,
                 const uint8_t* qb, const uint8_t* sb, int fb,
                 int64_t M, int64_t N, int64_t K,
                 const int64_t* rows_idx, int64_t nrows,
                 double* out, double* absum) {
    (void)M;
    int64_t nb = K / 32;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows_idx[i];
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0, ab = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double part = 0.0, apart = 0.0;
                for (int64_t j = b * 32; j < b * 32 + 32; ++j) {
                    double p = orc_decode(fa, qa[m * K + j]) * orc_decode(fb, qb[n * K + j]);
                    part += p;
                    apart += fabs(p);
                }
                double scale = orc_decode(FMT_E8M0, sa[m * nb + b]) *
                               orc_decode(FMT_E8M0, sb[n * nb + b]);
                y += scale * part;
                ab += scale * apart;
            }
            out[i * N + n] = y;
            absum[i * N + n] = ab;
        }
    }
}

/* NVFP4: y = sgA sgB sum_b sA_b sB_b sum_{i<16} qA qB   ([NV] sec 7.3, 7.4) */
void orc_nv_gemm(const uint8_t* qa, const uint8_t* sa, float sga,
                 const uint8_t* qb, const uint8_t* sb, float sgb,
                 int64_t M, int64_t N, int64_t K,
                 const int64_t* rows_idx, int64_t nrows,
                 double* out, double* absum) {
    (void)M;
    int64_t nb = K / 16;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows_idx[i];
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0, ab = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double part = 0.0, apart = 0.0;
                for (int64_t j = b * 16; j < b * 16 + 16; ++j) {
                    uint8_t ba = qa[m * (K / 2) + j / 2], bb = qb[n * (K / 2) + j / 2];
                    uint8_t ca = (j & 1) ? (ba >> 4) : (ba & 0xF);
                    uint8_t cb = (j & 1) ? (bb >> 4) : (bb & 0xF);
                    double p = orc_decode(FMT_E2M1, ca) * orc_decode(FMT_E2M1, cb);
                    part += p;
                    apart += fabs(p);
                }
                double scale = orc_decode(FMT_E4M3, sa[m * nb + b]) *
                               orc_decode(FMT_E4M3, sb[n * nb + b]);
                y += scale * part;
                ab += scale * apart;
            }
            double g = (double)sga * (double)sgb;
            out[i * N + n] = g * y;
            absum[i * N + n] = g * ab;
        }
    }
}

/* DeepSeek: y = sum_kb sA[m][kb] sB[n/128][kb] sum_{k in kb} qA qB,
   sa plain [M][K/128], sb plain [N/128][K/128]   ([DS] sec 6.3) */
void orc_ds_gemm(const uint8_t* qa, const float* sa,
                 const uint8_t* qb, const float* sb,
                 int64_t M, int64_t N, int64_t K,
                 const int64_t* rows_idx, int64_t nrows,
                 double* out, double* absum) {
    (void)M;
    int64_t nb = K / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows_idx[i];
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0, ab = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double part = 0.0, apart = 0.0;
                for (int64_t j = b * 128; j < b * 128 + 128; ++j) {
                    double p = orc_decode(FMT_E4M3, qa[m * K + j]) * orc_decode(FMT_E4M3, qb[n * K + j]);
                    part += p;
                    apart += fabs(p);
                }
                double scale = (double)sa[m * nb + b] * (double)sb[(n / 128) * nb + b];
                y += scale * part;
                ab += fabs(scale) * apart;
            }
            out[i * N + n] = y;
            absum[i * N + n] = ab;
        }
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
