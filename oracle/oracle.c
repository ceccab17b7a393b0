/*
 * CPU oracle for the fused Gemma add-RMSNorm + FP8 / NVFP4 input quantization.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * CPU-baseline leg of the benchmark; never by the product path.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Everything here is written to be checked by eye against the pages:
 *   - number formats are encoded by exhaustive nearest search over their
 *     finite codes (ties to the even code), not by bit tricks;
 *   - the norm is evaluated in fp64; only the steps whose precision the pages
 *     fix are done in fp32 (the fp32 accumulation of partials, the residual
 *     add, and the quantizers' scale arithmetic, which the fused op must share
 *     with the standalone quantizers);
 *   - every step is one loop in the order the method states it.
 *
 * Build: plain C11, -ffp-contract=off (no fused multiply-add may merge two
 * roundings), optional -fopenmp for the row loop.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static int g_threads = 1;

void or_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int or_get_threads(void) { return g_threads; }

/* ------------------------------------------------------------------------ */
/* 16-bit activation formats                                                 */
/*   bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                   */
/*   fp16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                   */
/* ------------------------------------------------------------------------ */
typedef struct {
    int frac_bits; /* stored fraction bits                        */
    int exp_bits;
    int bias;
} fmt16;

static fmt16 fmt_of(int dtype) {
    fmt16 f;
    if (dtype == OR_BF16) {
        f.frac_bits = 7; f.exp_bits = 8; f.bias = 127;
    } else {
        f.frac_bits = 10; f.exp_bits = 5; f.bias = 15;
    }
    return f;
}

/* Exact value of a 16-bit pattern (every bf16/fp16 value is a double). */
double or_decode16(uint16_t bits, int dtype) {
    fmt16 f = fmt_of(dtype);
    int sign = (bits >> 15) & 1;
    int e = (bits >> f.frac_bits) & ((1 << f.exp_bits) - 1);
    int frac = bits & ((1 << f.frac_bits) - 1);
    int emax_field = (1 << f.exp_bits) - 1;
    double v;
    if (e == emax_field) {
        v = frac ? NAN : INFINITY;
    } else if (e == 0) { /* subnormal: frac * 2^(1 - bias - frac_bits) */
        v = ldexp((double)frac, 1 - f.bias - f.frac_bits);
    } else {             /* normal: (2^frac_bits + frac) * 2^(e - bias - frac_bits) */
        v = ldexp((double)((1 << f.frac_bits) + frac), e - f.bias - f.frac_bits);
    }
    return sign ? -v : v;
}

/* Round-to-nearest-even of a double onto the 16-bit format, overflow to inf.
 * The spacing of representable values at |v| is 2^(E - frac_bits) with E the
 * binade of |v| (never below the minimum normal exponent, which gives the
 * subnormals); rint() rounds the scaled value to the nearest integer, ties to
 * even, which is ties-to-even on the significand. */
uint16_t or_round16(double v, int dtype) {
    fmt16 f = fmt_of(dtype);
    int emin = 1 - f.bias;
    int emax = (1 << f.exp_bits) - 2 - f.bias;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) /* quiet NaN: exponent all ones, top fraction bit set */
        return (uint16_t)((((1u << f.exp_bits) - 1u) << f.frac_bits) | (1u << (f.frac_bits - 1)));
    double a = fabs(v);
    uint16_t inf_bits = (uint16_t)(((1u << f.exp_bits) - 1u) << f.frac_bits);
    if (isinf(a)) return sign | inf_bits;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;         /* binade: 2^E <= a < 2^(E+1)  */
    if (E < emin) E = emin; /* subnormal spacing            */
    double ulp = ldexp(1.0, E - f.frac_bits);
    double n = rint(a / ulp); /* exact scaling by a power of two, then RNE */
    double r = n * ulp;
    double max_finite = ldexp((double)((2 << f.frac_bits) - 1), emax - f.frac_bits);
    if (r > max_finite) return sign | inf_bits;
    /* encode the representable value r */
    if (r < ldexp(1.0, emin)) { /* subnormal (or zero) */
        uint16_t frac = (uint16_t)(r / ldexp(1.0, emin - f.frac_bits));
        return sign | frac;
    }
    frexp(r, &e2);
    int Er = e2 - 1;
    uint16_t frac = (uint16_t)(r / ldexp(1.0, Er - f.frac_bits) - (double)(1 << f.frac_bits));
    uint16_t ef = (uint16_t)(Er + f.bias);
    return sign | (uint16_t)(ef << f.frac_bits) | frac;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 fraction bits;    */
/* no infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448.        */
/* ------------------------------------------------------------------------ */
double or_e4m3_value(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int frac = code & 0x7;
    double v;
    if (e == 0xF && frac == 0x7) return NAN;
    if (e == 0) v = ldexp((double)frac, -9);            /* frac/8 * 2^(1-7) */
    else        v = ldexp((double)(8 + frac), e - 10);  /* (1+frac/8) * 2^(e-7) */
    return sign ? -v : v;
}

static double e4m3_magnitudes[0x7F]; /* value of each finite non-negative code */
static int e4m3_ready = 0;

static void e4m3_init(void) {
    if (e4m3_ready) return;
    for (int c = 0; c <= 0x7E; ++c) e4m3_magnitudes[c] = or_e4m3_value((uint8_t)c);
    e4m3_ready = 1;
}

/* Nearest finite E4M3 value, ties to the even code, saturating: anything
 * beyond 448 in magnitude (infinity included) becomes +-448; NaN stays NaN.
 * The sign of the input is kept, also when the magnitude rounds to zero. */
uint8_t or_e4m3_encode(double v) {
    e4m3_init();
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v)) return 0x7F | sign;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E; /* saturate (infinity included) */
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) { /* all finite non-negative codes */
        double d = fabs(e4m3_magnitudes[c] - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------ */
/* FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 fraction bit; all 16 codes are   */
/* finite: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.                            */
/* ------------------------------------------------------------------------ */
double or_e2m1_value(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 0x3;
    int frac = code & 0x1;
    double v;
    if (e == 0) v = 0.5 * frac;                         /* subnormal: frac/2 * 2^0 */
    else        v = ldexp(1.0 + 0.5 * frac, e - 1);     /* (1+frac/2) * 2^(e-1)  */
    return sign ? -v : v;
}

/* Nearest E2M1 value, ties to the even code, saturating at +-6; sign kept.
 * Saturation is taken before the search: for huge |v| every distance rounds
 * to the same double and the search alone would not find the largest code. */
uint8_t or_e2m1_encode(double v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 0x7; /* saturate (infinity included) */
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7; ++c) {
        double d = fabs(or_e2m1_value((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* E8M0: a bare biased exponent, value 2^(code - 127); 0xFF is NaN. */
double or_e8m0_value(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* ------------------------------------------------------------------------ */
/* 128x4 swizzled scale layout.  The (Mp, Kp) scale matrix, Mp = round_up(M,  */
/* 128), Kp = round_up(H/16, 4), is stored as tiles of 128 rows x 4 columns,  */
/* tile-major along k; inside a tile, rows m%32 are the outer index (16 B     */
/* apart), then (m%128)/32 (4 B apart), then k%4.                             */
/* ------------------------------------------------------------------------ */
int64_t or_swizzle_offset(int64_t m, int64_t k, int64_t Kp) {
    int64_t tile = (m / 128) * (Kp / 4) + k / 4;
    return tile * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4 + k % 4;
}

/* ------------------------------------------------------------------------ */
/* Quantizers, each applied to one row of the normed activation y (given as  */
/* fp32 values, all exactly representable since y is bf16/fp16).            */
/* ------------------------------------------------------------------------ */

/* Static per-tensor FP8: q = e4m3_satfinite(y / s), the division in fp32. */
static void quant_row_fp8(const float *yf, int64_t H, float s, uint8_t *q) {
    for (int64_t j = 0; j < H; ++j) {
        float v = yf[j] / s;
        q[j] = or_e4m3_encode((double)v);
    }
}

/* Element scale of an NVFP4 block: the global scale over the stored block
 * scale, one fp32 division; an all-zero block (stored scale 0) gets 0. */
static float nvfp4_element_scale(float g, uint8_t sf) {
    float sfv = (float)or_e4m3_value(sf);
    return sfv == 0.0f ? 0.0f : g / sfv;
}

/* NVFP4: per block of 16 elements, block scale sf = e4m3(g * (amax / 6)),
 * codes c = e2m1(y * (g / sf)), two codes per byte, the lower-indexed element
 * in the low nibble.  The scale byte of block b of row m is stored at the
 * swizzled offset. */
static void quant_row_nvfp4(const float *yf, int64_t m, int64_t H, float g,
                            uint8_t *q, uint8_t *block_scale) {
    int64_t B = H / 16;
    int64_t Kp = (B + 3) / 4 * 4;
    for (int64_t b = 0; b < B; ++b) {
        float amax = 0.0f;
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(yf[16 * b + j]));
        float sf32 = g * (amax / 6.0f);
        uint8_t sf = or_e4m3_encode((double)sf32);
        float es = nvfp4_element_scale(g, sf);
        uint8_t c[16];
        for (int j = 0; j < 16; ++j) {
            float v = yf[16 * b + j] * es;
            c[j] = or_e2m1_encode((double)v);
        }
        for (int i = 0; i < 8; ++i)
            q[8 * b + i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
        block_scale[or_swizzle_offset(m, b, Kp)] = sf;
    }
}

/* MXFP8 (OCP microscaling): per block of 32 elements, the shared scale is
 * X = 2^(floor(log2(amax)) - 8), 8 being the exponent of E4M3's largest
 * binade; it is stored as the E8M0 code floor(log2(amax)) - 8 + 127, clamped
 * to [0, 254] (an all-zero block gets code 0; an infinite amax, whose
 * floor(log2) is +inf, the top code 254).  Elements are
 * e4m3_satfinite(y / X), exact scaling by a power of two.  Scales are stored
 * row-major, (M, H/32). */
static void quant_row_mxfp8(const float *yf, int64_t H, uint8_t *q,
                            uint8_t *scale_row) {
    int64_t B = H / 32;
    for (int64_t b = 0; b < B; ++b) {
        double amax = 0.0;
        for (int j = 0; j < 32; ++j) amax = fmax(amax, fabs((double)yf[32 * b + j]));
        int code;
        if (amax == 0.0) {
            code = 0;
        } else if (isinf(amax)) {
            code = 254;
        } else {
            int e2;
            frexp(amax, &e2);
            code = (e2 - 1) - 8 + 127;
            if (code < 0) code = 0;
            if (code > 254) code = 254;
        }
        scale_row[b] = (uint8_t)code;
        double X = or_e8m0_value((uint8_t)code);
        for (int j = 0; j < 32; ++j)
            q[32 * b + j] = or_e4m3_encode((double)yf[32 * b + j] / X);
    }
}

static int check_mode_shape(int mode, int64_t H) {
    if (mode == OR_MODE_NVFP4 && H % 16 != 0) return -1;
    if (mode == OR_MODE_MXFP8 && H % 32 != 0) return -1;
    if (mode < OR_MODE_NONE || mode > OR_MODE_MXFP8) return -1;
    return 0;
}

static void quantize_row(const float *yf, int64_t m, int64_t M, int64_t H,
                         float scale, int mode, uint8_t *q, uint8_t *bs) {
    (void)M;
    if (mode == OR_MODE_FP8) {
        quant_row_fp8(yf, H, scale, q + m * H);
    } else if (mode == OR_MODE_NVFP4) {
        quant_row_nvfp4(yf, m, H, scale, q + m * (H / 2), bs);
    } else if (mode == OR_MODE_MXFP8) {
        quant_row_mxfp8(yf, H, q + m * H, bs + m * (H / 32));
    }
}

/* ------------------------------------------------------------------------ */
/* The method, one row at a time.                                            */
/* ------------------------------------------------------------------------ */
int or_gemma_add_rms_norm_quant(const uint16_t *x, int k, int64_t part_stride,
                                uint16_t *residual, const uint16_t *w,
                                float eps, float weight_bias, float scale,
                                int mode, uint8_t *q, uint8_t *block_scale,
                                uint16_t *y, int64_t M, int64_t H, int dtype) {
    if (M < 0 || H <= 0 || k < 1 || !x || !w) return -1;
    if (dtype != OR_BF16 && dtype != OR_FP16) return -1;
    if (check_mode_shape(mode, H)) return -1;
    if (mode == OR_MODE_NONE && !y) return -1;
    if (mode != OR_MODE_NONE && !q) return -1;
    if ((mode == OR_MODE_NVFP4 || mode == OR_MODE_MXFP8) && !block_scale) return -1;
    e4m3_init(); /* fill the code table before any thread reads it */

#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t m = 0; m < M; ++m) {
        uint16_t *h = (uint16_t *)malloc((size_t)H * sizeof(uint16_t));
        float *yf = (float *)malloc((size_t)H * sizeof(float));

        /* 1. The activation: one buffer, or k partials summed in fp32 in
         *    index order and rounded once to the activation dtype. */
        for (int64_t j = 0; j < H; ++j) {
            if (k == 1) {
                h[j] = x[m * H + j];
            } else {
                float acc = (float)or_decode16(x[m * H + j], dtype);
                for (int p = 1; p < k; ++p)
                    acc = acc + (float)or_decode16(x[p * part_stride + m * H + j], dtype);
                h[j] = or_round16((double)acc, dtype);
            }
        }

        /* 2. Residual add (fp32, rounded to the activation dtype); the
         *    residual buffer receives the sum in place. */
        if (residual) {
            for (int64_t j = 0; j < H; ++j) {
                float s = (float)or_decode16(h[j], dtype) +
                          (float)or_decode16(residual[m * H + j], dtype);
                h[j] = or_round16((double)s, dtype);
                residual[m * H + j] = h[j];
            }
        }

        /* 3. inv = 1 / sqrt(mean(h^2) + eps), in fp64. */
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double hv = or_decode16(h[j], dtype);
            ss += hv * hv;
        }
        double inv = 1.0 / sqrt(ss / (double)H + (double)eps);

        /* 4. y = dtype(h * inv * (weight_bias + w)), in fp64, one rounding. */
        for (int64_t j = 0; j < H; ++j) {
            double hv = or_decode16(h[j], dtype);
            double wv = or_decode16(w[j], dtype);
            uint16_t yb = or_round16(hv * inv * ((double)weight_bias + wv), dtype);
            if (y) y[m * H + j] = yb;
            yf[j] = (float)or_decode16(yb, dtype);
        }

        /* 5. Quantize the rounded y. */
        quantize_row(yf, m, M, H, scale, mode, q, block_scale);

        free(h);
        free(yf);
    }
    return 0;
}

int or_quantize_from_y(const uint16_t *y, float scale, int mode, uint8_t *q,
                       uint8_t *block_scale, int64_t M, int64_t H, int dtype) {
    if (M < 0 || H <= 0 || !y || !q) return -1;
    if (mode == OR_MODE_NONE || check_mode_shape(mode, H)) return -1;
    if ((mode == OR_MODE_NVFP4 || mode == OR_MODE_MXFP8) && !block_scale) return -1;
    e4m3_init();
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t m = 0; m < M; ++m) {
        float *yf = (float *)malloc((size_t)H * sizeof(float));
        for (int64_t j = 0; j < H; ++j) yf[j] = (float)or_decode16(y[m * H + j], dtype);
        quantize_row(yf, m, M, H, scale, mode, q, block_scale);
        free(yf);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Element-wise array forms of the format routines, for the test suite.      */
/* ------------------------------------------------------------------------ */
void or_decode16_array(const uint16_t *bits, double *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_decode16(bits[i], dtype);
}
void or_round16_array(const double *v, uint16_t *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_round16(v[i], dtype);
}
void or_e4m3_encode_array(const double *v, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_encode(v[i]);
}
void or_e2m1_encode_array(const double *v, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e2m1_encode(v[i]);
}
