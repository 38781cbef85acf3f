/*
 * ks_oracle.c -- the CPU oracle for row-wise RMSNorm and the fused residual-add RMSNorm, and for
 * the next operators of the same library: SwiGLU (silu_and_mul), Softmax and LayerNorm.
 *
 * TEST INFRASTRUCTURE. This file is the plain, slow, single-threaded definition that the CUDA
 * path is checked against. Only the test suite, the smoke check and the CPU-baseline leg of
 * bench.py may load it. It shares no code, header, table or helper with the CUDA library: the
 * casts, the reciprocal square root and the row loops below are written out here on their own.
 *
 * Build flags matter: it must be compiled with -ffp-contract=off -fno-fast-math so that every
 * statement rounds exactly once, in the order written (no fused multiply-add, no reassociation).
 *
 * What it follows (Kernscope, "Numerical contract"):
 *   RMSNorm:   x32 = fp32(x); scale = rsqrt(mean(x32^2 over the last axis) + eps);
 *              out = cast_to_input_dtype(x32 * scale * fp32(weight)); FP32 intermediates.
 *   Fused:     s = fp32(x_in) + fp32(residual_in); residual = cast(s);
 *              x = cast(s * rsqrt(mean(s^2) + eps) * fp32(weight)), normalising the FP32 s
 *              before it is rounded for storage.
 * Readings taken where the contract is silent (each also listed in the design notes):
 *   - the sum of squares runs left to right in fp32, each square rounded before it is added;
 *   - mean = ss / fp32(H), one IEEE division by the real width H (the TileLang-Ascend data path
 *     of the same page divides by hidden_size, not by the padded width);
 *   - rsqrt is the correctly rounded fp32 value of 1/sqrt(v);
 *   - the product is evaluated left to right: (x32 * scale) * fp32(weight);
 *   - cast_to_input_dtype rounds to nearest, ties to even; overflow gives +-inf; NaN stays NaN.
 *
 * A float64 twin of each op (the same steps in double, one rounding at the end, done by the
 * caller) serves as the high-precision reference the fp32 path is pinned against.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element-type codes used by this file only. */
enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* ------------------------------------------------------------------------------------------ */
/* Decoding: every fp16 and bf16 value is exactly representable in fp32 and in double.         */
/* ------------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32 word. */
static double decode_bf16(uint16_t b) {
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* zero or subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double decode_f32(uint32_t w) {
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int64_t i, int dtype) {
    switch (dtype) {
    case ORACLE_BF16: return decode_bf16(((const uint16_t *)base)[i]);
    case ORACLE_F16: return decode_f16(((const uint16_t *)base)[i]);
    default: return decode_f32(((const uint32_t *)base)[i]);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Encoding: round a double to the nearest value of a binary floating-point format, ties to    */
/* even (IEEE 754 roundTiesToEven), then write its bit pattern.                                 */
/* ------------------------------------------------------------------------------------------ */

/* Format parameters: p significand bits (including the hidden bit), smallest normal exponent
 * emin, largest exponent emax. */
static void format_params(int dtype, int *p, int *emin, int *emax) {
    switch (dtype) {
    case ORACLE_BF16: *p = 8; *emin = -126; *emax = 127; break;
    case ORACLE_F16: *p = 11; *emin = -14; *emax = 15; break;
    default: *p = 24; *emin = -126; *emax = 127; break;
    }
}

/* Returns the representable value nearest to v (ties to even), or +-inf past the overflow
 * threshold. Near v the representable values are the integer multiples of the quantum
 * q = 2^(max(exponent(v), emin) - (p - 1)); v / q is exact because q is a power of two, and
 * nearbyint() in the default rounding mode rounds half to even. */
static double round_to_format(double v, int dtype) {
    int p, emin, emax;
    format_params(dtype, &p, &emin, &emax);
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e2;
    frexp(fabs(v), &e2); /* |v| = f * 2^e2 with f in [0.5, 1): leading bit has exponent e2-1 */
    int lead = e2 - 1;
    if (lead < emin) lead = emin; /* subnormal range: the quantum stops shrinking */
    double q = ldexp(1.0, lead - (p - 1));
    double r = nearbyint(v / q) * q;
    double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > max_finite) return copysign(INFINITY, v);
    return r;
}

static uint16_t encode_bf16_exact(double r) {
    /* r is already a bf16 value (or +-inf / NaN): its fp32 word has a zero lower half. */
    if (isnan(r)) return 0x7FC0;
    float f = (float)r;
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(w >> 16);
}

static uint16_t encode_f16_exact(double r) {
    if (isnan(r)) return (uint16_t)(signbit(r) ? 0xFE00 : 0x7E00);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) { /* subnormal: a = m * 2^-24 */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    }
    int e2;
    frexp(a, &e2);
    int lead = e2 - 1;                                       /* a in [2^lead, 2^(lead+1)) */
    uint32_t m = (uint32_t)(a / ldexp(1.0, lead - 10)) - 1024; /* exact: a has <= 11 bits */
    return sign | (uint16_t)((uint32_t)(lead + 15) << 10) | (uint16_t)m;
}

static uint32_t encode_f32_exact(double r) {
    float f = (float)r; /* exact: r is already an fp32 value */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return w;
}

static void store_elem(void *base, int64_t i, int dtype, double v) {
    double r = round_to_format(v, dtype);
    switch (dtype) {
    case ORACLE_BF16: ((uint16_t *)base)[i] = encode_bf16_exact(r); break;
    case ORACLE_F16: ((uint16_t *)base)[i] = encode_f16_exact(r); break;
    default: ((uint32_t *)base)[i] = encode_f32_exact(r); break;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Correctly rounded fp32 reciprocal square root.                                              */
/* ------------------------------------------------------------------------------------------ */

/* Sign of (m*m*v - 1), computed exactly. m is the midpoint of two adjacent positive floats, so
 * it has at most 25 significant bits and m*m (at most 50 bits) is exact in double. The product
 * with v is split into hi + lo exactly with one fused multiply-add; rounding is monotone and 1
 * is representable, so hi alone decides unless hi == 1. */
static int sign_msq_v_minus_1(double m, float v) {
    double p = m * m;
    double hi = p * (double)v;
    double lo = fma(p, (double)v, -hi);
    if (hi < 1.0) return -1;
    if (hi > 1.0) return 1;
    return (lo < 0.0) ? -1 : (lo > 0.0 ? 1 : 0);
}

static int mantissa_is_even(float a) {
    uint32_t w;
    memcpy(&w, &a, sizeof w);
    return (w & 1u) == 0;
}

/* Nearest fp32 value to 1/sqrt(v), ties to even. For a > 0 the exact value 1/sqrt(v) is above
 * the midpoint m of two neighbours exactly when m*m*v < 1, so the double-precision estimate is
 * moved one float at a time until both neighbouring midpoints bracket the exact value. */
static float rsqrt_rn(float v) {
    if (isnan(v) || v < 0.0f) return NAN;
    if (v == 0.0f) return INFINITY;
    if (isinf(v)) return 0.0f;
    float r = (float)(1.0 / sqrt((double)v));
    for (;;) {
        float up = nextafterf(r, INFINITY);
        double m = 0.5 * ((double)r + (double)up);
        int c = sign_msq_v_minus_1(m, v);
        if (c < 0 || (c == 0 && mantissa_is_even(up))) r = up;
        else break;
    }
    for (;;) {
        float dn = nextafterf(r, 0.0f);
        double m = 0.5 * ((double)r + (double)dn);
        int c = sign_msq_v_minus_1(m, v);
        if (c > 0 || (c == 0 && mantissa_is_even(dn))) r = dn;
        else break;
    }
    return r;
}

/* ------------------------------------------------------------------------------------------ */
/* The fp32 contract path.                                                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * RMSNorm over `rows` rows of width H (row-major, contiguous), Kernscope "Numerical contract /
 * RMSNorm". y may be exactly x (each row is fully read before it is written). If u is not
 * NULL it receives the fp32 value of each output before the final cast.
 */
void oracle_rms_norm(const void *x, const void *w, void *y, float *u, int64_t rows, int64_t H,
                     float eps, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        float ss = 0.0f;
        for (int64_t j = 0; j < H; ++j) {
            float v = (float)load_elem(x, base + j, dtype);
            float sq = v * v;
            ss = ss + sq;
        }
        float mean = ss / (float)H;
        float scale = rsqrt_rn(mean + eps);
        for (int64_t j = 0; j < H; ++j) {
            float v = (float)load_elem(x, base + j, dtype);
            float t = v * scale;
            float o = t * (float)load_elem(w, j, dtype);
            if (u) u[base + j] = o;
            store_elem(y, base + j, dtype, (double)o);
        }
    }
}

/*
 * Fused residual-add RMSNorm, in place on x and residual, Kernscope "Numerical contract / Fused
 * residual-add RMSNorm": s = fp32(x) + fp32(r) (one fp32 add); r <- cast(s); x <- cast of the
 * normalised *unrounded* s times fp32(weight). Returns 0, or -1 if the row buffer could not be
 * allocated.
 */
int oracle_fused_add_rms_norm(void *x, void *r, const void *w, float *u, int64_t rows,
                              int64_t H, float eps, int dtype) {
    float *s = (float *)malloc((size_t)H * sizeof(float));
    if (!s) return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        float ss = 0.0f;
        for (int64_t j = 0; j < H; ++j) {
            float xv = (float)load_elem(x, base + j, dtype);
            float rv = (float)load_elem(r, base + j, dtype);
            s[j] = xv + rv;
            float sq = s[j] * s[j];
            ss = ss + sq;
        }
        for (int64_t j = 0; j < H; ++j) store_elem(r, base + j, dtype, (double)s[j]);
        float mean = ss / (float)H;
        float scale = rsqrt_rn(mean + eps);
        for (int64_t j = 0; j < H; ++j) {
            float t = s[j] * scale;
            float o = t * (float)load_elem(w, j, dtype);
            if (u) u[base + j] = o;
            store_elem(x, base + j, dtype, (double)o);
        }
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* The float64 twin: the same steps in double, unrounded results returned to the caller.      */
/* ------------------------------------------------------------------------------------------ */

void oracle_rms_norm_f64(const void *x, const void *w, double *yd, int64_t rows, int64_t H,
                         double eps, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double v = load_elem(x, base + j, dtype);
            ss += v * v;
        }
        double scale = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t j = 0; j < H; ++j)
            yd[base + j] = load_elem(x, base + j, dtype) * scale * load_elem(w, j, dtype);
    }
}

/* sd receives the double sum x + r (exact for 16-bit inputs), yd the normalised output. */
void oracle_fused_add_rms_norm_f64(const void *x, const void *r, const void *w, double *yd,
                                   double *sd, int64_t rows, int64_t H, double eps, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double s = load_elem(x, base + j, dtype) + load_elem(r, base + j, dtype);
            sd[base + j] = s;
            ss += s * s;
        }
        double scale = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t j = 0; j < H; ++j) yd[base + j] = sd[base + j] * scale * load_elem(w, j, dtype);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* The next operators of the same library (Kernscope, "Numerical contract": SwiGLU activation,  */
/* Softmax; kernel-set, "Operators": LayerNorm, named only).                                   */
/* ------------------------------------------------------------------------------------------ */

/* fp32 exp, read as the correctly rounded value of e^v: exp in double rounded once to fp32 (a
 * double rounding could differ only within 2^-29 of a midpoint). */
static float exp_rn(float v) { return (float)exp((double)v); }

/*
 * SwiGLU, Kernscope "Numerical contract / SwiGLU activation": for x of shape [rows, 2d],
 * gate = fp32(x[:, :d]), up = fp32(x[:, d:]), out = cast(gate * sigmoid(gate) * up), FP32
 * intermediates. Read as sigmoid(g) = 1 / (1 + exp(-g)) and the products left to right:
 * ((g * sigmoid(g)) * up). u (optional) receives the fp32 value before the cast.
 */
void oracle_silu_and_mul(const void *x, void *out, float *u, int64_t rows, int64_t d, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < d; ++j) {
            float g = (float)load_elem(x, i * 2 * d + j, dtype);
            float up = (float)load_elem(x, i * 2 * d + d + j, dtype);
            float e = exp_rn(-g);
            float den = 1.0f + e;
            float sig = 1.0f / den;
            float a = g * sig;
            float o = a * up;
            if (u) u[i * d + j] = o;
            store_elem(out, i * d + j, dtype, (double)o);
        }
    }
}

/*
 * Softmax over the last axis, Kernscope "Numerical contract / Softmax":
 * z = fp32(x) - max(fp32(x)); out = cast(exp(z) / sum(exp(z))). The maximum propagates NaN (as
 * the reference's torch.softmax does), which yields the stated non-finite rules literally: a row
 * with NaN or +inf, or a row that is all -inf, comes out NaN; -inf entries of a row with finite
 * values come out 0. The sum runs left to right in fp32.
 */
void oracle_softmax(const void *x, void *out, float *u, int64_t rows, int64_t H, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        float m = -INFINITY;
        int nan = 0;
        for (int64_t j = 0; j < H; ++j) {
            float v = (float)load_elem(x, base + j, dtype);
            if (isnan(v)) nan = 1;
            else if (v > m) m = v;
        }
        if (nan) m = NAN;
        float sum = 0.0f;
        for (int64_t j = 0; j < H; ++j) {
            float z = (float)load_elem(x, base + j, dtype) - m;
            sum = sum + exp_rn(z);
        }
        for (int64_t j = 0; j < H; ++j) {
            float z = (float)load_elem(x, base + j, dtype) - m;
            float o = exp_rn(z) / sum;
            if (u) u[base + j] = o;
            store_elem(out, base + j, dtype, (double)o);
        }
    }
}

/*
 * LayerNorm over the last axis (named on kernel-set's operator list; the contract is read as the
 * standard definition with the RMSNorm contract's FP32 discipline): mean = sum(x)/H, var =
 * sum((x - mean)^2)/H (two passes, population variance), rstd = rsqrt(var + eps), and
 * out = cast((((x - mean) * rstd) * w) + b), every step one fp32 rounding, sums left to right.
 * w and b may be NULL (then 1 and 0).
 */
void oracle_layer_norm(const void *x, const void *w, const void *b, void *out, float *u,
                       int64_t rows, int64_t H, float eps, int dtype) {
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t base = i * H;
        float s = 0.0f;
        for (int64_t j = 0; j < H; ++j) s = s + (float)load_elem(x, base + j, dtype);
        float mean = s / (float)H;
        float q = 0.0f;
        for (int64_t j = 0; j < H; ++j) {
            float dlt = (float)load_elem(x, base + j, dtype) - mean;
            float sq = dlt * dlt;
            q = q + sq;
        }
        float var = q / (float)H;
        float rstd = rsqrt_rn(var + eps);
        for (int64_t j = 0; j < H; ++j) {
            float dlt = (float)load_elem(x, base + j, dtype) - mean;
            float t = dlt * rstd;
            if (w) t = t * (float)load_elem(w, j, dtype);
            if (b) t = t + (float)load_elem(b, j, dtype);
            if (u) u[base + j] = t;
            store_elem(out, base + j, dtype, (double)t);
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Array helpers exposed for the pins.                                                         */
/* ------------------------------------------------------------------------------------------ */

void oracle_decode(const void *src, double *dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dtype);
}

void oracle_encode(const double *src, void *dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) store_elem(dst, i, dtype, src[i]);
}

void oracle_rsqrt(const float *v, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = rsqrt_rn(v[i]);
}

/* Bumped whenever the arithmetic above changes, so stale builds are detected. */
int oracle_version(void) { return 2; }
