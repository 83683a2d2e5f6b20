/*
 * oracle.c -- slow, plain CPU oracle for the fused residual-add + normalization
 * family (SkipSimplifiedLayerNormalization, GatedRMSNorm, SkipGroupNorm).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path; its binary16 conversion below is written from the IEEE 754-2008
 * binary16 definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction
 * bits, round-to-nearest-ties-to-even).
 *
 * Arithmetic contract (what every function below reproduces):
 *  - The residual sum S is formed in binary32, in the order (x + skip) + bias,
 *    and rounded ONCE to the tensor type T.  An absent bias is no add at all.
 *    ("The sum is rounded to the tensor type before the statistics see it",
 *    com.microsoft.SkipGroupNorm README, Description.)
 *  - Statistics and the normalized value are evaluated in binary64 from the
 *    T-rounded S (or X), then rounded once, to nearest-even, to T.
 *  - Build with -ffp-contract=off so that no fused multiply-add changes a
 *    binary32 sum; FLT_EVAL_METHOD must be 0 (x86-64 SSE, AArch64).
 *
 * Element type codes: 0 = float32, 1 = float16, 2 = bfloat16 (both 16-bit
 * types stored as uint16 bit patterns).  bfloat16 is not among the pages'
 * types; its conversion below is written from the format's definition (the
 * upper half of a binary32: 1 sign bit, 8 exponent bits with bias 127,
 * 7 fraction bits), rounding to nearest, ties to even.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 arithmetic evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary64, from the format definition.              */
/* ------------------------------------------------------------------------ */

/* Exact value of a binary16 pattern. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);            /* subnormal or zero: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

float orc_f16_to_f32(uint16_t h) {
    /* Every binary16 value is exactly representable in binary32. */
    return (float)orc_f16_to_f64(h);
}

/* Round a binary64 value to the nearest binary16, ties to even. */
uint16_t orc_f64_to_f16(double d) {
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    if (isnan(d)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(d);
    /* Largest finite binary16 is 65504 = (2 - 2^-10) * 2^15; the midpoint to
     * the next step (65536) is 65520 and ties go to the even neighbour, which
     * is 65536, i.e. overflow. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);            /* a = m * 2^E, m in [0.5, 1): unbiased exponent E-1 */
    int unb = E - 1;
    int q;                   /* exponent of one unit in the last place */
    if (unb < -14) q = -24;  /* subnormal range: fixed quantum 2^-24 */
    else q = unb - 10;
    double scaled = ldexp(a, -q);         /* exact: power-of-two scaling */
    double fl = floor(scaled);
    double frac = scaled - fl;            /* exact: scaled < 2^12 */
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    uint32_t ri = (uint32_t)r;
    uint32_t bits;
    if (unb < -14) {
        /* Subnormal: the pattern is the integer itself; ri == 1024 carries
         * into the smallest normal (exponent field 1, fraction 0). */
        bits = ri;
    } else {
        /* Normal: ri in [1024, 2048]; 2048 carries into the next binade. */
        bits = ((uint32_t)(unb + 15) << 10) + (ri - 1024);
    }
    if (bits >= 0x7c00) bits = 0x7c00;
    return (uint16_t)(sign | bits);
}

uint16_t orc_f32_to_f16(float f) {
    /* binary32 -> binary64 is exact, so this is a single rounding. */
    return orc_f64_to_f16((double)f);
}

void orc_f64_to_f16_array(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f16(in[i]);
}
void orc_f32_to_f16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(in[i]);
}
void orc_f16_to_f32_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary64, from the format definition.                        */
/* ------------------------------------------------------------------------ */

/* Exact value of a bfloat16 pattern. */
double orc_bf16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);            /* subnormal or zero: f * 2^-133 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1.f) * 2^(e-127) */
    }
    return sign ? -v : v;
}

float orc_bf16_to_f32(uint16_t h) {
    /* Every bfloat16 value is exactly representable in binary32. */
    return (float)orc_bf16_to_f64(h);
}

/* Round a binary64 value to the nearest bfloat16, ties to even. */
uint16_t orc_f64_to_bf16(double d) {
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    if (isnan(d)) return (uint16_t)(sign | 0x7fc0);
    double a = fabs(d);
    /* Largest finite bfloat16 is (2 - 2^-7) * 2^127; the midpoint to the next
     * step (2^128) is (2 - 2^-8) * 2^127, and a tie goes to the even
     * neighbour, 2^128, i.e. overflow. */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7f80);
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);            /* a = m * 2^E, m in [0.5, 1): unbiased exponent E-1 */
    int unb = E - 1;
    int q;                   /* exponent of one unit in the last place */
    if (unb < -126) q = -133; /* subnormal range: fixed quantum 2^-133 */
    else q = unb - 7;
    double scaled = ldexp(a, -q);         /* exact: power-of-two scaling */
    double fl = floor(scaled);
    double frac = scaled - fl;            /* exact: scaled < 2^9 */
    const int odd = fmod(fl, 2.0) != 0.0;
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && odd)) r = fl + 1.0;
    uint32_t ri = (uint32_t)r;
    uint32_t bits;
    if (unb < -126) {
        /* Subnormal: the pattern is the integer itself; ri == 128 carries
         * into the smallest normal (exponent field 1, fraction 0). */
        bits = ri;
    } else {
        /* Normal: ri in [128, 256]; 256 carries into the next binade. */
        bits = ((uint32_t)(unb + 127) << 7) + (ri - 128);
    }
    if (bits >= 0x7f80) bits = 0x7f80;
    return (uint16_t)(sign | bits);
}

uint16_t orc_f32_to_bf16(float f) {
    /* binary32 -> binary64 is exact, so this is a single rounding. */
    return orc_f64_to_bf16((double)f);
}

void orc_f64_to_bf16_array(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(in[i]);
}
void orc_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}
void orc_bf16_to_f32_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Element access                                                            */
/* ------------------------------------------------------------------------ */

static float ld_f32(const void* p, int dtype, int64_t i) {
    if (dtype == ORC_F16) return orc_f16_to_f32(((const uint16_t*)p)[i]);
    if (dtype == ORC_BF16) return orc_bf16_to_f32(((const uint16_t*)p)[i]);
    return ((const float*)p)[i];
}

/* Store a binary64 value at type T, rounding once to nearest-even. */
static void st_from_f64(void* p, int dtype, int64_t i, double v) {
    if (dtype == ORC_F16) ((uint16_t*)p)[i] = orc_f64_to_f16(v);
    else if (dtype == ORC_BF16) ((uint16_t*)p)[i] = orc_f64_to_bf16(v);
    else ((float*)p)[i] = (float)v;  /* C conversion rounds to nearest-even */
}

/* The residual sum at type T, returned as its exact value.
 * (x + skip) in binary32, then + bias in binary32 when a bias is present,
 * then one rounding to T.  SkipGroupNorm README, Description; the same
 * reading is applied to SkipSimplifiedLayerNormalization. */
static double residual_sum(float x, float skip, const void* bias, int dtype,
                           int64_t bias_index, void* s_out, int64_t s_index) {
    float t = x + skip;
    if (bias) t = t + ld_f32(bias, dtype, bias_index);
    double s;
    if (dtype == ORC_F16) {
        uint16_t h = orc_f32_to_f16(t);
        s = orc_f16_to_f64(h);
        if (s_out) ((uint16_t*)s_out)[s_index] = h;
    } else if (dtype == ORC_BF16) {
        uint16_t h = orc_f32_to_bf16(t);
        s = orc_bf16_to_f64(h);
        if (s_out) ((uint16_t*)s_out)[s_index] = h;
    } else {
        s = (double)t;
        if (s_out) ((float*)s_out)[s_index] = t;
    }
    return s;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* com.microsoft.SkipSimplifiedLayerNormalization                           */
/* README, Description / Inputs / Outputs / Attributes:                      */
/*   S = input + skip (+ bias);  output = S / sqrt(mean(S^2) + epsilon) * gamma */
/*   over the last axis of length hidden; input_skip_bias_sum = S.           */
/*   mean (U=f32) is 0 for the simplified form; inv_std_var is the inverse RMS.*/
/* ------------------------------------------------------------------------ */
int orc_skip_rms(const void* input, const void* skip, const void* gamma,
                 const void* bias, void* output, void* sum_out,
                 float* mean_out, float* inv_std_out,
                 int64_t rows, int64_t hidden, int dtype, float epsilon) {
    if (rows < 0 || hidden <= 0) return 1;
    double* srow = (double*)malloc((size_t)hidden * sizeof(double));
    if (!srow) return 2;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            int64_t i = r * hidden + j;
            double s = residual_sum(ld_f32(input, dtype, i), ld_f32(skip, dtype, i),
                                    bias, dtype, j, sum_out, i);
            srow[j] = s;
            ss += s * s;
        }
        double ms = ss / (double)hidden;
        double inv = 1.0 / sqrt(ms + (double)epsilon);
        for (int64_t j = 0; j < hidden; ++j) {
            double y = srow[j] * inv * (double)ld_f32(gamma, dtype, j);
            st_from_f64(output, dtype, r * hidden + j, y);
        }
        if (mean_out) mean_out[r] = 0.0f;
        if (inv_std_out) inv_std_out[r] = (float)inv;
    }
    free(srow);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* com.microsoft.GatedRMSNorm README, Description:                           */
/*   Y = X * rsqrt(mean(X^2) + epsilon) * scale * SiLU(gate), the mean taken  */
/*   over each contiguous span of C = numel(scale) elements; rows = numel/C. */
/*   SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)).                            */
/* ------------------------------------------------------------------------ */
int orc_gated_rms(const void* x, const void* gate, const void* scale, void* y,
                  int64_t numel, int64_t C, int dtype, float epsilon) {
    if (C <= 0 || numel < 0 || numel % C != 0) return 1;
    int64_t rows = numel / C;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < C; ++j) {
            double v = (double)ld_f32(x, dtype, r * C + j);
            ss += v * v;
        }
        double ms = ss / (double)C;
        double inv = 1.0 / sqrt(ms + (double)epsilon);
        for (int64_t j = 0; j < C; ++j) {
            int64_t i = r * C + j;
            double v = (double)ld_f32(x, dtype, i);
            double g = (double)ld_f32(gate, dtype, i);
            double out = v * inv * (double)ld_f32(scale, dtype, j) * silu(g);
            st_from_f64(y, dtype, i, out);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* com.microsoft.SkipGroupNorm README, Description / Inputs / Attributes:    */
/*   S = X + skip + bias (rounded to T);                                     */
/*   Y = gamma * (S - mean) / sqrt(variance + epsilon) + beta, then SiLU when */
/*   activation == 1; mean and (population) variance per batch item over the */
/*   C/groups channels of a group and every spatial position.                */
/*   X is (N,H,W,C) when channels_last != 0, else (N,C,H,W).                 */
/*   skip_bcast != 0: skip holds one value per (n, c) at offset n*C + c.     */
/*   gamma/beta have their own element type M.                               */
/* ------------------------------------------------------------------------ */
static int64_t sgn_index(int channels_last, int64_t n, int64_t c, int64_t h,
                         int64_t w, int64_t C, int64_t H, int64_t W) {
    if (channels_last) return ((n * H + h) * W + w) * C + c;
    return ((n * C + c) * H + h) * W + w;
}

int orc_skip_group(const void* x, const void* skip, int skip_bcast,
                   const void* bias, const void* gamma, const void* beta,
                   void* y, void* s_out, int64_t N, int64_t C, int64_t H,
                   int64_t W, int dtype, int mdtype, int groups, float epsilon,
                   int activation, int channels_last) {
    if (N < 0 || C <= 0 || H <= 0 || W <= 0 || groups <= 0 || C % groups != 0)
        return 1;
    if (activation != 0 && activation != 1) return 1;
    int64_t cpg = C / groups;
    int64_t cnt = cpg * H * W;
    double* sv = (double*)malloc((size_t)cnt * sizeof(double));
    if (!sv) return 2;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < groups; ++g) {
            /* pass 1: residual sums of the group, and their mean */
            int64_t k = 0;
            double sum = 0.0;
            for (int64_t cc = 0; cc < cpg; ++cc) {
                int64_t c = g * cpg + cc;
                for (int64_t h = 0; h < H; ++h)
                    for (int64_t w = 0; w < W; ++w) {
                        int64_t i = sgn_index(channels_last, n, c, h, w, C, H, W);
                        int64_t si = skip_bcast ? n * C + c : i;
                        double s = residual_sum(ld_f32(x, dtype, i), ld_f32(skip, dtype, si),
                                                bias, dtype, c, s_out, i);
                        sv[k++] = s;
                        sum += s;
                    }
            }
            double mean = sum / (double)cnt;
            /* pass 2: centred population variance */
            double m2 = 0.0;
            for (int64_t t = 0; t < cnt; ++t) {
                double d = sv[t] - mean;
                m2 += d * d;
            }
            double var = m2 / (double)cnt;
            double rstd = 1.0 / sqrt(var + (double)epsilon);
            /* pass 3: normalize, affine, optional SiLU */
            k = 0;
            for (int64_t cc = 0; cc < cpg; ++cc) {
                int64_t c = g * cpg + cc;
                double ga = (double)ld_f32(gamma, mdtype, c);
                double be = (double)ld_f32(beta, mdtype, c);
                for (int64_t h = 0; h < H; ++h)
                    for (int64_t w = 0; w < W; ++w) {
                        int64_t i = sgn_index(channels_last, n, c, h, w, C, H, W);
                        double z = ga * (sv[k++] - mean) * rstd + be;
                        if (activation == 1) z = silu(z);
                        st_from_f64(y, dtype, i, z);
                    }
            }
        }
    }
    free(sv);
    return 0;
}
