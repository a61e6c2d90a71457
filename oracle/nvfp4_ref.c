/*
 * CPU oracle for NVFP4 quantisation of the attention output.
 * TEST INFRASTRUCTURE ONLY (see oracle.h): never linked into or called by the CUDA library.
 *
 * The pages ("NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md", kernel plan item 7, "FP4 quantization for
 * NVFP4-1.1") name the format without defining it.  The definition used here is the one the
 * library is specified with: E2M1 element codes, one E4M3 (OCP E4M3FN) scale per block of 16
 * consecutive values, and an FP32 per-tensor scale s_g = amax / (6 * 448).
 *
 * Steps, written out in the order of that definition:
 *   1. amax = max |x_i| over the whole tensor; s_g = fp32_round_nearest(amax / 2688)
 *      (skipped by oracle_nvfp4_quantize_scaled, which takes s_g from the caller).
 *   2. per block of 16: sc = E4M3_round_nearest_even_satfinite(amax_block / (6 s_g)).
 *   3. per element: code = E2M1_round_nearest_even_satfinite(x_i / (dec(sc) * s_g)), sign kept.
 *   4. packing: element 2i in bits 3:0, element 2i+1 in bits 7:4.
 * Roundings are done by searching the whole finite value set of the target format for the
 * nearest value (ties to the even code), on FP64 quotients.  The FP64 quotient of two FP32
 * values cannot land on a rounding midpoint of a 2- or 4-significant-bit format unless the
 * exact quotient is on it, so this equals rounding the exact quotient.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

double oracle_e4m3_decode(uint8_t code)
{
    const int sign = code >> 7;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest of the 127 non-negative finite E4M3FN values (codes 0x00..0x7E) to |v|;
 * a tie goes to the code whose lowest (mantissa) bit is 0.  Values above 448 give 448. */
uint8_t oracle_e4m3_round(double v)
{
    const double a = fabs(v);
    if (a >= 448.0) /* satfinite: everything at or above the largest finite value */
        return 0x7E;
    int best = 0;
    double best_err = fabs(a - oracle_e4m3_decode(0));
    for (int c = 1; c <= 0x7E; ++c) {
        const double err = fabs(a - oracle_e4m3_decode((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)best;
}

static const double k_e2m1_values[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_decode(uint8_t code)
{
    const double m = k_e2m1_values[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest E2M1 magnitude to |v| (ties to the even code), saturating at 6; the sign bit of v
 * is copied, so a negative value that rounds to zero gives the code 0x8. */
uint8_t oracle_e2m1_round(double v)
{
    const double a = fabs(v);
    if (a >= 6.0) /* satfinite */
        return (uint8_t)(7 | (signbit(v) ? 8 : 0));
    int best = 0;
    double best_err = a;
    for (int c = 1; c < 8; ++c) {
        const double err = fabs(a - k_e2m1_values[c]);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 8 : 0));
}

/* Steps 2-4 of the definition with a given per-tensor scale s_g (the single-pass form: a caller
 * that knows s_g in advance, e.g. from an earlier step's amax, skips step 1).  Block scales above
 * the E4M3 range and elements above 6 saturate.  An s_g that is not a positive finite number
 * encodes every block as zero (as amax = 0 does in step 1). */
int oracle_nvfp4_quantize_scaled(const float* x, int64_t n, float s_g, uint8_t* codes, uint8_t* scales)
{
    if (!x || !codes || !scales || n < 0 || n % 16 != 0)
        return -1;
    const int usable = s_g > 0.0f && !isinf(s_g);
    memset(codes, 0, (size_t)(n / 2));
    for (int64_t blk = 0; blk < n / 16; ++blk) {
        const float* xb = x + blk * 16;
        /* 2. block scale */
        float amax_b = 0.0f;
        for (int i = 0; i < 16; ++i) {
            const float a = fabsf(xb[i]);
            if (a > amax_b)
                amax_b = a;
        }
        uint8_t sc = 0;
        if (usable)
            sc = oracle_e4m3_round((double)amax_b / (6.0 * (double)s_g));
        scales[blk] = sc;
        /* 3. element codes against den = dec(sc) * s_g (exact in FP64) */
        const double den = usable ? oracle_e4m3_decode(sc) * (double)s_g : 0.0;
        for (int i = 0; i < 16; ++i) {
            uint8_t c = 0;
            if (den > 0.0)
                c = oracle_e2m1_round((double)xb[i] / den);
            /* 4. packing */
            const int64_t e = blk * 16 + i;
            if ((e & 1) == 0)
                codes[e / 2] |= c;
            else
                codes[e / 2] |= (uint8_t)(c << 4);
        }
    }
    return 0;
}

int oracle_nvfp4_quantize(const float* x, int64_t n, uint8_t* codes, uint8_t* scales,
                          float* tensor_scale)
{
    if (!x || !codes || !scales || !tensor_scale || n < 0 || n % 16 != 0)
        return -1;

    /* 1. global amax and the per-tensor scale (one FP32 rounding of amax / 2688) */
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    const float s_g = (float)((double)amax / 2688.0);
    *tensor_scale = s_g;
    /* 2.-4. */
    return oracle_nvfp4_quantize_scaled(x, n, s_g, codes, scales);
}
