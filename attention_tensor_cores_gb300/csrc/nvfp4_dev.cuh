// NVFP4 encoding on the device: E2M1 element codes, one E4M3 (OCP E4M3FN) scale per block of 16
// consecutive values, per-tensor scale s_g (the format of the NVFP4 step of the kernel plan in
// "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md", item 7).  Shared by the quantiser kernel and the attention
// epilogues.  Every rounding is exact (nearest, ties to the even code, saturating):
//
//   block scale  sc   = E4M3(amax_b / (6 s_g))
//   element code c_i  = E2M1(x_i / (dec(sc) s_g)), sign kept
//
// Each decision asks whether |x| rounds up across a threshold t * s_g, where t is a grid midpoint
// times a small exact factor (6 for the block scale, dec(sc) for the elements), so t has at most 7
// significant bits and is exact in FP32.  Rounding up means |x| > t s_g, or |x| == t s_g when the
// upper code is even.  Write t s_g = hi + lo exactly (hi = fl(t s_g), lo = fma(t, s_g, -hi)).  No
// float lies strictly between hi and t s_g, so for a float |x| that question is the single
// comparison |x| >= U with U = hi when lo < 0 (or lo == 0 and the tie rounds up) and U = the next
// float above hi otherwise.  The bounds are computed once per block, so each element costs seven
// plain comparisons.  lo is exact while t s_g stays well inside the normal range; for s_g outside
// [2^-90, 2^100] the FP64 route below is used instead (rounding of FP64 quotients, whose products
// with the grid midpoints have at most 31 significant bits).
#pragma once

#include <cstdint>

namespace atc_gb300 {

// ---- FP64 route ------------------------------------------------------------------------------------

// E4M3FN code nearest to v >= 0 (ties to the even code), saturating at 448 (code 0x7E).
// Codes are monotonic in value: subnormal m * 2^-9 has code m, normal (8 + m) * 2^(e - 10) has
// code 8 * e + m, so code = 8 * (e - 1) + rint(v * 2^(10 - e)) across the whole range.
__device__ __forceinline__ uint32_t e4m3_round_sat_f64(double v)
{
    if (!(v > 0.0)) return 0;
    if (v >= 448.0) return 0x7E;
    int E;
    frexp(v, &E);                 // v = f * 2^E, f in [0.5, 1): floor(log2 v) = E - 1
    const int e = E + 6;          // exponent field if v were normal
    uint32_t code;
    if (e >= 1)
        code = static_cast<uint32_t>(8 * (e - 1) + static_cast<int>(rint(ldexp(v, 10 - e))));
    else
        code = static_cast<uint32_t>(rint(ldexp(v, 9)));
    return code > 0x7E ? 0x7Eu : code;
}

__device__ __forceinline__ double e4m3_value_f64(uint32_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 7;
    return e == 0 ? ldexp(static_cast<double>(m), -9) : ldexp(static_cast<double>(8 + m), e - 10);
}

// E2M1 code of x against den > 0 from the midpoints {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} * den.
__device__ __forceinline__ uint32_t e2m1_code_f64(float x, double den)
{
    const double a = fabs(static_cast<double>(x));
    const double mids[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 7; ++k) {
        const double t = mids[k] * den;
        // above the midpoint: round up; on it: up only when the upper code (k + 1) is even
        if (a > t || (a == t && (k & 1))) c = k + 1;
    }
    return c | (signbit(x) ? 8u : 0u);
}

// ---- FP32 route ------------------------------------------------------------------------------------

__device__ __forceinline__ float e4m3_value_f32(uint32_t c)
{
    const uint32_t e = (c >> 3) & 0xF, m = c & 7;
    // normal: (1 + m/8) * 2^(e - 7), built from its FP32 fields; subnormal: m * 2^-9
    return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
}

// Smallest float a >= 0 that rounds up across the threshold t * s (t * s taken exactly: see the
// file comment); tie_up: whether a == t * s rounds up.
__device__ __forceinline__ float round_up_bound(float t, float s, bool tie_up)
{
    const float hi = __fmul_rn(t, s);
    const float lo = __fmaf_rn(t, s, -hi);
    return (lo < 0.f || (lo == 0.f && tie_up)) ? hi : __uint_as_float(__float_as_uint(hi) + 1u);
}

// Approximate E4M3 code of q >= 0 (may be one off near a midpoint; corrected by the caller).
__device__ __forceinline__ uint32_t e4m3_candidate(float q)
{
    if (!(q > 0.f)) return 0;
    if (q >= 448.f) return 0x7E;
    const int E = static_cast<int>((__float_as_uint(q) >> 23) & 0xFF) - 127;   // floor(log2 q), q normal
    const int e = E + 7;
    uint32_t c;
    if (e >= 1)
        c = static_cast<uint32_t>(8 * (e - 1)) + static_cast<uint32_t>(rintf(q * __uint_as_float(static_cast<uint32_t>(130 - E) << 23)));
    else
        c = static_cast<uint32_t>(rintf(q * 512.f));
    return c > 0x7E ? 0x7Eu : c;
}

// E4M3 block scale of a block with max |x| = ab under s_g (FP32 route).
__device__ __forceinline__ uint32_t e4m3_block_scale_f32(float ab, float sg)
{
    // candidate from an approximate quotient (within one code of the nearest), then moved to the
    // exact nearest code across the midpoints 6 * (v_c + v_c+1) / 2 * s_g (6 * midpoint is exact)
    uint32_t c = e4m3_candidate(__fdividef(ab, __fmul_rn(6.f, sg)));
#pragma unroll 1
    for (int it = 0; it < 3 && c < 0x7E; ++it) {
        const float t = __fmul_rn(e4m3_value_f32(c) + e4m3_value_f32(c + 1), 3.f);
        if (ab >= round_up_bound(t, sg, !((c + 1) & 1))) ++c;
        else break;
    }
#pragma unroll 1
    for (int it = 0; it < 3 && c > 0; ++it) {
        const float t = __fmul_rn(e4m3_value_f32(c - 1) + e4m3_value_f32(c), 3.f);
        if (!(ab >= round_up_bound(t, sg, !(c & 1)))) --c;
        else break;
    }
    return c;
}

// Round-up bounds of one block's E2M1 midpoints mid_k * dec(sc) * s_g (ties to the even code: a
// tie at midpoint k rounds up when k is odd).
struct E2m1Bounds {
    float u[7];
};

__device__ __forceinline__ E2m1Bounds e2m1_bounds(float dsc, float sg)
{
    const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
    E2m1Bounds b;
#pragma unroll
    for (int k = 0; k < 7; ++k) b.u[k] = round_up_bound(__fmul_rn(mids[k], dsc), sg, k & 1);   // mid * dsc exact
    return b;
}

__device__ __forceinline__ uint32_t e2m1_code_f32(float x, const E2m1Bounds& b)
{
    const float a = fabsf(x);
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 7; ++k) c += a >= b.u[k] ? 1u : 0u;
    return c | ((__float_as_uint(x) >> 28) & 8u);
}

// ---- block encoders --------------------------------------------------------------------------------

// An s_g that is not a positive finite number encodes every block as zero.
__device__ __forceinline__ bool nvfp4_scale_usable(float sg) { return sg > 0.f && sg <= 3.4028234663852886e38f; }
__device__ __forceinline__ bool nvfp4_fp32_route(float sg) { return sg >= 0x1p-90f && sg <= 0x1p100f; }

// Encodes v[0..15]: returns the E4M3 scale code and the 16 element codes as two words (element 2i
// in bits 3:0 and element 2i + 1 in bits 7:4 of byte i).
__device__ __forceinline__ uint32_t nvfp4_encode16(const float* v, float sg, uint32_t& lo, uint32_t& hi)
{
    lo = hi = 0;
    if (!nvfp4_scale_usable(sg)) return 0;
    float ab = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    if (nvfp4_fp32_route(sg)) {
        const uint32_t sc = e4m3_block_scale_f32(ab, sg);
        if (sc == 0) return 0;
        const E2m1Bounds t = e2m1_bounds(e4m3_value_f32(sc), sg);
#pragma unroll
        for (int i = 0; i < 8; ++i) lo |= e2m1_code_f32(v[i], t) << (4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) hi |= e2m1_code_f32(v[8 + i], t) << (4 * i);
        return sc;
    }
    const uint32_t sc = e4m3_round_sat_f64(static_cast<double>(ab) / (6.0 * static_cast<double>(sg)));
    const double den = e4m3_value_f64(sc) * static_cast<double>(sg);
    if (den > 0.0) {
        // fully unrolled: a run-time index would force the caller's v[] into local memory
#pragma unroll
        for (int i = 0; i < 8; ++i) lo |= e2m1_code_f64(v[i], den) << (4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) hi |= e2m1_code_f64(v[8 + i], den) << (4 * i);
    }
    return sc;
}

// One value per lane, blocks of 16 consecutive lanes (a fully active warp whose lane l holds column
// col with col % 32 == l).  Writes the code byte of each even column and the scale of each block.
__device__ __forceinline__ void nvfp4_encode_lanes(float x, float sg, int col, uint8_t* codes_row, uint8_t* scales_row)
{
    float ab = fabsf(x);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, o));
    uint32_t sc = 0, c = 0;
    if (nvfp4_scale_usable(sg)) {
        if (nvfp4_fp32_route(sg)) {
            sc = e4m3_block_scale_f32(ab, sg);
            if (sc) c = e2m1_code_f32(x, e2m1_bounds(e4m3_value_f32(sc), sg));
        } else {
            sc = e4m3_round_sat_f64(static_cast<double>(ab) / (6.0 * static_cast<double>(sg)));
            const double den = e4m3_value_f64(sc) * static_cast<double>(sg);
            if (den > 0.0) c = e2m1_code_f64(x, den);
        }
    }
    const uint32_t next = __shfl_down_sync(0xffffffffu, c, 1);
    if (!(col & 1)) codes_row[col >> 1] = static_cast<uint8_t>(c | (next << 4));
    if (!(col & 15)) scales_row[col >> 4] = static_cast<uint8_t>(sc);
}

}  // namespace atc_gb300
