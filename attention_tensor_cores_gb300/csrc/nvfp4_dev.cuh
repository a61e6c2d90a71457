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
// float above hi otherwise.  A block computes its seven element bounds once and counts, per element,
// the bounds |x| reaches; one value alone takes a binary search over the bounds it needs.  lo is
// exact while t s_g stays well inside the normal range; for s_g outside [2^-90, 2^100] the FP64
// route below is used instead (rounding of FP64 quotients, whose products with the grid midpoints
// have at most 31 significant bits).
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

// Round-up bound of E4M3 code c in 1..126 for the block scale: the smallest amax_b that rounds to
// c or above is 6 s_g times the midpoint between the values of codes c - 1 and c (ties to the even
// code).  That midpoint is (2c - 1) 2^-10 for c <= 8 (the subnormal codes and the first normal one).
// Above, it is the float halfway between the two values' bit patterns: normal codes are 2^20 apart
// in FP32 bits (v_c has bits (c << 20) + 0x3C000000), and within a binade, and across one since the
// midpoint lies in the lower binade, FP32 values are linear in their bits.  6 * midpoint has at most
// 7 significant bits, so it is exact.
__device__ __forceinline__ float e4m3_up_bound(uint32_t c, float sg)
{
    const float odd = __fsub_rn(__uint_as_float(0x4B000000u + 2u * c - 1u), 8388608.f);   // 2c - 1, exact
    const float mid = c > 8u ? __uint_as_float((c << 20) + 0x3BF80000u) : __fmul_rn(odd, 0x1p-10f);
    return round_up_bound(__fmul_rn(mid, 6.f), sg, !(c & 1u));
}

// E4M3 block scale of a block with max |x| = ab under s_g (FP32 route).  A candidate comes from the
// approximate quotient q = ab * (1 / (6 s_g)) (relative error a few 2^-24), rounded half up at
// E4M3 resolution on q's bits; normal E4M3 values are more than 2^-4 apart relative to their size
// (2^-9 apart below 2^-6), so the candidate is at most one code from the exact nearest and one exact
// check on each side settles it.
__device__ __forceinline__ uint32_t e4m3_block_scale_f32(float ab, float sg)
{
    const float q = __fmul_rn(ab, __fdividef(1.f, __fmul_rn(6.f, sg)));
    uint32_t c = q < 0x1p-6f ? __float_as_uint(__fadd_rn(q, 0x1p14f)) - 0x46800000u   // rint(q * 2^9)
                             : ((__float_as_uint(q) + 0x80000u) >> 20) - 960u;        // 8 e + m, e = exponent - 120
    c = min(c, 0x7Eu);
    if (c < 0x7Eu && ab >= e4m3_up_bound(c + 1u, sg)) ++c;
    else if (c > 0u && !(ab >= e4m3_up_bound(c, sg))) --c;
    return c;
}

// Round-up bounds of one block's E2M1 midpoints mid_k * dec(sc) * s_g (ties to the even code: a
// tie at midpoint k rounds up when k is odd).
struct E2m1Bounds {
    float u[7];
    float K, P[7];   // the step form: K = 2^(23 - e), e the exponent of pred(u[0]); P[k] = K * pred(u[k])
};

__device__ __forceinline__ E2m1Bounds e2m1_bounds(float dsc, float sg)
{
    const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
    E2m1Bounds b;
#pragma unroll
    for (int k = 0; k < 7; ++k) b.u[k] = round_up_bound(__fmul_rn(mids[k], dsc), sg, k & 1);   // mid * dsc exact
    b.K = __uint_as_float((277u - ((__float_as_uint(b.u[0]) - 1u) >> 23)) << 23);
#pragma unroll
    for (int k = 0; k < 7; ++k) b.P[k] = __fmul_rn(b.K, __uint_as_float(__float_as_uint(b.u[k]) - 1u));   // exact
    return b;
}

// E2M1 code of x from a block's bounds: how many bounds |x| reaches, counted on the FMA pipe (a
// search's comparisons and selects would load the ALU pipe instead).  |x| >= u[k] exactly when
// |x| > pred(u[k]), as no float lies between them.  The fma K |x| - P[k] is exact before its one
// rounding, so its sign is right, and when positive it is at least K times the gap between
// pred(u[k]) and the next float, which is at least 2^(e - 23) = 1 / K: its saturation is 1 or 0
// (a NaN saturates to 0).  The seven steps are summed onto 1.5 * 2^23, whose low mantissa bits then
// hold the count.
__device__ __forceinline__ uint32_t e2m1_code_f32(float x, const E2m1Bounds& b)
{
    const float a = fabsf(x);
    float acc = 12582912.f;
#pragma unroll
    for (int k = 0; k < 7; ++k) acc = __fadd_rn(acc, __saturatef(__fmaf_rn(a, b.K, -b.P[k])));
    return (__float_as_uint(acc) - 0x4B400000u) | ((__float_as_uint(x) >> 28) & 8u);
}

// The code of one value by a binary search over the bounds, which increase with k: three
// comparisons, computing only the three bounds the search visits.  A NaN reaches none.
__device__ __forceinline__ uint32_t e2m1_code_f32(float x, float dsc, float sg)
{
    const float a = fabsf(x);
    const bool p2 = a >= round_up_bound(__fmul_rn(1.75f, dsc), sg, true);
    const bool p1 = a >= round_up_bound(__fmul_rn(p2 ? 3.5f : 0.75f, dsc), sg, true);
    const float m0 = p2 ? (p1 ? 5.f : 2.5f) : (p1 ? 1.25f : 0.25f);
    const bool p0 = a >= round_up_bound(__fmul_rn(m0, dsc), sg, false);
    return (p2 ? 4u : 0u) + (p1 ? 2u : 0u) + (p0 ? 1u : 0u) + ((__float_as_uint(x) >> 28) & 8u);
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
            if (sc) c = e2m1_code_f32(x, e4m3_value_f32(sc), sg);
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
