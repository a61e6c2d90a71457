// NVFP4 quantisation of an FP32 tensor on the GPU ("NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md",
// kernel plan item 7, "FP4 quantization for NVFP4-1.1"; the format is E2M1 codes, one E4M3
// scale per block of 16 consecutive values and an FP32 per-tensor scale amax / (6 * 448)).
//
// Two passes, because the per-tensor scale depends on every value:
//   1. amax: grid-wide max |x| (warp shuffles, one atomicMax per warp on the FP32 bit pattern,
//      which orders like the value for non-negative floats);
//   2. quant: one thread per 16-value block.  s_g = fp32(amax / 2688).  The block scale is the
//      E4M3 value nearest (ties to even, saturating at 448) to amax_b / (6 s_g), rounded from the
//      FP64 quotient by scaling to an integer grid and rint() (round half to even).  Element codes
//      come from exact FP64 comparisons against the E2M1 rounding midpoints times
//      den = e4m3 * s_g: every midpoint * den product has at most 31 significant bits, so the
//      comparisons, and with them the ties, are exact.  The attention path fuses pass 1 into its
//      epilogue (atomicMax while writing the FP32 output), so only pass 2 runs after it.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fmha {
namespace {

__global__ void amax_kernel(const float* __restrict__ x, int64_t n, unsigned* amax_bits)
{
    float m = 0.f;
    const int64_t n4 = n / 4;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = x4[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax_bits, __float_as_uint(m));
}

// E4M3FN code nearest to v >= 0 (ties to the even code), saturating at 448 (code 0x7E).
// Codes are monotonic in value: subnormal m * 2^-9 has code m, normal (8 + m) * 2^(e - 10) has
// code 8 * e + m, so code = 8 * (e - 1) + rint(v * 2^(10 - e)) across the whole range.
__device__ __forceinline__ uint32_t e4m3_round_sat(double v)
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

__device__ __forceinline__ double e4m3_value(uint32_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 7;
    return e == 0 ? ldexp(static_cast<double>(m), -9) : ldexp(static_cast<double>(8 + m), e - 10);
}

// Midpoints between consecutive E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
__device__ __forceinline__ uint32_t e2m1_code(float x, double den)
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

__global__ void quant_kernel(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ codes,
                             uint8_t* __restrict__ scales, float* tensor_scale, const unsigned* amax_bits)
{
    const float amax = __uint_as_float(*amax_bits);
    const float sg = __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = sg;
    for (int64_t blk = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; blk < nblocks;
         blk += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4* xb = reinterpret_cast<const float4*>(x + blk * 16);
        float v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = xb[i];
            v[4 * i] = t.x;
            v[4 * i + 1] = t.y;
            v[4 * i + 2] = t.z;
            v[4 * i + 3] = t.w;
        }
        float ab = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
        uint32_t sc = 0;
        if (sg > 0.f) sc = e4m3_round_sat(static_cast<double>(ab) / (6.0 * static_cast<double>(sg)));
        scales[blk] = static_cast<uint8_t>(sc);
        const double den = e4m3_value(sc) * static_cast<double>(sg);
        uint32_t lo = 0, hi = 0;
        if (den > 0.0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) lo |= e2m1_code(v[i], den) << (4 * i);
#pragma unroll
            for (int i = 0; i < 8; ++i) hi |= e2m1_code(v[8 + i], den) << (4 * i);
        }
        reinterpret_cast<uint2*>(codes)[blk] = make_uint2(lo, hi);
    }
}

}  // namespace

int launch_nvfp4(const float* x, uint8_t* codes, uint8_t* scales, float* tensor_scale, unsigned* amax_bits, int64_t n,
                 bool amax_ready, cudaStream_t st)
{
    const int nsm = num_sms() > 0 ? num_sms() : 148;
    if (!amax_ready) {
        FMHA_CHECK_CUDA(cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), st));
        if (n > 0) {
            const int64_t want = (n / 4 + 255) / 256;
            const int grid = static_cast<int>(want < 4 * nsm ? (want > 0 ? want : 1) : 4 * nsm);
            amax_kernel<<<grid, 256, 0, st>>>(x, n, amax_bits);
            FMHA_CHECK_LAUNCH("amax_kernel");
            count_launch();
        }
    }
    const int64_t nblocks = n / 16;
    const int64_t want = (nblocks + 255) / 256;
    const int grid = static_cast<int>(want < 8 * nsm ? (want > 0 ? want : 1) : 8 * nsm);
    if (!amax_ready) timing_mark_begin(st);
    quant_kernel<<<grid, 256, 0, st>>>(x, nblocks, codes, scales, tensor_scale, amax_bits);
    if (!amax_ready) timing_mark_end(st);
    FMHA_CHECK_LAUNCH("quant_kernel");
    count_launch();
    return FMHA_OK;
}

}  // namespace fmha
