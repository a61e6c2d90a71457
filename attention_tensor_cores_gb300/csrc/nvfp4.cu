// NVFP4 quantisation of an FP32 tensor on the GPU ("NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md",
// kernel plan item 7, "FP4 quantization for NVFP4-1.1"; the format is E2M1 codes, one E4M3
// scale per block of 16 consecutive values and an FP32 per-tensor scale amax / (6 * 448)).
//
// Two passes, because the per-tensor scale depends on every value:
//   1. amax: grid-wide max |x| (warp shuffles, one atomicMax per warp on the FP32 bit pattern,
//      which orders like the value for non-negative floats);
//   2. quant: one thread per 16-value block.  s_g = fp32(amax / 2688), or the caller's s_g.  The
//      block scale and element codes are the exactly rounded ones of nvfp4_dev.cuh (FP32 exact
//      comparisons against the rounding midpoints).  The attention path fuses pass 1 into its
//      epilogue (atomicMax while writing the FP32 output), so only pass 2 runs after it; with a
//      given s_g the epilogues encode directly and neither pass runs.
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_dev.cuh"
#include "ptx.cuh"

namespace atc_gb300 {
namespace {

__global__ void amax_kernel(const float* __restrict__ x, int64_t n, unsigned* amax_bits)
{
    griddep_launch_dependents();
    griddep_wait();
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

__global__ void quant_kernel(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ codes,
                             uint8_t* __restrict__ scales, float* tensor_scale, const unsigned* amax_bits,
                             const float* sg_in)
{
    griddep_launch_dependents();
    griddep_wait();
    // s_g: given by the caller, or fp32(amax / 2688) (one correctly rounded division)
    const float sg = sg_in ? *sg_in : __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0 && tensor_scale) *tensor_scale = sg;
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
        uint32_t lo, hi;
        scales[blk] = static_cast<uint8_t>(nvfp4_encode16(v, sg, lo, hi));
        reinterpret_cast<uint2*>(codes)[blk] = make_uint2(lo, hi);
    }
}

}  // namespace

int launch_nvfp4(const float* x, uint8_t* codes, uint8_t* scales, float* tensor_scale, unsigned* amax_bits, int64_t n,
                 bool amax_ready, cudaStream_t st, const float* sg_in)
{
    const int nsm = num_sms() > 0 ? num_sms() : 148;
    if (!amax_ready && !sg_in) {
        FMHA_CHECK_CUDA(cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), st));
        if (n > 0) {
            const int64_t want = (n / 4 + 255) / 256;
            const int grid = static_cast<int>(want < 4 * nsm ? (want > 0 ? want : 1) : 4 * nsm);
            FMHA_CHECK_CUDA(launch_pdl(amax_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, x, n, amax_bits));
            count_launch();
        }
    }
    const int64_t nblocks = n / 16;
    const int64_t want = (nblocks + 255) / 256;
    const int grid = static_cast<int>(want < 8 * nsm ? (want > 0 ? want : 1) : 8 * nsm);
    if (!amax_ready) timing_mark_begin(st);
    const cudaError_t e = launch_pdl(quant_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, x, nblocks, codes,
                                     scales, tensor_scale, const_cast<const unsigned*>(amax_bits), sg_in);
    if (!amax_ready) timing_mark_end(st);
    FMHA_CHECK_CUDA(e);
    count_launch();
    return FMHA_OK;
}

}  // namespace atc_gb300
