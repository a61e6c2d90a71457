// Host-side FP8 (E4M3) and FP4 (E2M1) conversions from CUDA's own headers, called (not
// reimplemented) so that the NVFP4 oracle's roundings are pinned to an independent source.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

extern "C" unsigned char host_cvt_e2m1_rn(float x)
{
    return (unsigned char)__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest);
}

extern "C" unsigned char host_cvt_e4m3_satfinite(float x)
{
    return (unsigned char)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

extern "C" unsigned char host_cvt_e4m3_from_double_satfinite(double x)
{
    return (unsigned char)__nv_cvt_double_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
