// C-ABI layer of libfmha.so: argument validation, error reporting, the device status word,
// TMA tensor-map encoding, and dispatch to the kernel launchers.  See include/fmha.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace fmha {

// ---- errors ------------------------------------------------------------------------------------
static thread_local std::string g_last_error;

int set_error(int code, const std::string& msg)
{
    g_last_error = msg;
    return code;
}

int cuda_error(cudaError_t e, const char* what)
{
    return set_error(FMHA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

// ---- device status word ----------------------------------------------------------------------------
// One int per device in this library's module: kernels write a nonzero code when a bounded wait
// expires.  Its address is looked up once per device and passed to kernels as a pointer.
static __device__ int g_status_word;
static constexpr int kMaxDevices = 64;
static std::atomic<int*> g_status_addr[kMaxDevices];
static std::atomic<int> g_num_sms[kMaxDevices];
static std::atomic<long long> g_wait_limit{0};

int* device_status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_status_addr[dev].load();
    if (!p) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
        p = static_cast<int*>(addr);
        g_status_addr[dev].store(p);
    }
    return p;
}

long long wait_limit()
{
    const long long v = g_wait_limit.load();
    return v > 0 ? v : 4000000000LL;   // ~2 s at 2 GHz
}

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = g_num_sms[dev].load();
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_num_sms[dev].store(n);
    }
    return n;
}

// ---- TMA tensor maps -------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                   const uint32_t* box)
{
    auto fn = encode_fn();
    if (!fn) return set_error(FMHA_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    cuuint64_t gdim[5];
    cuuint64_t gstride[5];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i > 0) gstride[i - 1] = strides_bytes[i - 1];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim, gstride, bdim, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d, rank %d, dim0 %llu, box0 %u)", (int)r,
                 rank, (unsigned long long)dims[0], box[0]);
        return set_error(FMHA_ERR_CUDA, buf);
    }
    return FMHA_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace fmha

using namespace fmha;

// ================================================================================================
// C ABI
// ================================================================================================
extern "C" {

const char* fmha_error_string(int code)
{
    switch (code) {
        case FMHA_OK: return "FMHA_OK";
        case FMHA_ERR_INVALID: return "FMHA_ERR_INVALID: invalid argument";
        case FMHA_ERR_UNSUPPORTED: return "FMHA_ERR_UNSUPPORTED: valid but not supported";
        case FMHA_ERR_WORKSPACE: return "FMHA_ERR_WORKSPACE: workspace missing or too small";
        case FMHA_ERR_CUDA: return "FMHA_ERR_CUDA: CUDA call or kernel launch failed";
        case FMHA_ERR_TIMEOUT: return "FMHA_ERR_TIMEOUT: a kernel's bounded wait expired";
        default: return "unknown fmha status";
    }
}

const char* fmha_last_error(void) { return g_last_error.c_str(); }

void fmha_set_wait_limit(long long cycles) { g_wait_limit.store(cycles > 0 ? cycles : 0); }

int fmha_num_sms(void) { return num_sms(); }

int fmha_check_status(fmha_stream_t stream)
{
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "cudaMemcpyFromSymbol(status)");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_error(e, "cudaMemcpyToSymbol(status)");
        return set_error(FMHA_ERR_TIMEOUT, "a kernel's bounded wait expired (device status word set)");
    }
    return FMHA_OK;
}

int fmha_qk_gemm(const void* q, const void* k, float* s, int Sq, int Skv, int D, fmha_stream_t stream)
{
    if (!q || !k || !s) return set_error(FMHA_ERR_INVALID, "fmha_qk_gemm: NULL pointer");
    if (Sq <= 0 || Skv <= 0) return set_error(FMHA_ERR_INVALID, "fmha_qk_gemm: Sq and Skv must be positive");
    if (D != 16 && D != 64 && D != 128 && D != 512)
        return set_error(FMHA_ERR_INVALID, "fmha_qk_gemm: D must be 16, 64, 128 or 512");
    if (!aligned16(q) || !aligned16(k) || !aligned16(s))
        return set_error(FMHA_ERR_INVALID, "fmha_qk_gemm: pointers must be 16-byte aligned");
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    return launch_qk_gemm(q, k, s, Sq, Skv, D, reinterpret_cast<cudaStream_t>(stream));
}

int fmha_selftest(int which, const void* in, void* out, size_t out_bytes, int param, fmha_stream_t stream)
{
    if (!out || (which != 1 && !in)) return set_error(FMHA_ERR_INVALID, "fmha_selftest: NULL pointer");
    if (!aligned16(in) || !aligned16(out)) return set_error(FMHA_ERR_INVALID, "fmha_selftest: misaligned");
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    return launch_selftest(which, in, out, out_bytes, param, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
