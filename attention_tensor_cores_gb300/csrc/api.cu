// C-ABI layer of libfmha.so: argument validation, error reporting, the device status word,
// TMA tensor-map encoding, and dispatch to the kernel launchers.  See include/fmha.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace atc_gb300 {

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
static constexpr int kDevMergeLost = 6;   // the value the split-KV merge leaves (ptx.cuh)
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

// ---- launch accounting / timing hook --------------------------------------------------------------
static std::atomic<long long> g_launches{0};
static thread_local cudaEvent_t g_ev_begin = nullptr;
static thread_local cudaEvent_t g_ev_end = nullptr;

void count_launch(int n) { g_launches.fetch_add(n); }

cudaError_t set_smem_limit_once(const void* func, int bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    static std::mutex mu;
    static struct Done {
        const void* func;
        int dev, bytes;
    } done[256];
    static int n_done = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < n_done; ++i)
            if (done[i].func == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    }
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0) {
        std::lock_guard<std::mutex> lk(mu);
        if (n_done < 256) done[n_done++] = {func, dev, bytes};
    }
    return e;
}

static std::atomic<unsigned long long> g_call_tag{0};
unsigned long long next_call_tag() { return ((g_call_tag.fetch_add(1) + 1) & ((1ull << 48) - 1)) | (1ull << 47); }

void timing_mark_begin(cudaStream_t st)
{
    if (g_ev_begin) cudaEventRecord(g_ev_begin, st);
}

void timing_mark_end(cudaStream_t st)
{
    if (g_ev_end) cudaEventRecord(g_ev_end, st);
    g_ev_begin = g_ev_end = nullptr;
}

unsigned pdl_attribute(cudaStream_t st, cudaLaunchAttribute* attr)
{
    // a graph being captured keeps plain stream order (its nodes then depend on whole kernels)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (cs != cudaStreamCaptureStatusNone) return 0;
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    return 1;
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

// The driver-API encoder needs a context current on the calling thread.  The runtime makes its
// primary context current lazily, at a thread's first call that needs one, so a host thread whose first
// CUDA call is this library's would have none: bind the current device's primary context first (once
// per thread; a later cudaSetDevice by the caller binds that device's).
static void bind_primary_context()
{
    thread_local bool bound = false;
    if (bound) return;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) bound = true;
    (void)cudaGetLastError();
}

int make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                   const uint32_t* box)
{
    bind_primary_context();
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

}  // namespace atc_gb300

using namespace atc_gb300;

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
        case FMHA_ERR_RACE: return "FMHA_ERR_RACE: overlapping calls on one workspace left a split-KV merge unsettled";
        default: return "unknown fmha status";
    }
}

const char* fmha_last_error(void) { return g_last_error.c_str(); }

void fmha_set_wait_limit(long long cycles) { g_wait_limit.store(cycles > 0 ? cycles : 0); }

int fmha_num_sms(void) { return num_sms(); }

long long fmha_launch_count(void) { return g_launches.load(); }

void fmha_time_next_call(void* start_event, void* stop_event)
{
    g_ev_begin = static_cast<cudaEvent_t>(start_event);
    g_ev_end = static_cast<cudaEvent_t>(stop_event);
}

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
        if (v == kDevMergeLost)
            return set_error(FMHA_ERR_RACE, "a split-KV merge counter never settled (device status word set)");
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

// ---- attention ---------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool use_decode_path(int Hq, int Hkv, int Sq) { return static_cast<long long>(Hq / Hkv) * Sq <= 16; }

// Workspace: [path scratch][NVFP4 amax word].  The path scratch of the decode path holds the
// tile prefix, the split partials and (NVFP4 without out_f32) the FP32 staging of O; that of the
// row-tile path the work-item counter (causal or ragged) and the FP32 staging of O, last.
static size_t workspace_bytes(const AttnArgs& a, int num_splits)
{
    size_t w = a.D == 512 ? wide_workspace_bytes(a, num_splits)
               : use_decode_path(a.Hq, a.Hkv, a.Sq) ? decode_workspace_bytes(a, num_splits) : prefill_workspace_bytes(a, num_splits);
    w = align256(w);
    if (a.out_kind == FMHA_OUT_NVFP4 && !a.nv_sg) w += 256;   // amax word of the two-pass NVFP4 path
    return w;
}

static int validate(const void* q, const void* k, const void* v, const void* out, int B, int Hq, int Hkv, int Sq,
                    int Skv, int D, float scale, const fmha_opts* o)
{
    if (!q || !k || !v || !out) return set_error(FMHA_ERR_INVALID, "NULL q/k/v/out");
    // the kernels take each row's maximum of the raw scores and scale it afterwards, which needs scale > 0
    if (!(scale > 0.f) || !(scale < INFINITY)) return set_error(FMHA_ERR_INVALID, "scale must be a positive finite number");
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0)
        return set_error(FMHA_ERR_INVALID, "need B >= 0, Hq > 0, Hkv > 0, Sq >= 0, Skv >= 1");
    if (Hq % Hkv != 0) return set_error(FMHA_ERR_INVALID, "Hq must be a multiple of Hkv");
    if (D != 64 && D != 128 && D != 512) return set_error(FMHA_ERR_INVALID, "D must be 64, 128 or 512");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return set_error(FMHA_ERR_INVALID, "q/k/v/out must be 16-byte aligned");
    if (static_cast<long long>(B) * Hkv * Skv >= (1LL << 31) || static_cast<long long>(B) * Hq * Sq >= (1LL << 31))
        return set_error(FMHA_ERR_UNSUPPORTED, "more than 2^31 rows");
    if (o) {
        if (o->out_kind < FMHA_OUT_BF16 || o->out_kind > FMHA_OUT_NVFP4) return set_error(FMHA_ERR_INVALID, "bad out_kind");
        if (o->num_splits < 0) return set_error(FMHA_ERR_INVALID, "num_splits must be >= 0");
        if (o->wide_variant < FMHA_WIDE_AUTO || o->wide_variant > FMHA_WIDE_PAIR)
            return set_error(FMHA_ERR_INVALID, "bad wide_variant");
        if (o->out_kind == FMHA_OUT_NVFP4) {
            if (!o->out_scales || !o->out_tensor_scale)
                return set_error(FMHA_ERR_INVALID, "NVFP4 output needs out_scales and out_tensor_scale");
            if ((o->out_f32 && !aligned16(o->out_f32)))
                return set_error(FMHA_ERR_INVALID, "out_f32 must be 16-byte aligned");
            if ((reinterpret_cast<uintptr_t>(o->nvfp4_scale_in) & 3) || (reinterpret_cast<uintptr_t>(o->out_amax) & 3))
                return set_error(FMHA_ERR_INVALID, "nvfp4_scale_in and out_amax must be 4-byte aligned");
        }
        if (o->seqlens_k && (reinterpret_cast<uintptr_t>(o->seqlens_k) & 3))
            return set_error(FMHA_ERR_INVALID, "seqlens_k must be 4-byte aligned");
        if (o->workspace && (reinterpret_cast<uintptr_t>(o->workspace) & 255))
            return set_error(FMHA_ERR_INVALID, "workspace must be 256-byte aligned");
    }
    return FMHA_OK;
}

static AttnArgs make_args(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                          int Sq, int Skv, int D, float scale, const fmha_opts* o)
{
    AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Sq = Sq;
    a.Skv = Skv;
    a.D = D;
    a.scale = scale;
    a.seqlens = o ? o->seqlens_k : nullptr;
    a.out_kind = o ? o->out_kind : FMHA_OUT_BF16;
    a.out_f32 = (o && o->out_kind == FMHA_OUT_NVFP4) ? o->out_f32 : nullptr;
    a.causal = (o && o->causal) ? 1 : 0;
    a.nv_sg = (o && o->out_kind == FMHA_OUT_NVFP4) ? o->nvfp4_scale_in : nullptr;
    a.wide_variant = o ? o->wide_variant : FMHA_WIDE_AUTO;
    return a;
}

size_t fmha_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D, const fmha_opts* opts)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0 || Hq % Hkv) return 0;
    AttnArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, B, Hq, Hkv, Sq, Skv, D, 1.f, opts);
    return workspace_bytes(a, opts ? opts->num_splits : 1);
}

int fmha_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv, int Sq,
                int Skv, int D, float scale, fmha_stream_t stream, const fmha_opts* opts)
{
    int rc = validate(q, k, v, out, B, Hq, Hkv, Sq, Skv, D, scale, opts);
    if (rc) return rc;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) return set_error(FMHA_ERR_INVALID, "lse must be 4-byte aligned");
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    AttnArgs a = make_args(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, scale, opts);
    void* ws = opts ? opts->workspace : nullptr;
    // automatic split-KV (decode) or work-item counter (row-tile) when the caller supplied a
    // workspace; whole units in a fixed order otherwise
    const int num_splits = (opts && (opts->num_splits != 0 || ws)) ? opts->num_splits : 1;
    const size_t ws_bytes = opts ? opts->workspace_bytes : 0;
    const size_t need = workspace_bytes(a, num_splits);
    if (need > 0 && (!ws || ws_bytes < need))
        return set_error(FMHA_ERR_WORKSPACE, "workspace missing or smaller than fmha_workspace_size()");
    if (static_cast<long long>(B) * Hq * Sq == 0) return FMHA_OK;
    const bool nvfp4 = a.out_kind == FMHA_OUT_NVFP4;
    const bool two_pass = nvfp4 && !a.nv_sg;
    const size_t path_bytes = two_pass ? need - 256 : need;
    // |O| max: the caller's out_amax when given, else (two passes) the word after the path scratch
    unsigned* amax = nullptr;
    if (nvfp4 && opts->out_amax)
        amax = reinterpret_cast<unsigned*>(opts->out_amax);
    else if (two_pass)
        amax = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + path_bytes);
    if (amax) {
        a.amax_slot = reinterpret_cast<float*>(amax);
        FMHA_CHECK_CUDA(cudaMemsetAsync(amax, 0, sizeof(unsigned), st));
    }
    if (nvfp4 && a.nv_sg) {
        // single pass: the epilogues write the codes and block scales themselves
        a.nv_codes = static_cast<uint8_t*>(out);
        a.nv_scales = opts->out_scales;
        a.nv_ts = opts->out_tensor_scale;
    }
    if (D == 512)
        rc = launch_wide(a, num_splits, ws, path_bytes, st);
    else if (use_decode_path(Hq, Hkv, Sq))
        rc = launch_decode(a, num_splits, ws, path_bytes, st);
    else
        rc = launch_prefill(a, num_splits, ws, path_bytes, st);
    if (rc) return rc;
    if (two_pass) {
        // the FP32 O the quantiser reads: caller's out_f32, else the staging area of the workspace
        const float* src = a.out_f32;
        if (!src) {
            const size_t n = static_cast<size_t>(B) * Hq * Sq * D;
            src = reinterpret_cast<const float*>(static_cast<uint8_t*>(ws) + path_bytes - align256(n * 4));
        }
        rc = launch_nvfp4(src, static_cast<uint8_t*>(out), opts->out_scales, opts->out_tensor_scale, amax,
                          static_cast<int64_t>(B) * Hq * Sq * D, true, st);
    }
    return rc;
}

int fmha_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv, int Sq, int Skv,
             int D, float scale, fmha_stream_t stream)
{
    return fmha_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, scale, stream, nullptr);
}

// ---- attention from host memory ----------------------------------------------------------------------------
// dev_buf: staged Q | K | V | O | LSE | attention workspace (sized for the largest batch chunk).
struct HostLayout {
    size_t q, k, v, o, lse, ws, ws_bytes, total;
    int chunks, bc;   // batch chunks and entries per chunk (the last chunk may have fewer)
};

static fmha_opts host_call_opts(const fmha_opts* o)
{
    fmha_opts w{};
    w.out_kind = o ? o->out_kind : FMHA_OUT_BF16;
    w.num_splits = o ? o->num_splits : 0;
    w.causal = o ? o->causal : 0;
    w.wide_variant = o ? o->wide_variant : FMHA_WIDE_AUTO;
    return w;
}

static HostLayout host_layout(int B, int Hq, int Hkv, int Sq, int Skv, int D, const fmha_opts* o)
{
    HostLayout L{};
    const size_t esz = (o && o->out_kind == FMHA_OUT_F32) ? 4 : 2;
    const size_t nq = static_cast<size_t>(B) * Hq * Sq * D, nkv = static_cast<size_t>(B) * Hkv * Skv * D;
    const int want = B >= 2 ? (B < 4 ? B : 4) : 1;
    L.bc = B > 0 ? (B + want - 1) / want : 0;
    L.chunks = B > 0 ? (B + L.bc - 1) / L.bc : 0;
    size_t off = 0;
    L.q = off;
    off += align256(nq * 2);
    L.k = off;
    off += align256(nkv * 2);
    L.v = off;
    off += align256(nkv * 2);
    L.o = off;
    off += align256(nq * esz);
    L.lse = off;
    off += align256(static_cast<size_t>(B) * Hq * Sq * 4);
    const fmha_opts w = host_call_opts(o);
    L.ws_bytes = L.bc > 0 ? fmha_workspace_size(L.bc, Hq, Hkv, Sq, Skv, D, &w) : 0;
    L.ws = off;
    off += align256(L.ws_bytes);
    L.total = off;
    return L;
}

// Per device: the copy stream and events of chunked host calls (created once, kept for the
// library's lifetime) and the lock that keeps one host thread enqueuing at a time.
struct HostAux {
    cudaStream_t cs;
    cudaEvent_t start, copied[4];
    bool ready;
};
static HostAux g_host_aux[kMaxDevices];
static std::mutex g_host_mu;

static HostAux* host_aux()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    HostAux& h = g_host_aux[dev];
    if (!h.ready) {
        if (cudaStreamCreateWithFlags(&h.cs, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        bool ok = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < 4 && ok; ++i) ok = cudaEventCreateWithFlags(&h.copied[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return nullptr;
        h.ready = true;
    }
    return &h;
}

size_t fmha_host_buffer_size(int B, int Hq, int Hkv, int Sq, int Skv, int D, const fmha_opts* opts)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0 || Hq % Hkv) return 0;
    return host_layout(B, Hq, Hkv, Sq, Skv, D, opts).total;
}

int fmha_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* out_host, float* lse_host, int B,
                  int Hq, int Hkv, int Sq, int Skv, int D, float scale, fmha_stream_t stream, const fmha_opts* opts,
                  void* dev_buf, size_t dev_buf_bytes)
{
    if (!q_host || !k_host || !v_host || !out_host) return set_error(FMHA_ERR_INVALID, "fmha_fwd_host: NULL host pointer");
    if (opts && (opts->seqlens_k || opts->out_kind == FMHA_OUT_NVFP4 || opts->out_scales || opts->out_tensor_scale ||
                 opts->out_f32 || opts->nvfp4_scale_in || opts->out_amax || opts->workspace || opts->workspace_bytes))
        return set_error(FMHA_ERR_UNSUPPORTED,
                         "fmha_fwd_host: options limited to out_kind (BF16/F32), num_splits, causal and wide_variant");
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0 || Hq % Hkv)
        return set_error(FMHA_ERR_INVALID, "need B >= 0, Hq > 0, Hkv > 0 dividing Hq, Sq >= 0, Skv >= 1");
    const HostLayout L = host_layout(B, Hq, Hkv, Sq, Skv, D, opts);
    if (!dev_buf || (reinterpret_cast<uintptr_t>(dev_buf) & 255) || dev_buf_bytes < L.total)
        return set_error(FMHA_ERR_WORKSPACE, "fmha_fwd_host: dev_buf missing, not 256-byte aligned or smaller than fmha_host_buffer_size()");
    uint8_t* base = static_cast<uint8_t*>(dev_buf);
    fmha_opts w = host_call_opts(opts);
    int rc = validate(base + L.q, base + L.k, base + L.v, base + L.o, B, Hq, Hkv, Sq, Skv, D, scale, &w);
    if (rc) return rc;
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    if (static_cast<long long>(B) * Hq * Sq == 0) return FMHA_OK;
    w.workspace = L.ws_bytes ? base + L.ws : nullptr;
    w.workspace_bytes = L.ws_bytes;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t esz = w.out_kind == FMHA_OUT_F32 ? 4 : 2;
    const size_t qb = static_cast<size_t>(Hq) * Sq * D * 2, kvb = static_cast<size_t>(Hkv) * Skv * D * 2;
    const size_t ob = static_cast<size_t>(Hq) * Sq * D * esz, lb = static_cast<size_t>(Hq) * Sq * 4;

    std::lock_guard<std::mutex> lock(g_host_mu);
    HostAux* aux = nullptr;
    if (L.chunks > 1) {
        aux = host_aux();
        if (!aux) return set_error(FMHA_ERR_CUDA, "fmha_fwd_host: cannot create the copy stream");
        // the copies must not overwrite staging that earlier work on `stream` still reads
        FMHA_CHECK_CUDA(cudaEventRecord(aux->start, st));
        FMHA_CHECK_CUDA(cudaStreamWaitEvent(aux->cs, aux->start, 0));
    }
    const auto* qh = static_cast<const uint8_t*>(q_host);
    const auto* kh = static_cast<const uint8_t*>(k_host);
    const auto* vh = static_cast<const uint8_t*>(v_host);
    for (int c = 0; c < L.chunks; ++c) {
        const int b0 = c * L.bc, nb = (B - b0 < L.bc) ? B - b0 : L.bc;
        cudaStream_t cs = aux ? aux->cs : st;
        FMHA_CHECK_CUDA(cudaMemcpyAsync(base + L.q + b0 * qb, qh + b0 * qb, nb * qb, cudaMemcpyHostToDevice, cs));
        FMHA_CHECK_CUDA(cudaMemcpyAsync(base + L.k + b0 * kvb, kh + b0 * kvb, nb * kvb, cudaMemcpyHostToDevice, cs));
        FMHA_CHECK_CUDA(cudaMemcpyAsync(base + L.v + b0 * kvb, vh + b0 * kvb, nb * kvb, cudaMemcpyHostToDevice, cs));
        if (aux) {
            FMHA_CHECK_CUDA(cudaEventRecord(aux->copied[c], cs));
            FMHA_CHECK_CUDA(cudaStreamWaitEvent(st, aux->copied[c], 0));
        }
        float* lse_dev = lse_host ? reinterpret_cast<float*>(base + L.lse + b0 * lb) : nullptr;
        rc = fmha_fwd_ex(base + L.q + b0 * qb, base + L.k + b0 * kvb, base + L.v + b0 * kvb, base + L.o + b0 * ob, lse_dev,
                         nb, Hq, Hkv, Sq, Skv, D, scale, stream, &w);
        if (rc) return rc;
        FMHA_CHECK_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + b0 * ob, base + L.o + b0 * ob, nb * ob,
                                        cudaMemcpyDeviceToHost, st));
        if (lse_host)
            FMHA_CHECK_CUDA(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse_host) + b0 * lb, lse_dev, nb * lb,
                                            cudaMemcpyDeviceToHost, st));
    }
    return FMHA_OK;
}

// ---- standalone NVFP4 ------------------------------------------------------------------------------------
static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

size_t nvfp4_scales_bytes(int64_t n)
{
    if (n < 0) return 0;
    return align16(static_cast<size_t>(n / 16)) + 16;
}

int nvfp4_quantize_scaled(const float* x, uint8_t* q, uint8_t* scales, int64_t n, const float* tensor_scale,
                          fmha_stream_t stream)
{
    if (!x || !q || !scales || !tensor_scale) return set_error(FMHA_ERR_INVALID, "nvfp4_quantize_scaled: NULL pointer");
    if (n < 0 || n % 16 != 0) return set_error(FMHA_ERR_INVALID, "nvfp4_quantize_scaled: n must be a non-negative multiple of 16");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3))
        return set_error(FMHA_ERR_INVALID, "nvfp4_quantize_scaled: x 16-byte, q 8-byte, tensor_scale 4-byte aligned");
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    if (n == 0) return FMHA_OK;
    return launch_nvfp4(x, q, scales, nullptr, nullptr, n, true, reinterpret_cast<cudaStream_t>(stream), tensor_scale);
}

int nvfp4_quantize(const float* x, uint8_t* q, uint8_t* scales, int64_t n, fmha_stream_t stream)
{
    if (!x || !q || !scales) return set_error(FMHA_ERR_INVALID, "nvfp4_quantize: NULL pointer");
    if (n < 0 || n % 16 != 0) return set_error(FMHA_ERR_INVALID, "nvfp4_quantize: n must be a non-negative multiple of 16");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7) || (reinterpret_cast<uintptr_t>(scales) & 15))
        return set_error(FMHA_ERR_INVALID, "nvfp4_quantize: x and scales 16-byte, q 8-byte aligned");
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");
    uint8_t* tail = scales + align16(static_cast<size_t>(n / 16));
    return launch_nvfp4(x, q, scales, reinterpret_cast<float*>(tail), reinterpret_cast<unsigned*>(tail + 4), n, false,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
