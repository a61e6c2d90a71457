// Host-side helpers shared by the library's translation units: error reporting, the device
// status word, bounded-wait limit, TMA tensor-map encoding, and the launch functions each
// kernel file exports to the C-ABI layer (api.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/fmha.h"

namespace atc_gb300 {

// ---- errors ------------------------------------------------------------------------------
int set_error(int code, const std::string& msg);  // records msg for fmha_last_error(), returns code
int cuda_error(cudaError_t e, const char* what);  // FMHA_ERR_CUDA with the CUDA message
#define FMHA_CHECK_CUDA(expr)                                      \
    do {                                                           \
        cudaError_t e__ = (expr);                                  \
        if (e__ != cudaSuccess) return ::atc_gb300::cuda_error(e__, #expr); \
    } while (0)
#define FMHA_CHECK_LAUNCH(what)                                                 \
    do {                                                                        \
        cudaError_t e__ = cudaGetLastError();                                   \
        if (e__ != cudaSuccess) return ::atc_gb300::cuda_error(e__, what);           \
    } while (0)

// ---- device status word and wait limit -------------------------------------------------------
int* device_status_ptr();   // device address of the library's status word (current device)
long long wait_limit();     // cycles
int num_sms();              // SMs of the current device

// ---- launch accounting and the dominant-kernel timing hook ---------------------------------------
void count_launch(int n = 1);                 // kernels this library launched (process-wide)
unsigned long long next_call_tag();           // unique per call (48 bits, never 0): tags arrival counters
// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) once per (kernel, device)
cudaError_t set_smem_limit_once(const void* func, int bytes);
void timing_mark_begin(cudaStream_t st);      // records the pending start event (one-shot), if any
void timing_mark_end(cudaStream_t st);        // records the pending stop event and clears the hook

// ---- programmatic dependent launch --------------------------------------------------------------
// The library's kernels are launched with the programmatic-serialization attribute, so that a call's
// kernel is placed on SMs and runs its prologue while the previous kernel of the stream drains
// (back-to-back decode B8 H32 Skv4096 on one GB300: 85.3 -> 83.1 us per call).  Each of them executes
// griddepcontrol.wait before its first global memory access (ptx.cuh).  Writes the attribute and
// returns 1, or returns 0 while the stream is being captured into a graph.
unsigned pdl_attribute(cudaStream_t st, cudaLaunchAttribute* attr);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = pdl_attribute(st, attr);
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- TMA ---------------------------------------------------------------------------------------
// Encodes a tiled map over a BF16 tensor with up to 3 dims (dim 0 innermost), 128-byte swizzle,
// out-of-bounds elements filled with zero.  dims/box in elements, strides in bytes (dims 1..).
int make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box);

// ---- launchers (each validates nothing: api.cu has done it) ----------------------------------
int launch_qk_gemm(const void* q, const void* k, float* s, int Sq, int Skv, int D, cudaStream_t st);
int launch_selftest(int which, const void* in, void* out, size_t out_bytes, int param, cudaStream_t st);

struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;          // final output (BF16 / F32) or NULL when the output is NVFP4
    float* lse;         // may be NULL
    int B, Hq, Hkv, Sq, Skv, D;
    float scale;
    const int32_t* seqlens;  // device, may be NULL
    int out_kind;            // FMHA_OUT_*
    float* out_f32;          // FP32 O destination (NVFP4 path), else NULL
    float* amax_slot;        // NVFP4 path: |O| max accumulator (uint bits), else NULL
    int causal;              // bottom-right aligned causal mask
    // single-pass NVFP4 (given s_g): the epilogues encode O directly, else all NULL
    const float* nv_sg;      // device s_g
    uint8_t* nv_codes;       // E2M1 codes [rows][D/2]
    uint8_t* nv_scales;      // E4M3 block scales [rows][D/16]
    float* nv_ts;            // receives s_g
    int wide_variant;        // D = 512: FMHA_WIDE_* (fmha_opts.wide_variant)
};

// Decode / small-group path (query rows per key/value head <= 16): swap-AB kernels.
size_t decode_workspace_bytes(const AttnArgs& a, int splits_mode);
int launch_decode(const AttnArgs& a, int num_splits, void* ws, size_t ws_bytes, cudaStream_t st);

// Row-tile path (128 query rows per tile).  sched_mode != 1 (a caller workspace is in use): causal
// and ragged problems take their work items from a counter in the workspace.
size_t prefill_workspace_bytes(const AttnArgs& a, int sched_mode);
int launch_prefill(const AttnArgs& a, int sched_mode, void* ws, size_t ws_bytes, cudaStream_t st);

// Wide-head path (D = 512): CTA pairs split the value columns, stream-K over 128-key tiles, or
// whole units per pair without a workspace when num_splits == 1.
size_t wide_workspace_bytes(const AttnArgs& a, int num_splits);
int launch_wide(const AttnArgs& a, int num_splits, void* ws, size_t ws_bytes, cudaStream_t st);

// NVFP4
// NVFP4 quantiser: s_g from sg_in when given (no amax pass), else from *amax_bits (computed here
// unless amax_ready).
int launch_nvfp4(const float* x, uint8_t* codes, uint8_t* scales, float* tensor_scale, unsigned* amax_bits,
                 int64_t n, bool amax_ready, cudaStream_t st, const float* sg_in = nullptr);

}  // namespace atc_gb300
