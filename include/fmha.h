/*
 * fmha.h - C ABI of the GB300 (sm_103a) fused attention library, libfmha.so.
 *
 * Computes O = softmax(scale * Q K^T) V over BF16 Q/K/V, with an online (running max / sum)
 * softmax and O rescale across key/value tiles, a split-KV decode path with a combine step,
 * and optional NVFP4 quantisation of O.  Sources:
 *   - "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md" (nvfp4-megamoe-kernel), kernel plan items 1-7:
 *     TMA loads of Q/K/V, tcgen05 MMA with a Tensor Memory accumulator, in-kernel softmax with
 *     O rescale, multi-KV-tile support, FP4 quantisation for NVFP4;
 *   - "CURRENT_ISSUE.md" @4b129c1, QK verify kernel: tensors laid out (B, H, S, D) contiguous;
 *   - "CURRENT_ISSUE.md" @57d67e6, "The 4x Bug": the raw S = Q K^T check (fmha_qk_gemm).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never allocates
 *     or frees device memory, never synchronises (except fmha_check_status) and launches only
 *     on `stream`.  Inputs are read-only; outputs must not alias inputs.
 *   - Kernels are launched with programmatic dependent launch (except while `stream` is being
 *     captured into a graph): a call's kernel may be placed on the SMs while the previous kernel of
 *     `stream` finishes, but touches no global memory until that kernel has completed, so calls keep
 *     plain stream order (a call may read what the previous kernel wrote, or overwrite what it read).
 *   - Layouts are contiguous, row-major: Q/O [B][Hq][Sq][D], K/V [B][Hkv][Skv][D], LSE [B][Hq][Sq].
 *   - Grouped-query attention: query head hq reads key/value head hq / (Hq / Hkv).
 *   - LSE is the natural logarithm of sum_j exp(scale * q.k_j) (scale included), FP32.
 *   - A key set of size 0 (seqlens_k[b] == 0) gives O = 0 and LSE = -inf.
 *   - Tensor pointers must be 16-byte aligned (LSE, seqlens_k, nvfp4_scale_in and out_amax:
 *     4-byte; the workspace: 256-byte).  D must be 64, 128 or 512 (16 is also accepted by
 *     fmha_qk_gemm).
 *   - Return value: FMHA_OK or an fmha_status code; nothing aborts or throws.  A failed call
 *     leaves a message for fmha_error_string(code) / fmha_last_error() of the calling thread.
 *   - Asynchronous device-side failures (a bounded wait inside a kernel that timed out) are
 *     reported by fmha_check_status().
 */
#ifndef FMHA_H_
#define FMHA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers; NULL = the legacy default stream. */
typedef struct CUstream_st* fmha_stream_t;

typedef enum {
    FMHA_OK = 0,
    FMHA_ERR_INVALID = 1,     /* bad argument: NULL pointer, Hq % Hkv != 0, unsupported D, misalignment */
    FMHA_ERR_UNSUPPORTED = 2, /* valid request that this library does not implement */
    FMHA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than fmha_workspace_size() */
    FMHA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or kernel launch failed */
    FMHA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (see fmha_check_status) */
    FMHA_ERR_RACE = 6         /* a split-KV merge counter never settled: calls sharing one
                                 workspace (or the allocation-free scratch) overlapped on the
                                 GPU, so some output rows may be unmerged (see fmha_check_status) */
} fmha_status;

typedef enum {
    FMHA_OUT_BF16 = 0,  /* out: BF16 [B,Hq,Sq,D] */
    FMHA_OUT_F32 = 1,   /* out: FP32 [B,Hq,Sq,D] */
    FMHA_OUT_NVFP4 = 2  /* out: packed E2M1 codes [B,Hq,Sq,D/2] (element 2i in bits 3:0),
                           plus out_scales / out_tensor_scale below */
} fmha_out_kind;

typedef struct {
    int out_kind;             /* fmha_out_kind; default FMHA_OUT_BF16 */
    const int32_t* seqlens_k; /* device int32[B], 0 <= seqlens_k[b] <= Skv: keys at or beyond
                                 seqlens_k[b] are never read (ragged batches); NULL = all Skv */
    int num_splits;           /* 0 = automatic split-KV; 1 = no split (each (b, kv-head) handled
                                 by one CTA, or by one CTA pair for D = 512; no workspace needed
                                 for BF16/F32 output).  With 0 and
                                 a workspace, causal or ragged problems on the 128-row path (more
                                 than 16 query rows per key/value head) also take their work items
                                 from a counter in the workspace (balanced across SMs); with 1, or
                                 no workspace, in a fixed order.  0 without a workspace acts as 1 */
    void* workspace;          /* device scratch of at least fmha_workspace_size() bytes (256-B
                                 aligned); contents on entry do not matter */
    size_t workspace_bytes;
    uint8_t* out_scales;      /* NVFP4: E4M3 block scales [B,Hq,Sq,D/16] */
    float* out_tensor_scale;  /* NVFP4: device float[1], the per-tensor scale s_g */
    float* out_f32;           /* optional, NVFP4 only: the FP32 O that was quantised */
    int causal;               /* 1: bottom-right aligned causal mask: with n keys, query i of Sq sees
                                 keys 0 .. i + n - Sq (a query that sees none gets O = 0,
                                 LSE = -inf); 0 = all keys */
    const float* nvfp4_scale_in; /* NVFP4, optional: device float[1], a given per-tensor scale s_g
                                 (e.g. an earlier step's max|O| / 2688).  Set: single pass, the
                                 attention epilogues write codes and block scales with this s_g
                                 directly; no amax pass, no FP32 staging, no workspace for NVFP4.
                                 Blocks beyond 6 * 448 * s_g saturate; an s_g that is not a
                                 positive finite number gives all-zero codes and scales;
                                 *out_tensor_scale receives s_g.  NULL: s_g = fp32(max|O| / 2688)
                                 of this O (two passes) */
    float* out_amax;          /* optional, NVFP4 only: device float[1], receives max|O| (FP32) of
                                 this call (with two passes it is also the max the quantiser uses) */
    int wide_variant;         /* D = 512 kernel (fmha_wide_variant); results agree within rounding */
} fmha_opts;

/* Kernel variants for D = 512 (the value columns are split over a pair of CTAs either way). */
typedef enum {
    FMHA_WIDE_AUTO = 0,        /* the faster one measured on GB300: FMHA_WIDE_INDEPENDENT */
    FMHA_WIDE_INDEPENDENT = 1, /* two independent CTAs: each loads every K tile, computes the full S */
    FMHA_WIDE_PAIR = 2         /* a cluster of two CTAs running pair MMAs (tcgen05 cta_group::2): each
                                  CTA loads half of every K tile, the PV product runs over a doubled
                                  contraction; dense keys only (with seqlens_k the independent CTAs
                                  run) */
} fmha_wide_variant;

/*
 * Attention forward with default options (BF16 output, dense keys, no workspace, no split).
 *   q: BF16 [B,Hq,Sq,D]; k, v: BF16 [B,Hkv,Skv,D]; out: BF16 [B,Hq,Sq,D];
 *   lse: FP32 [B,Hq,Sq] or NULL; scale: multiplies Q K^T before the softmax, a positive finite number
 *   (FMHA_ERR_INVALID otherwise: the kernels scale each row's maximum score after taking it).
 * Same as fmha_fwd_ex(..., opts = NULL): every (b, kv-head) unit is handled whole by one CTA (for
 * D = 512 by one CTA pair, each CTA writing its half of the value columns), so nothing needs a
 * workspace.  Decode shapes with few units leave SMs idle this way; fmha_fwd_ex with a workspace
 * splits the keys over every SM instead.
 */
int fmha_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
             int Sq, int Skv, int D, float scale, fmha_stream_t stream);

/*
 * Attention forward with options (output kind, ragged key lengths, causal mask, split-KV, NVFP4).
 * opts == NULL means all defaults.  Split-KV, the balanced work-item order and NVFP4 output need
 * opts->workspace; calls that share one workspace must be ordered on one stream.
 */
int fmha_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                int Sq, int Skv, int D, float scale, fmha_stream_t stream, const fmha_opts* opts);

/* Bytes of workspace fmha_fwd_ex needs for this problem and these options (0 if none). */
size_t fmha_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D, const fmha_opts* opts);

/*
 * Attention from host memory: copies Q, K and V to the device, runs fmha_fwd_ex, and copies O and
 * the LSE back, all ordered after the work already on `stream`.  Returns once everything is
 * enqueued: synchronise `stream` before reading out_host / lse_host.
 *   q_host, k_host, v_host: host BF16 arrays in the fmha_fwd layouts; out_host: host O, BF16 or
 *   (opts->out_kind == FMHA_OUT_F32) FP32 [B,Hq,Sq,D]; lse_host: host FP32 [B,Hq,Sq] or NULL.
 *   Page-locked host memory (cudaHostAlloc, cudaHostRegister) makes the copies asynchronous;
 *   pageable memory works, but the copies then hold up the calling thread.
 *   dev_buf: device memory of at least fmha_host_buffer_size() bytes, 256-byte aligned, owned by the
 *   caller; it stages Q, K, V, O and the LSE and holds the attention workspace, so the call
 *   allocates nothing.  Calls that share dev_buf must be ordered on one stream.
 *   opts: as for fmha_fwd_ex, limited to out_kind (BF16 or F32), num_splits, causal and
 *   wide_variant; seqlens_k, the NVFP4 fields and the workspace fields must be NULL / 0
 *   (FMHA_ERR_UNSUPPORTED otherwise).  opts == NULL: BF16 output, automatic split-KV.
 * With B >= 2 the batch runs in up to four chunks of whole batch entries, so that the copy of one
 * chunk's inputs overlaps the attention of the one before (an internal copy stream per device, joined
 * back to `stream` through events; calls from several host threads are serialised while they
 * enqueue).  Errors: FMHA_ERR_INVALID (NULL or bad arguments), FMHA_ERR_WORKSPACE (dev_buf missing,
 * misaligned or too small), FMHA_ERR_UNSUPPORTED, FMHA_ERR_CUDA; with an error nothing is enqueued,
 * except for FMHA_ERR_CUDA from a failing copy or launch, after which out_host is unspecified.
 */
int fmha_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* out_host, float* lse_host, int B,
                  int Hq, int Hkv, int Sq, int Skv, int D, float scale, fmha_stream_t stream, const fmha_opts* opts,
                  void* dev_buf, size_t dev_buf_bytes);

/* Bytes of device memory fmha_fwd_host needs for this problem and these options (0 if invalid). */
size_t fmha_host_buffer_size(int B, int Hq, int Hkv, int Sq, int Skv, int D, const fmha_opts* opts);

/*
 * NVFP4 quantisation of an FP32 tensor x[n], n % 16 == 0 (the NVFP4 step of the pages' kernel
 * plan, "FP4 quantization for NVFP4-1.1"):
 *   s_g = fp32(amax / (6 * 448)); per block of 16: sc = E4M3(amax_block / (6 s_g)) (round to
 *   nearest even, saturating at 448); code_i = E2M1(x_i / (sc * s_g)) (nearest even, saturating
 *   at 6, sign copied).  amax == 0 gives all-zero codes and scales.
 *   q: uint8[n/2] codes, element 2i in bits 3:0 and 2i+1 in bits 7:4.
 *   scales: nvfp4_scales_bytes(n) bytes: E4M3 scales [n/16], then at byte offset
 *   align16(n/16) the FP32 s_g, then 12 bytes the call uses as scratch.
 */
int nvfp4_quantize(const float* x, uint8_t* q, uint8_t* scales, int64_t n, fmha_stream_t stream);

/* Size in bytes of the `scales` buffer nvfp4_quantize needs for n values. */
size_t nvfp4_scales_bytes(int64_t n);

/*
 * NVFP4 encoding of x[n] (n % 16 == 0) with a given per-tensor scale: tensor_scale is a device
 * float[1] holding s_g.  q: n/2 bytes of E2M1 codes (as nvfp4_quantize); scales: n/16 bytes of
 * E4M3 block scales (no trailing s_g).  Same roundings as nvfp4_quantize; blocks beyond
 * 6 * 448 * s_g saturate and an s_g that is not a positive finite number gives all zeros.
 * Errors: FMHA_ERR_INVALID for NULL pointers, n < 0, n % 16 != 0, or x not 16-byte, q not 8-byte
 * or tensor_scale not 4-byte aligned.
 */
int nvfp4_quantize_scaled(const float* x, uint8_t* q, uint8_t* scales, int64_t n, const float* tensor_scale,
                          fmha_stream_t stream);

/*
 * Test hook: raw S = Q K^T in FP32, no scale ("CURRENT_ISSUE.md" @57d67e6, "The 4x Bug":
 * the single tcgen05 MMA product checked against a scalar dot product).
 *   q: BF16 [Sq,D], k: BF16 [Skv,D], s: FP32 [Sq,Skv]; D in {16, 64, 128, 512}.
 */
int fmha_qk_gemm(const void* q, const void* k, float* s, int Sq, int Skv, int D, fmha_stream_t stream);

/*
 * Test hook: layout self-checks of the building blocks.  Each writes its results to `out`
 * (device, `out_bytes` bytes, see the test-suite for the layouts) from inputs in `in`:
 *   which = 1: Tensor Memory round trip (tcgen05.st then tcgen05.ld, 32x32b shape);
 *   which = 2: O^T = V^T P^T with V^T an MN-major shared-memory operand (decode PV form);
 *   which = 3: O = P V with P in Tensor Memory and V MN-major in shared memory (TS form).
 */
int fmha_selftest(int which, const void* in, void* out, size_t out_bytes, int param, fmha_stream_t stream);

/*
 * Waits for `stream`, then returns FMHA_ERR_TIMEOUT if any kernel of this library timed out
 * in a bounded wait since the last call, FMHA_ERR_RACE if a split-KV merge found its arrival
 * counter changing under it (overlapping calls on one workspace), clearing that state in both
 * cases; FMHA_ERR_CUDA if the stream reports an error; else FMHA_OK.
 */
int fmha_check_status(fmha_stream_t stream);

/* Bounded-wait limit in SM clock cycles for later launches (0 = default, about 2 s). */
void fmha_set_wait_limit(long long cycles);

/*
 * Split-KV decode that allocates nothing.  The pages have no counterpart: it serves callers that
 * cannot hand the library a workspace, such as plug-ins and foreign-language bindings that see
 * only tensor pointers and have no allocator to ask, or latency-critical loops that must not call
 * cudaMalloc (it can synchronise the device and its latency is unbounded).
 *   Same arguments and results as fmha_fwd (BF16 out, optional LSE) plus seqlens_k (device
 *   int32[B] or NULL, as in fmha_opts); at most 16 query rows per key/value head, D = 64 or 128.
 *   The split-KV scratch (partials and tile prefix) is a fixed array of FMHA_NOALLOC_SCRATCH_BYTES
 *   inside the library, held by every GPU that loads it until the process exits; a problem that
 *   needs more returns FMHA_ERR_WORKSPACE with the size in fmha_last_error().  The library calls
 *   no allocation routine.  The first call on a device looks up that device's address of the
 *   array (make it before any stream capture).  All calls on a device share the array: calls that
 *   overlap on the GPU race and must be ordered by the caller.
 */
#define FMHA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
int fmha_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                            int Hkv, int Sq, int Skv, int D, float scale, const int32_t* seqlens_k,
                            fmha_stream_t stream);

/* Number of kernels this library has launched in this process (all devices, all threads). */
long long fmha_launch_count(void);

/*
 * Timing hook, one-shot and per calling thread: the next attention / quantisation call records
 * `start_event` on its stream immediately before launching its dominant kernel (the attention
 * kernel; the quantiser for nvfp4_quantize) and `stop_event` right after it.  Both are
 * cudaEvent_t handles owned by the caller; NULL, NULL clears the hook.
 */
void fmha_time_next_call(void* start_event, void* stop_event);

/* Static text for a status code. */
const char* fmha_error_string(int code);

/* Message of the last failing call on this thread ("" if none). */
const char* fmha_last_error(void);

/* Number of SMs of the current device as the library sees it (0 on failure). */
int fmha_num_sms(void);

#ifdef __cplusplus
}
#endif
#endif /* FMHA_H_ */
