/*
 * CPU oracle for fused multi-head attention and NVFP4 quantisation of its output.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load this library. The product path (the CUDA
 * library) never calls it, links it or shares code with it.
 *
 * Plain C99, FP64 arithmetic, no tiling, no fusion, no online softmax: each function is
 * the textbook definition written out so that it can be checked by eye.
 *
 * Sources (pages "nvfp4-megamoe-kernel" CURRENT_ISSUE.md and NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md):
 *   - the computation: "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md", kernel plan items 1-7
 *     (QK GEMM, in-kernel softmax with O rescale, PV GEMM, FP4 quantisation);
 *   - tensor layout (B, H, S, D) contiguous: "CURRENT_ISSUE.md" @4b129c1, the Q load of the
 *     QK verify kernel (batch stride H*HD);
 *   - the raw S = Q*K^T check: "CURRENT_ISSUE.md" @57d67e6, "The 4x Bug" (HD=16, SK=128).
 * The NVFP4 format (E2M1 values, 16-element blocks, E4M3 block scales, FP32 per-tensor
 * scale amax/(6*448)) is fixed by the benchmark spec of this library; the pages name
 * the format ("NVFP4-1.1") without defining it.
 */
#ifndef FMHA_ORACLE_H
#define FMHA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Attention rows.  q [B,Hq,Sq,D], k/v [B,Hkv,Skv,D], BF16 bit patterns, contiguous.
 * rows: flat query-row indices r = (b*Hq + hq)*Sq + i (NULL = all B*Hq*Sq rows, in order).
 * seqlens_k: int32[B] valid keys per batch (NULL = Skv for all).
 * causal: 0, or 1 for the bottom-right aligned causal mask: with n valid keys, query i
 *         (0 <= i < Sq) sees keys j <= i + n - Sq only.
 * o: double[nrows][D]; lse: double[nrows] (natural log of sum_j exp(s_j)).
 * Empty key set (no visible key): o = 0, lse = -inf.
 * Returns 0, or -1 on bad arguments.  Uses OpenMP threads when built with -fopenmp. */
int oracle_attention_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int B, int Hq, int Hkv, int Sq, int Skv, int D, double scale,
                         const int32_t* seqlens_k, int causal, const int64_t* rows, int64_t nrows,
                         double* o, double* lse);

/* Raw scores S[i][j] = sum_d q[i][d]*k[j][d], no scale. q [Sq,D], k [Skv,D] BF16 bits. */
int oracle_qk_f64(const uint16_t* q, const uint16_t* k, int Sq, int Skv, int D, double* s);

/* NVFP4 quantisation of x[n] (n % 16 == 0).
 * codes: uint8[n/2], element 2i in bits 3:0, element 2i+1 in bits 7:4, code = sign<<3 | e<<1 | m.
 * scales: uint8[n/16], E4M3FN bit patterns.  *tensor_scale = s_g (dequantised x ~ e2m1 * e4m3 * s_g). */
int oracle_nvfp4_quantize(const float* x, int64_t n, uint8_t* codes, uint8_t* scales,
                          float* tensor_scale);

/* The same encoding with a given per-tensor scale s_g (steps 2-4 only); s_g that is not a positive
 * finite number gives all-zero codes and scales. */
int oracle_nvfp4_quantize_scaled(const float* x, int64_t n, float s_g, uint8_t* codes, uint8_t* scales);

/* Helpers exposed for the self-tests. */
double oracle_e4m3_decode(uint8_t code);            /* E4M3FN bits -> value (NaN for 0x7F/0xFF) */
uint8_t oracle_e4m3_round(double v);                /* |v| >= 0 -> nearest E4M3FN, ties even, saturating */
double oracle_e2m1_decode(uint8_t code);            /* 4-bit code -> value */
uint8_t oracle_e2m1_round(double v);                /* v -> nearest E2M1, ties even, saturating, sign kept */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
