/*
 * CPU FP64 oracle: attention O = softmax(scale * Q K^T) V, and the raw Q K^T product.
 * TEST INFRASTRUCTURE ONLY (see oracle.h): never linked into or called by the CUDA library.
 *
 * What it follows:
 *   - "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md" (nvfp4-megamoe-kernel), kernel plan: the QK GEMM,
 *     the softmax over keys with the running O rescale, and the PV GEMM.  The rescale is only a
 *     route to the same value, so the oracle computes the plain two-pass softmax instead.
 *   - "CURRENT_ISSUE.md" @4b129c1, QK verify kernel: Q laid out (B, H, 1, HD) with batch stride
 *     H*HD, i.e. contiguous BHSD; the same layout is taken for K, V and O.
 *   - "CURRENT_ISSUE.md" @57d67e6, "The 4x Bug": the raw S = Q K^T product (no scale) that the
 *     MMA result is checked against.
 * Readings where the pages are silent: grouped-query attention maps query head hq to key/value
 * head hq / (Hq/Hkv); LSE is the natural log of sum_j exp(s_j) with the scale included; keys at
 * or beyond seqlens_k[b] do not exist; an empty key set gives O = 0 and LSE = -inf.
 * The causal variant (the pages aim at decode; causal masking is the usual companion of prefill
 * and of multi-token decode) aligns the mask bottom-right: with n keys, query i of Sq sees keys
 * 0 .. i + n - Sq, i.e. the last query sees every key.
 */
#include "oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* BF16 -> double is exact: the BF16 bits are the top half of an FP32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_attention_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int B, int Hq, int Hkv, int Sq, int Skv, int D, double scale,
                         const int32_t* seqlens_k, int causal, const int64_t* rows, int64_t nrows,
                         double* o, double* lse)
{
    if (!q || !k || !v || !o || B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || D <= 0)
        return -1;
    if (Hq % Hkv != 0)
        return -1;
    const int64_t total = (int64_t)B * Hq * Sq;
    if (!rows)
        nrows = total;
    const int group = Hq / Hkv;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t t = 0; t < nrows; ++t) {
        const int64_t r = rows ? rows[t] : t;
        if (r < 0 || r >= total) {
            bad |= 1;
            continue;
        }
        const int64_t i = r % Sq;
        const int64_t hq = (r / Sq) % Hq;
        const int64_t b = r / ((int64_t)Sq * Hq);
        const int64_t kvh = hq / group;
        int64_t n = seqlens_k ? seqlens_k[b] : Skv;
        if (n < 0 || n > Skv) {
            bad |= 1;
            continue;
        }
        if (causal) {
            /* keys 0 .. i + n - Sq are visible */
            const int64_t last = i + n - Sq;
            n = last < 0 ? 0 : (last + 1 < n ? last + 1 : n);
        }
        const uint16_t* qrow = q + r * D;
        const uint16_t* kbase = k + (b * Hkv + kvh) * (int64_t)Skv * D;
        const uint16_t* vbase = v + (b * Hkv + kvh) * (int64_t)Skv * D;
        double* orow = o + t * D;

        if (n == 0) {
            for (int d = 0; d < D; ++d)
                orow[d] = 0.0;
            if (lse)
                lse[t] = -INFINITY;
            continue;
        }

        /* scores s_j = scale * sum_d q_d k_{j,d} */
        double* s = (double*)malloc((size_t)n * sizeof(double));
        if (!s) {
            bad |= 1;
            continue;
        }
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += bf16_bits_to_double(qrow[d]) * bf16_bits_to_double(kbase[j * D + d]);
            s[j] = scale * acc;
        }
        /* pass 1: the maximum, pass 2: the exponentials and their sum */
        double m = s[0];
        for (int64_t j = 1; j < n; ++j)
            if (s[j] > m)
                m = s[j];
        double l = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        /* o_d = sum_j p_j v_{j,d} / l */
        for (int d = 0; d < D; ++d)
            orow[d] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            const double p = s[j];
            const uint16_t* vrow = vbase + j * D;
            for (int d = 0; d < D; ++d)
                orow[d] += p * bf16_bits_to_double(vrow[d]);
        }
        for (int d = 0; d < D; ++d)
            orow[d] /= l;
        if (lse)
            lse[t] = m + log(l);
        free(s);
    }
    return bad ? -1 : 0;
}

int oracle_qk_f64(const uint16_t* q, const uint16_t* k, int Sq, int Skv, int D, double* s)
{
    if (!q || !k || !s || Sq < 0 || Skv < 0 || D <= 0)
        return -1;
    for (int i = 0; i < Sq; ++i)
        for (int j = 0; j < Skv; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += bf16_bits_to_double(q[(int64_t)i * D + d]) *
                       bf16_bits_to_double(k[(int64_t)j * D + d]);
            s[(int64_t)i * Skv + j] = acc;
        }
    return 0;
}
