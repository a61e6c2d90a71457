// Building-block kernels that are checked on their own before the attention kernels use them:
//   * qk_gemm_kernel: raw S = Q K^T through TMA (128-byte swizzle) -> tcgen05.mma (SS) -> TMEM ->
//     tcgen05.ld.  This is the check the pages were stuck on ("CURRENT_ISSUE.md" @57d67e6,
//     "The 4x Bug": one MMA of Q (one row padded to 128) against K, HD=16, SK=128); with integer
//     inputs the result must be bit-exact, which rules out any constant factor.
//   * selftest 1: Tensor Memory store/load round trip with the 32x32b shape, two stores in a row
//     (the pages' "TMEM multi-store bug" was a second 16x256b.x1 store failing).
//   * selftest 2: O^T = V^T P^T, V^T an MN-major operand written by TMA, P^T K-major written by
//     threads with the 128-byte swizzle (the decode kernel's PV product).
//   * selftest 3: O = P V with P in Tensor Memory (TS form) and V MN-major in shared memory (the
//     row-tile kernel's PV product).
//   * selftest 4: the CTA-pair MMA (tcgen05 cta_group::2, M = 256) in both operand forms: which rows of
//     A and D, and which half of B's columns, live in which CTA of the pair, and the two ways a pair
//     can signal across its CTAs (a commit or a TMA completion aimed at the other CTA's mbarrier, or
//     a relay through an ordinary cluster-scope arrive).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace atc_gb300 {
namespace {

constexpr int kQkThreads = 128;

// One CTA computes a 128 x 128 tile of S; D is walked in chunks of 64 (one 128-byte swizzle
// atom width), each chunk loaded by TMA and consumed by up to four K=16 MMAs.
__global__ void __launch_bounds__(kQkThreads) qk_gemm_kernel(const __grid_constant__ CUtensorMap qmap,
                                                             const __grid_constant__ CUtensorMap kmap, float* s,
                                                             int Sq, int Skv, int D, int* status,
                                                             long long limit)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;            // 128 rows x 128 B
    uint8_t* sB = smem + 16384;    // 128 rows x 128 B
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32;
    const int m0 = blockIdx.y * 128;
    const int n0 = blockIdx.x * 128;
    WaitCtl wc{&abort_flag, status, limit};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);

    if (threadIdx.x == 0) {
        const int chunks = (D + 63) / 64;
        for (int c = 0; c < chunks; ++c) {
            if (!aborted(wc)) {
                mbar_arrive_expect_tx(&bars[0], 2 * 16384);
                tma_load_2d(sA, &qmap, &bars[0], c * 64, m0);
                tma_load_2d(sB, &kmap, &bars[0], c * 64, n0);
            }
            mbar_wait(&bars[0], c & 1, wc);
            tc_fence_after();
            const int ksteps = min(4, (D - c * 64) / 16);
            if (!aborted(wc)) {
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint64_t da = sdesc_sw128(smem_u32(sA) + kk * 32, 16, 1024);
                    const uint64_t db = sdesc_sw128(smem_u32(sB) + kk * 32, 16, 1024);
                    mma_ss(tmem, da, db, idesc, (c > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars[1]);
            }
            mbar_wait(&bars[1], c & 1, wc);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Epilogue: warp w owns TMEM lanes 32w..32w+31 = rows m0 + 32w + lane.
    const int row = m0 + warp * 32 + static_cast<int>(lane_id());
    for (int col = 0; col < 128; col += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_addr(tmem, warp * 32, col), r);
        tmem_ld_wait();
        if (row < Sq && !aborted(wc)) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int n = n0 + col + i;
                if (n < Skv) s[static_cast<size_t>(row) * Skv + n] = __uint_as_float(r[i]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---- selftest 1: TMEM round trip --------------------------------------------------------------
__global__ void __launch_bounds__(128) tmem_roundtrip_kernel(uint32_t* out)
{
    __shared__ uint32_t tmem_base_slot;
    const int warp = threadIdx.x / 32;
    if (warp == 0) {
        tmem_alloc(&tmem_base_slot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    const uint32_t lane = warp * 32 + lane_id();
    uint32_t w[16];
    for (int chunk = 0; chunk < 4; ++chunk) {   // four stores in a row, columns 16*chunk..
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = lane * 1000u + chunk * 16u + i;
        tmem_st16(tmem_addr(tmem, warp * 32, chunk * 16), w);
    }
    tmem_st_wait();
    uint32_t r[32];
    tmem_ld32(tmem_addr(tmem, warp * 32, 0), r);
    tmem_ld_wait();
    for (int i = 0; i < 32; ++i) out[lane * 64 + i] = r[i];
    uint32_t r2[16];
    for (int chunk = 2; chunk < 4; ++chunk) {
        tmem_ld16(tmem_addr(tmem, warp * 32, chunk * 16), r2);
        tmem_ld_wait();
        for (int i = 0; i < 16; ++i) out[lane * 64 + chunk * 16 + i] = r2[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// Byte offset of BF16 element (row r, column k) in a K-major operand built of 128-byte-swizzled
// atoms of 64 columns; `atom_bytes` = rows * 128 (distance between 64-column atoms).
__device__ __forceinline__ uint32_t sw128_offset(int r, int k, uint32_t atom_bytes)
{
    const int a = k >> 6, kk = k & 63;
    return a * atom_bytes + r * 128 + ((((kk >> 3) ^ (r & 7)) & 7) << 4) + ((kk & 7) << 1);
}

// ---- selftest 2: O^T[d][q] = sum_kv V[kv][d] P[q][kv], D = 64 or 128, 16 query columns ----------
__global__ void __launch_bounds__(128) pv_swapab_kernel(const __grid_constant__ CUtensorMap vmap,
                                                        const uint16_t* P, float* out, int D, int* status,
                                                        long long limit)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sV = smem;                 // D/64 boxes of 128 kv rows x 128 B
    uint8_t* sP = smem + 2 * 16384;     // 2 atoms of 16 q rows x 128 B
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    WaitCtl wc{&abort_flag, status, limit};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_slot, 32);
        tmem_relinquish();
    }
    // P^T operand: thread t writes kv column t of all 16 query rows.
    for (int q = 0; q < 16; ++q) {
        const int kv = threadIdx.x;
        *reinterpret_cast<uint16_t*>(sP + sw128_offset(q, kv, 2048)) = P[q * 128 + kv];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    if (threadIdx.x == 0) {
        const int boxes = D / 64;
        mbar_arrive_expect_tx(&bars[0], boxes * 16384);
        for (int bx = 0; bx < boxes; ++bx) tma_load_2d(sV + bx * 16384, &vmap, &bars[0], bx * 64, 0);
        mbar_wait(&bars[0], 0, wc);
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 16, true, false);
        const uint32_t lbo = (D >= 128) ? 16384u : 0u;   // second 64-row block of M (d); D=64: repeat
        if (!aborted(wc)) {
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t da = sdesc_sw128(smem_u32(sV) + ks * 2048, lbo, 1024);
                const uint64_t db = sdesc_sw128(smem_u32(sP) + (ks >> 2) * 2048 + (ks & 3) * 32, 16, 1024);
                mma_ss(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&bars[1]);
        }
        mbar_wait(&bars[1], 0, wc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t r[16];
    tmem_ld16(tmem_addr(tmem, warp * 32, 0), r);
    tmem_ld_wait();
    const int lane = threadIdx.x;
    for (int i = 0; i < 16; ++i) out[lane * 16 + i] = __uint_as_float(r[i]);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 32);
}

// ---- selftest 3: O[q][d] = sum_kv P[q][kv] V[kv][d], P in TMEM, N = D in {64, 128, 256} --------
__global__ void __launch_bounds__(128) pv_ts_kernel(const __grid_constant__ CUtensorMap vmap, const uint16_t* P,
                                                    float* out, int D, int* status, long long limit)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sV = smem;   // D/64 boxes of 128 kv rows x 128 B
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    WaitCtl wc{&abort_flag, status, limit};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    const uint32_t p_cols = 256;   // P at columns 256..319, O at columns 0..D-1
    // P row q = thread: 128 BF16 -> 64 packed columns (element 2c in bits 15:0).
    {
        const int q = threadIdx.x;
        for (int chunk = 0; chunk < 4; ++chunk) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = (chunk * 16 + i) * 2;
                w[i] = static_cast<uint32_t>(P[q * 128 + k]) | (static_cast<uint32_t>(P[q * 128 + k + 1]) << 16);
            }
            tmem_st16(tmem_addr(tmem, warp * 32, p_cols + chunk * 16), w);
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const int boxes = D / 64;
        mbar_arrive_expect_tx(&bars[0], boxes * 16384);
        for (int bx = 0; bx < boxes; ++bx) tma_load_2d(sV + bx * 16384, &vmap, &bars[0], bx * 64, 0);
        mbar_wait(&bars[0], 0, wc);
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, D, false, true);
        if (!aborted(wc)) {
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t db = sdesc_sw128(smem_u32(sV) + ks * 2048, 16384, 1024);
                mma_ts(tmem, tmem + p_cols + ks * 8, db, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&bars[1]);
        }
        mbar_wait(&bars[1], 0, wc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int q = threadIdx.x;
    for (int col = 0; col < D; col += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_addr(tmem, warp * 32, col), r);
        tmem_ld_wait();
        for (int i = 0; i < 16; ++i) out[q * D + col + i] = __uint_as_float(r[i]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- selftest 4: CTA-pair MMA -----------------------------------------------------------------
// flags bit 0 = 0 (SS): D[256][128] = A[256][64] B[128][64]^T, both K-major; CTA r of the pair loads A
//   rows 128r.. and B rows 64r.. into its own shared memory.
// flags bit 0 = 1 (TS): D[256][256] = A[256][32] V[32][256]; each CTA writes its 128 rows of A into its
//   own Tensor Memory; V is MN-major and CTA r loads its columns 128r..128r+127.
// flags bit 1: the leader's commit also arrives on the odd CTA's barrier directly (else the leader
//   relays the completion with a cluster-scope arrive).  bit 2: the odd CTA's TMA counts its bytes
//   on the leader's barrier (else the odd CTA waits for its own copy and relays an arrive).
// out: [2][128][N] FP32 (CTA rank, TMEM lane, column), then 2 floats: 1 where a CTA's wait gave up.
constexpr int kPairRegion = 32768;
constexpr int kPairSmem = 2 * kPairRegion + 1024;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128)
    pair_mma_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap, const uint16_t* A,
                    float* out, int flags, int* status, long long limit)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                  // SS: 128 rows x 128 B
    uint8_t* sB = smem + kPairRegion;    // SS: 64 rows x 128 B; TS: two atoms of 32 rows x 128 B
    __shared__ uint64_t full_local, full_pair, done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    const uint32_t rank = cluster_ctarank();
    const int ts = flags & 1;
    const bool direct_commit = (flags & 2) != 0, direct_tma = (flags & 4) != 0;
    const int N = ts ? 256 : 128;
    WaitCtl wc{&abort_flag, status, limit};
    // both regions zeroed, so a read outside what the copies wrote shows up as zeros
    for (int i = threadIdx.x; i < 2 * kPairRegion / 16; i += 128) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&full_local, 1);
        mbar_init(&full_pair, direct_tma ? 1 : 2);
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(&tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the other CTA's barriers are initialised before anything arrives on them
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t leader_full = mapa_shared(smem_u32(&full_pair), 0);
    const uint32_t other_done = mapa_shared(smem_u32(&done), rank ^ 1u);
    if (ts) {
        // this CTA's rows of A as packed BF16 pairs at Tensor Memory column 256 (element 2c in bits 15:0)
        const int row = 128 * static_cast<int>(rank) + static_cast<int>(threadIdx.x);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = static_cast<uint32_t>(A[row * 32 + 2 * i]) | (static_cast<uint32_t>(A[row * 32 + 2 * i + 1]) << 16);
        tmem_st16(tmem_addr(tmem, warp * 32, 256), w);
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' Tensor Memory operands are written
    tc_fence_after();
    const uint32_t own = ts ? 8192u : 16384u + 8192u;   // bytes this CTA loads
    if (threadIdx.x == 0) {
        if (rank == 0) {
            mbar_arrive_expect_tx(&full_pair, direct_tma ? 2 * own : own);
            if (!ts) tma_load_3d(sA, &amap, &full_pair, 0, 0, 0);
            if (!ts) tma_load_3d(sB, &bmap, &full_pair, 0, 0, 0);
            else {
                tma_load_3d(sB, &bmap, &full_pair, 0, 0, 0);
                tma_load_3d(sB + 4096, &bmap, &full_pair, 64, 0, 0);
            }
        } else if (direct_tma) {
            if (!ts) tma_load_3d_pair(sA, &amap, leader_full, 0, 128, 0);
            if (!ts) tma_load_3d_pair(sB, &bmap, leader_full, 0, 64, 0);
            else {
                tma_load_3d_pair(sB, &bmap, leader_full, 128, 0, 0);
                tma_load_3d_pair(sB + 4096, &bmap, leader_full, 192, 0, 0);
            }
        } else {
            mbar_arrive_expect_tx(&full_local, own);
            if (!ts) tma_load_3d(sA, &amap, &full_local, 0, 128, 0);
            if (!ts) tma_load_3d(sB, &bmap, &full_local, 0, 64, 0);
            else {
                tma_load_3d(sB, &bmap, &full_local, 128, 0, 0);
                tma_load_3d(sB + 4096, &bmap, &full_local, 192, 0, 0);
            }
            if (mbar_wait(&full_local, 0, wc)) mbar_arrive_cluster(leader_full);
        }
        if (rank == 0) {
            if (mbar_wait_cluster(&full_pair, 0, wc)) {
                tc_fence_after();
                if (!ts) {
                    constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, false);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss_pair(tmem, sdesc_sw128(smem_u32(sA) + kk * 32, 16, 1024),
                                    sdesc_sw128(smem_u32(sB) + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
                } else {
                    constexpr uint32_t idesc = idesc_bf16_f32(256, 256, false, true);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_ts_pair(tmem, tmem + 256 + ks * 8, sdesc_sw128(smem_u32(sB) + ks * 2048, 4096, 1024), idesc,
                                    ks > 0 ? 1u : 0u);
                }
                mma_commit_pair(smem_u32(&done));
                if (direct_commit) mma_commit_pair(other_done);
                if (!direct_commit && mbar_wait(&done, 0, wc)) mbar_arrive_cluster(other_done);
            }
        }
    }
    __syncwarp();
    const bool ok = mbar_wait_cluster(&done, 0, wc);
    tc_fence_after();
    for (int c = 0; c < N; c += 32) {
        uint32_t r[32];
        tmem_ld32p(tmem_addr(tmem, warp * 32, c), r);
        tmem_ld_wait();
        float* o = out + (static_cast<size_t>(rank) * 128 + threadIdx.x) * N + c;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
    }
    if (threadIdx.x == 0) out[2 * 128 * N + rank] = (ok && !aborted(wc)) ? 0.f : 1.f;
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA frees Tensor Memory or exits while the other may still use its barriers
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

}  // namespace

int launch_qk_gemm(const void* q, const void* k, float* s, int Sq, int Skv, int D, cudaStream_t st)
{
    CUtensorMap qmap, kmap;
    const uint32_t box[2] = {64, 128};
    uint64_t qd[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Sq)};
    uint64_t kd[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Skv)};
    uint64_t stride[1] = {static_cast<uint64_t>(D) * 2};
    int rc = make_tmap_bf16(&qmap, q, 2, qd, stride, box);
    if (rc) return rc;
    rc = make_tmap_bf16(&kmap, k, 2, kd, stride, box);
    if (rc) return rc;
    const size_t smem = 2 * 16384 + 1024;
    FMHA_CHECK_CUDA(cudaFuncSetAttribute(qk_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid((Skv + 127) / 128, (Sq + 127) / 128);
    qk_gemm_kernel<<<grid, kQkThreads, smem, st>>>(qmap, kmap, s, Sq, Skv, D, device_status_ptr(), wait_limit());
    FMHA_CHECK_LAUNCH("qk_gemm_kernel");
    count_launch();
    return FMHA_OK;
}

int launch_selftest(int which, const void* in, void* out, size_t out_bytes, int param, cudaStream_t st)
{
    if (which == 1) {
        if (out_bytes < 128 * 64 * 4) return set_error(FMHA_ERR_INVALID, "selftest 1: out too small");
        tmem_roundtrip_kernel<<<1, 128, 0, st>>>(static_cast<uint32_t*>(out));
        FMHA_CHECK_LAUNCH("tmem_roundtrip_kernel");
        return FMHA_OK;
    }
    if (which == 2 || which == 3) {
        const int D = param;
        const bool ok = (which == 2) ? (D == 64 || D == 128) : (D == 64 || D == 128 || D == 256);
        if (!ok) return set_error(FMHA_ERR_INVALID, "selftest: unsupported D");
        const size_t need = (which == 2) ? 128 * 16 * 4 : static_cast<size_t>(128) * D * 4;
        if (out_bytes < need) return set_error(FMHA_ERR_INVALID, "selftest: out too small");
        // in = V [128][D] BF16, then P (which 2: [16][128], which 3: [128][128]) BF16
        CUtensorMap vmap;
        const uint32_t box[2] = {64, 128};
        uint64_t dims[2] = {static_cast<uint64_t>(D), 128};
        uint64_t stride[1] = {static_cast<uint64_t>(D) * 2};
        int rc = make_tmap_bf16(&vmap, in, 2, dims, stride, box);
        if (rc) return rc;
        const uint16_t* P = static_cast<const uint16_t*>(in) + 128 * D;
        if (which == 2) {
            const size_t smem = 2 * 16384 + 4096 + 1024;
            FMHA_CHECK_CUDA(cudaFuncSetAttribute(pv_swapab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            pv_swapab_kernel<<<1, 128, smem, st>>>(vmap, P, static_cast<float*>(out), D, device_status_ptr(),
                                                   wait_limit());
            FMHA_CHECK_LAUNCH("pv_swapab_kernel");
        } else {
            const size_t smem = static_cast<size_t>(D / 64) * 16384 + 1024;
            FMHA_CHECK_CUDA(cudaFuncSetAttribute(pv_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            pv_ts_kernel<<<1, 128, smem, st>>>(vmap, P, static_cast<float*>(out), D, device_status_ptr(),
                                               wait_limit());
            FMHA_CHECK_LAUNCH("pv_ts_kernel");
        }
        return FMHA_OK;
    }
    if (which == 4) {
        // in: A (SS: [256][64], TS: [256][32]) then B (SS: [128][64], TS: V [32][256]), BF16 row-major
        const int ts = param & 1;
        const int N = ts ? 256 : 128;
        if (out_bytes < (static_cast<size_t>(2) * 128 * N + 2) * 4) return set_error(FMHA_ERR_INVALID, "selftest 4: out too small");
        const uint16_t* A = static_cast<const uint16_t*>(in);
        const uint16_t* B = A + (ts ? 256 * 32 : 256 * 64);
        CUtensorMap amap, bmap;
        {
            const uint64_t dims[3] = {64, 256, 1};
            const uint64_t strides[2] = {128, 256 * 128};
            const uint32_t box[3] = {64, 128, 1};
            int rc = make_tmap_bf16(&amap, A, 3, dims, strides, box);
            if (rc) return rc;
        }
        {
            const uint64_t dims[3] = {ts ? 256u : 64u, ts ? 32u : 128u, 1};
            const uint64_t strides[2] = {ts ? 512u : 128u, ts ? 32u * 512u : 128u * 128u};
            const uint32_t box[3] = {64, ts ? 32u : 64u, 1};
            int rc = make_tmap_bf16(&bmap, B, 3, dims, strides, box);
            if (rc) return rc;
        }
        FMHA_CHECK_CUDA(cudaFuncSetAttribute(pair_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem));
        pair_mma_kernel<<<2, 128, kPairSmem, st>>>(amap, bmap, A, static_cast<float*>(out), param, device_status_ptr(),
                                                   wait_limit());
        FMHA_CHECK_LAUNCH("pair_mma_kernel");
        return FMHA_OK;
    }
    return set_error(FMHA_ERR_INVALID, "selftest: unknown test id");
}

}  // namespace atc_gb300
