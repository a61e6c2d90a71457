// Row-tile attention: 128 query rows per MMA tile, for problems with more than 16 query rows per
// key/value head (prefill, large GQA groups).
//
// Follows the kernel plan of "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md" (nvfp4-megamoe-kernel): TMA for
// Q/K/V, tcgen05 MMA into a Tensor Memory accumulator, softmax warps reading S with tcgen05.ld and
// writing P back to Tensor Memory for the PV product ("SS" QK, "TS" PV with A = P in TMEM), the
// in-kernel softmax with O rescale over several KV tiles.  The GB300 design:
//
//  * A persistent CTA owns a PAIR of 128-row query tiles of one (b, kv-head) unit and streams
//    that unit's K/V tiles (128 keys) through TMA rings.  Two softmax warpgroups (one per query
//    tile) ping-pong: while one computes exponentials the tensor core runs the other's MMAs.
//  * Tensor Memory (512 columns) for D = 64: S0, S1 (128 each), P0, P1 (64 each, BF16 pairs),
//    O0, O1 (64 each).  For D = 128 P is written over the first half of its S buffer.
//  * Rows are one per thread (thread t of a warpgroup owns TMEM lane t), so row max / sum need
//    no cross-thread reduction.
//  * Lazy rescale: the running max m used for P only moves when a tile's max exceeds it by more
//    than 2^8 (log2 units), so O in TMEM is rescaled (ld/mul/st) only a few times per row; P
//    stays <= 256, and the final O / l and LSE use the same m, so the result is exact.
//  * One MMA thread polls the readiness of every pending QK / PV (non-blocking mbarrier tests)
//    and issues whichever can go, so a slow softmax of one tile never blocks the other's MMAs.
//  * Work items (unit, query-tile pair) come from a global atomic counter when the caller gives a
//    workspace (causal and ragged problems, whose items differ in size), else in a fixed strided
//    order.  The TMA warp claims the next item once it has issued the loads of the current one and
//    hands item numbers to the MMA and softmax warps through a small shared-memory ring.  Causal
//    items are numbered heaviest first within groups of units whose K/V fit comfortably in L2, so
//    the greedy claim order approximates longest-job-first and the light items fill the tail.
//  * Every wait is bounded (clock64 limit); a timeout sets the device status word and the CTA
//    drains without issuing more copies or MMAs.
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_dev.cuh"
#include "ptx.cuh"

namespace atc_gb300 {
namespace {

constexpr int kTM = 128;          // query rows per tile (MMA M)
// Threads: 2 softmax warpgroups + TMA warp + MMA warp.  The counter-order kernel adds two idle warps
// so that its third warpgroup is whole (setmaxnreg acts on whole warpgroups) and splits registers:
// the launch gives every thread 168 (384 x 168 = 64512 of the SM's 65536); the third warpgroup drops
// to kRegsCtl and the softmax warpgroups rise to kRegsSoftmax, which holds a whole row of S (128
// floats) and its packed P without spilling: 2*128*208 + 128*88 = 64512, and on each SM quarter
// (warps w, w+4, w+8) the control warp frees exactly what its two softmax warps take.  The
// fixed-order kernel keeps 10 warps at 168 registers, which measured faster for dense problems.
template <bool RING>
constexpr int prefill_threads() { return RING ? 384 : 320; }
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsCtl = 88;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsCtl <= prefill_threads<true>() * 168, "register split exceeds the launch allocation");
static_assert(2 * kRegsSoftmax + kRegsCtl <= 512, "register split exceeds an SM quarter");
constexpr float kLog2eP = 1.4426950408889634f;
constexpr float kLn2P = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kItemSlots = 4;     // work-item ring between the TMA warp and the consumers

template <int D>
struct PrefillCfg {
    // 128 keys per tile (a QK MMA of N = 128 runs at the full rate; N = 64 at 64 %).  At D = 64
    // each query tile has its own S buffer.  At D = 128 the two O buffers take 256 columns, so the
    // two query tiles take one S buffer in turns: a QK waits for the other tile's softmax to read S,
    // never for its own PV (P has buffers of its own).
    static constexpr bool kSharedS = (D == 128);
    static constexpr int kTN = 128;
    static constexpr int kAtoms = D / 64;
    static constexpr int kQStages = (D == 64) ? 2 : 1;
    static constexpr int kStages = (D == 64) ? 4 : 2;
    static constexpr int kQTileBytes = kAtoms * kTM * 128;
    static constexpr int kQBytes = 2 * kQTileBytes;
    static constexpr int kKVBytes = kAtoms * kTN * 128;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQStages * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kSmemBytes = kOffV + kStages * kKVBytes + 1024;
    // Tensor Memory columns: S_q at col_s(q), P_q (BF16 pairs) at kColP + q * kPStride, O_q at kColO + q * D
    static constexpr uint32_t col_s(int q) { return kSharedS ? 0u : static_cast<uint32_t>(q * kTN); }
    static constexpr uint32_t kColP = kSharedS ? kTN : 2 * kTN;
    static constexpr uint32_t kPStride = kTN / 2;
    static constexpr uint32_t kColO = 512 - 2 * D;
    static_assert(kColP + 2 * kPStride <= kColO, "Tensor Memory layout");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct PrefillParams {
    int U;          // units = B * Hkv
    int Hkv;
    int R;          // query rows per unit = (Hq / Hkv) * Sq
    int Skv;
    int pairs;      // ceil(R / 256)
    int Sq;         // query rows per head: row r of a unit is query r % Sq
    int group;      // causal item order: units per group
    int* sched;     // global work-item counter (zeroed before the launch), NULL = fixed order
    float c;        // scale * log2(e)
    const int32_t* seqlens;
    void* out;
    int out_f32;
    float* lse;
    float* o_stage;
    unsigned* amax_bits;
    const float* nv_sg;      // single-pass NVFP4: given s_g; codes/scales written here, else NULL
    uint8_t* nv_codes;
    uint8_t* nv_scales;
    float* nv_ts;
    int* status;
    long long limit;
};

__device__ __forceinline__ int unit_keys(const PrefillParams& p, int u)
{
    return p.seqlens ? p.seqlens[u / p.Hkv] : p.Skv;
}

// Unit and query-tile pair of work item r.  Without the mask: unit-major.  With it, later rows see
// more keys, so items go group by group (p.group units at a time) and within a group from the last
// pair of every unit down to the first: heaviest first, units of a group side by side.
template <bool CAUSAL>
__device__ __forceinline__ void item_coords(const PrefillParams& p, int r, int& u, int& pair)
{
    if (!CAUSAL) {
        u = r / p.pairs;
        pair = r - u * p.pairs;
        return;
    }
    const int per_group = p.group * p.pairs;
    const int g = r / per_group;
    const int rr = r - g * per_group;
    const int gsz = min(p.group, p.U - g * p.group);
    const int level = rr / gsz;
    u = g * p.group + (rr - level * gsz);
    pair = p.pairs - 1 - level;
}

// Fixed (counter-free) item order: round k of CTA c takes item k*G + c.  With the causal mask, whose
// items are numbered heaviest first, odd rounds take k*G + G-1-c instead, so a CTA that drew a heavy
// item in one round draws a light one in the next and the CTAs' totals even out.
template <bool CAUSAL>
__device__ __forceinline__ int fixed_item(int k)
{
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return k * G + ((CAUSAL && (k & 1)) ? G - 1 - c : c);
}

// Key tiles query tile q of a pair needs: none when its rows are all past R; with the causal
// mask only those up to the last key its rows can see (row r sees keys < r % Sq + n - Sq + 1).
template <bool CAUSAL, int kTN>
__device__ __forceinline__ int tile_count(const PrefillParams& p, int pair, int q, int n)
{
    const int a = pair * 2 * kTM + q * kTM;
    if (a >= p.R || n <= 0) return 0;
    const int T = (n + kTN - 1) / kTN;
    if (!CAUSAL) return T;
    const int b = min(a + kTM - 1, p.R - 1);
    const int sa = a % p.Sq, sb = b % p.Sq;
    const int max_s = (b - a + 1 >= p.Sq || sa > sb) ? p.Sq - 1 : sb;
    const int lim = max_s + n - p.Sq + 1;   // keys 0 .. lim - 1 visible to some row of the tile
    return lim <= 0 ? 0 : min(T, (lim + kTN - 1) / kTN);
}

__device__ __forceinline__ void drain_wait_p(uint64_t* bar, uint32_t parity, long long limit)
{
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

struct PRing {
    uint32_t idx = 0, phase = 0;
    int n;
    __device__ explicit PRing(int stages) : n(stages) {}
    __device__ void advance()
    {
        if (++idx == static_cast<uint32_t>(n)) {
            idx = 0;
            phase ^= 1;
        }
    }
};

// RING: 12 warps with the register split, work items handed out through the shared-memory ring
// (from the workspace counter when p.sched is set, else in the fixed order), and the single-pass
// NVFP4 epilogue.  !RING: 10 warps at 168 registers, fixed order, no NVFP4 encoder (dense problems).
template <int D, bool CAUSAL, bool RING>
__global__ void __launch_bounds__(prefill_threads<RING>(), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ PrefillParams p)
{
    using C = PrefillCfg<D>;
    constexpr int S = C::kStages;
    constexpr int kTN = C::kTN;
    constexpr int QS = C::kQStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ uint64_t q_full[QS], q_empty[QS], k_full[S], k_empty[S], v_full[S], v_empty[S];
    __shared__ uint64_t s_full[2], s_free[2], p_full[2], o_done[2], mma_done;
    __shared__ uint64_t item_full[kItemSlots], item_empty[kItemSlots];
    __shared__ int item_q[kItemSlots];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32;
    griddep_launch_dependents();
    const WaitCtl wc{&abort_flag, p.status, p.limit};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < QS; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128);
            mbar_init(&p_full[i], 128);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(&mma_done, 1);
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + 8);   // the MMA thread and one lane of each softmax warp
        }
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    griddep_wait();   // the previous kernel of the stream has completed: global memory from here on
    if (RING && blockIdx.x == 0 && threadIdx.x == 0 && p.nv_ts) *p.nv_ts = *p.nv_sg;   // single-pass NVFP4: report s_g
    const int n_items = p.U * p.pairs;

    // Each setmaxnreg dominates only its own role's code (the register budget of code after a join
    // would be the smaller one) and is executed by whole warpgroups.
    if (warp >= 8) {
        if constexpr (RING) setmaxnreg_dec<kRegsCtl>();
        if (warp == 8) {
            // ------------------------------------------------ TMA producer
            if (lane_id() == 0) {
                tma_prefetch_desc(&qmap);
                tma_prefetch_desc(&kmap);
                tma_prefetch_desc(&vmap);
                PRing qr(QS), kr(S), vr(S);
                uint32_t kcnt[S], vcnt[S], qcnt[QS];
                for (int i = 0; i < S; ++i) kcnt[i] = vcnt[i] = 0;
                for (int i = 0; i < QS; ++i) qcnt[i] = 0;
                PRing ir(kItemSlots);
                int round = 0;   // fixed order: this CTA's round
                int item = (RING && p.sched) ? atomicAdd(p.sched, 1) : fixed_item<CAUSAL>(0);
                for (;;) {
                    const bool more = item < n_items;
                    if constexpr (RING) {
                        // hand the item (or the end mark) to the MMA and softmax warps
                        if (!mbar_wait(&item_empty[ir.idx], ir.phase ^ 1, wc)) break;
                        item_q[ir.idx] = more ? item : -1;
                        mbar_arrive(&item_full[ir.idx]);
                        ir.advance();
                    }
                    if (!more) break;
                    int u, pair;
                    item_coords<CAUSAL>(p, item, u, pair);
                    const int r0 = pair * 2 * kTM;
                    const int n = unit_keys(p, u);
                    const int T = max(tile_count<CAUSAL, C::kTN>(p, pair, 0, n), tile_count<CAUSAL, C::kTN>(p, pair, 1, n));
                    // the next item is claimed once this one's loads are issued, so a CTA takes new
                    // work only shortly before it runs out
                    const int next = fixed_item<CAUSAL>(round + 1);
                    if (T == 0) {
                        item = (RING && p.sched) ? atomicAdd(p.sched, 1) : next;
                        ++round;
                        continue;
                    }
                    mbar_wait(&q_empty[qr.idx], qr.phase ^ 1, wc);
                    if (!aborted(wc)) {
                        uint8_t* dst = smem + C::kOffQ + qr.idx * C::kQBytes;
                        mbar_arrive_expect_tx(&q_full[qr.idx], C::kQBytes);
                        for (int q = 0; q < 2; ++q)
                            for (int a = 0; a < C::kAtoms; ++a)
                                tma_load_3d(dst + q * C::kQTileBytes + a * (kTM * 128), &qmap, &q_full[qr.idx], a * 64,
                                            r0 + q * kTM, u);
                        ++qcnt[qr.idx];
                    }
                    qr.advance();
                    for (int t = 0; t < T; ++t) {
                        mbar_wait(&k_empty[kr.idx], kr.phase ^ 1, wc);
                        if (!aborted(wc)) {
                            uint8_t* dst = smem + C::kOffK + kr.idx * C::kKVBytes;
                            mbar_arrive_expect_tx(&k_full[kr.idx], C::kKVBytes);
                            for (int a = 0; a < C::kAtoms; ++a)
                                tma_load_3d(dst + a * (kTN * 128), &kmap, &k_full[kr.idx], a * 64, t * kTN, u);
                            ++kcnt[kr.idx];
                        }
                        kr.advance();
                        mbar_wait(&v_empty[vr.idx], vr.phase ^ 1, wc);
                        if (!aborted(wc)) {
                            uint8_t* dst = smem + C::kOffV + vr.idx * C::kKVBytes;
                            mbar_arrive_expect_tx(&v_full[vr.idx], C::kKVBytes);
                            for (int a = 0; a < C::kAtoms; ++a)
                                tma_load_3d(dst + a * (kTN * 128), &vmap, &v_full[vr.idx], a * 64, t * kTN, u);
                            ++vcnt[vr.idx];
                        }
                        vr.advance();
                    }
                    item = (RING && p.sched) ? atomicAdd(p.sched, 1) : next;
                    ++round;
                }
                for (int i = 0; i < S; ++i) {
                    if (kcnt[i]) drain_wait_p(&k_full[i], (kcnt[i] - 1) & 1, kDrainLimit);
                    if (vcnt[i]) drain_wait_p(&v_full[i], (vcnt[i] - 1) & 1, kDrainLimit);
                }
                for (int i = 0; i < QS; ++i)
                    if (qcnt[i]) drain_wait_p(&q_full[i], (qcnt[i] - 1) & 1, kDrainLimit);
            }
        } else if (warp == 9) {
            // ------------------------------------------------ MMA issuer (polls, issues whatever is ready)
            if (lane_id() == 0) {
                constexpr uint32_t idesc_qk = idesc_bf16_f32(kTM, kTN, false, false);
                constexpr uint32_t idesc_pv = idesc_bf16_f32(kTM, D, false, true);
                PRing qr(QS);
                uint32_t gtile = 0;          // global K/V tile counter (ring position of tile 0 of an item)
                uint32_t nqk[2] = {0, 0};    // QKs issued per query tile over the kernel's life
                uint32_t nqk_all = 0;        // QKs issued over the kernel's life (shared S buffer)
                uint32_t npv[2] = {0, 0};    // PVs issued per query tile
                PRing ir(kItemSlots);
                int round = 0;
                for (;;) {
                    int item;
                    if constexpr (RING) {
                        if (!mbar_wait(&item_full[ir.idx], ir.phase, wc)) break;
                        item = item_q[ir.idx];
                        mbar_arrive(&item_empty[ir.idx]);
                        ir.advance();
                        if (item < 0) break;
                    } else {
                        item = fixed_item<CAUSAL>(round++);
                        if (item >= n_items) break;
                    }
                    int u, pair;
                    item_coords<CAUSAL>(p, item, u, pair);
                    const int n = unit_keys(p, u);
                    const int Tq[2] = {tile_count<CAUSAL, C::kTN>(p, pair, 0, n), tile_count<CAUSAL, C::kTN>(p, pair, 1, n)};
                    const int T = max(Tq[0], Tq[1]);
                    if (T == 0) continue;
                    mbar_wait(&q_full[qr.idx], qr.phase, wc);
                    tc_fence_after();
                    const uint32_t sQ = smem_u32(smem + C::kOffQ + qr.idx * C::kQBytes);
                    int jq[2] = {0, 0}, jp[2] = {0, 0};
                    long long t_idle = clock64();
                    int idle_polls = 0;
                    while ((jp[0] < Tq[0] || jp[1] < Tq[1]) && !aborted(wc)) {
                        bool did = false;
    #pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (jq[q] < Tq[q]) {
                                const uint32_t g = gtile + jq[q];
                                bool ok = mbar_test(&k_full[g % S], (g / S) & 1);
                                if constexpr (C::kSharedS) {
                                    // one S buffer: QKs in a fixed order (tile 0 then tile 1 at each key
                                    // tile, then whichever tile has key tiles left), each once the
                                    // softmax has read the previous QK's S
                                    const int nxt = (jq[0] < Tq[0] && (jq[0] <= jq[1] || jq[1] >= Tq[1])) ? 0 : 1;
                                    if (q != nxt) ok = false;
                                    if (ok && nqk_all > 0) ok = mbar_test(&s_free[0], (nqk_all - 1) & 1);
                                } else {
                                    if (ok && nqk[q] > 0) ok = mbar_test(&s_free[q], (nqk[q] - 1) & 1);
                                }
                                if (ok) {
                                    tc_fence_after();
                                    // descriptors once; K steps add constant offsets to the address fields
                                    const uint64_t dq = sdesc_sw128(sQ + q * C::kQTileBytes, 16, 1024);
                                    const uint64_t dk = sdesc_sw128(smem_u32(smem + C::kOffK + (g % S) * C::kKVBytes), 16, 1024);
                                    const uint32_t dS = tmem + C::col_s(q);
    #pragma unroll
                                    for (int kk = 0; kk < D / 16; ++kk)
                                        mma_ss(dS, dq + (((kk >> 2) * (kTM * 128) + (kk & 3) * 32) >> 4),
                                               dk + (((kk >> 2) * (kTN * 128) + (kk & 3) * 32) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
                                    mma_commit(&s_full[q]);
                                    ++nqk[q];
                                    ++nqk_all;
                                    ++jq[q];
                                    // the last of the query tiles that need K_g releases it
                                    if (Tq[q ^ 1] <= jq[q] - 1 || jq[q ^ 1] >= jq[q]) mma_commit(&k_empty[g % S]);
                                    did = true;
                                }
                            }
                            if (jp[q] < jq[q]) {
                                const uint32_t g = gtile + jp[q];
                                bool ok = mbar_test(&p_full[q], npv[q] & 1);
                                if (ok) ok = mbar_test(&v_full[g % S], (g / S) & 1);
                                if (ok) {
                                    tc_fence_after();
                                    const uint64_t dv = sdesc_sw128(smem_u32(smem + C::kOffV + (g % S) * C::kKVBytes), kTN * 128, 1024);
                                    const uint32_t dO = tmem + C::kColO + q * D;
                                    const uint32_t aP = tmem + C::kColP + q * C::kPStride;
    #pragma unroll
                                    for (int ks = 0; ks < kTN / 16; ++ks)
                                        mma_ts(dO, aP + ks * 8, dv + ((ks * 2048) >> 4), idesc_pv, (jp[q] > 0 || ks > 0) ? 1u : 0u);
                                    mma_commit(&o_done[q]);
                                    ++npv[q];
                                    ++jp[q];
                                    if (Tq[q ^ 1] <= jp[q] - 1 || jp[q ^ 1] >= jp[q]) mma_commit(&v_empty[g % S]);
                                    did = true;
                                }
                            }
                        }
                        if (did) {
                            t_idle = clock64();
                            idle_polls = 0;
                        } else if (++idle_polls > 4) {
                            __nanosleep(40);   // leave issue slots to the softmax warps on this SM quarter
                        }
                        if (!did && clock64() - t_idle > p.limit) {
                            abort_flag = 1;
                            atomicExch(p.status, kDevTimeout);
                        }
                    }
                    if (!aborted(wc)) mma_commit(&q_empty[qr.idx]);
                    qr.advance();
                    gtile += T;
                }
                mma_commit(&mma_done);
                drain_wait_p(&mma_done, 0, kDrainLimit);
            }
        }
    } else {
        if constexpr (RING) setmaxnreg_inc<kRegsSoftmax>();
        // ------------------------------------------------ softmax / rescale / epilogue, one row per thread
        const int q = warp / 4;
        const int wl = warp % 4;
        const uint32_t lane_base = static_cast<uint32_t>(wl * 32) << 16;
        const int row_in_tile = wl * 32 + static_cast<int>(lane_id());
        const uint32_t tS = tmem + lane_base + C::col_s(q);
        const uint32_t tP = tmem + lane_base + C::kColP + q * C::kPStride;
        const uint32_t tO = tmem + lane_base + C::kColO + q * D;
        const float nv_sg = (RING && p.nv_sg) ? *p.nv_sg : 0.f;
        uint32_t gt = 0;     // tiles processed by this warpgroup over the kernel's life (S/P/O rings)
        uint32_t gring = 0;  // K/V ring position of the current item's first tile
        PRing ir(kItemSlots);
        int round = 0;
        for (;;) {
            int item;
            if constexpr (RING) {
                // the whole warp leaves together (the TMEM accesses below are warp-collective)
                if (!__all_sync(0xffffffffu, mbar_wait(&item_full[ir.idx], ir.phase, wc))) break;
                item = item_q[ir.idx];
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(&item_empty[ir.idx]);
                ir.advance();
                if (item < 0) break;
            } else {
                item = fixed_item<CAUSAL>(round++);
                if (item >= n_items) break;
            }
            int u, pair;
            item_coords<CAUSAL>(p, item, u, pair);
            const int row = pair * 2 * kTM + q * kTM + row_in_tile;
            const int n = unit_keys(p, u);
            const int T = tile_count<CAUSAL, C::kTN>(p, pair, q, n);
            // keys this row sees: 0 .. lim - 1
            const int lim = CAUSAL ? min(n, (row < p.R ? row : 0) % p.Sq + n - p.Sq + 1) : n;
            float m_run = -INFINITY, l = 0.f;
            for (int j = 0; j < T; ++j, ++gt) {
                mbar_wait(&s_full[q], gt & 1, wc);
                tc_fence_after();
                float s[kTN];
                uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
                for (int c4 = 0; c4 < kTN / 32; ++c4) tmem_ld32p(tS + c4 * 32, su + c4 * 32);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&s_free[C::kSharedS ? 0 : q]);
                if ((j + 1) * kTN > lim) {
#pragma unroll
                    for (int i = 0; i < kTN; ++i)
                        if (j * kTN + i >= lim) s[i] = -INFINITY;
                }
                float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int i = 4; i < kTN; i += 8) {
                    mx[0] = fmax3(mx[0], s[i], s[i + 1]);
                    mx[1] = fmax3(mx[1], s[i + 2], s[i + 3]);
                    if (i + 4 < kTN) {
                        mx[2] = fmax3(mx[2], s[i + 4], s[i + 5]);
                        mx[3] = fmax3(mx[3], s[i + 6], s[i + 7]);
                    }
                }
                const float mt = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * p.c;
                const bool rescale = mt > m_run + kRescaleLog2;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ex2_approx(m_run - mt);
                    m_run = mt;
                }
                // p = 2^(s*c - m) with packed FP32x2 scale-subtract and sums.  With the shared S
                // buffer (D = 128) P goes to Tensor Memory 64 keys at a time as it is produced
                // (measured 1 % faster there; at D = 64 it measured 2 % slower than one store
                // after all the exponentials).
                constexpr bool kChunkP = C::kSharedS;
                const uint64_t cc = f32x2(p.c, p.c);
                // causal: a row with no visible key yet keeps m = -inf (no -inf - -inf = NaN)
                const float mu = (CAUSAL && m_run == -INFINITY) ? 0.f : -m_run;
                const uint64_t nm = f32x2(mu, mu);
                uint32_t pk[kTN / 2];
                uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < kTN / 64; ++c) {
#pragma unroll
                    for (int i = c * 64; i < c * 64 + 64; i += 2) {
                        float x0, x1;
                        f32x2_split(ffma2(f32x2(s[i], s[i + 1]), cc, nm), x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        ls[(i >> 1) & 3] = fadd2(ls[(i >> 1) & 3], f32x2(p0, p1));
                        pk[i >> 1] = pack_bf16x2(p0, p1);
                    }
                    if constexpr (kChunkP) {
                        if (c == 0) {
                            // PV of the previous tile must be done: its P buffer is reused
                            if (j > 0) mbar_wait(&o_done[q], (gt - 1) & 1, wc);
                            tc_fence_after();
                            __syncwarp();   // tcgen05.st is warp-collective
                        }
                        tmem_st32(tP + c * 32, pk + c * 32);
                    }
                }
                float la, lb;
                f32x2_split(fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3])), la, lb);
                l = fmaf(l, alpha, la + lb);
                if constexpr (!kChunkP) {
                    // PV of the previous tile must be done: its P buffer is reused and O must be stable.
                    if (j > 0) mbar_wait(&o_done[q], (gt - 1) & 1, wc);
                    tc_fence_after();
                }
                // tcgen05.ld/st are warp-collective (.sync.aligned): rescale if any lane of the warp
                // needs it (alpha = 1 for the others), never under a per-lane branch.
                if (__any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld32p(tO + c4 * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + c4 * 32, o);
                    }
                }
                // Keys at or beyond n of a ragged unit may be anything in memory (NaN in padding) and
                // P = 0 does not cancel NaN in the MMA: zero those V rows of a partial tile.  Both
                // warpgroups write the same zeros; each makes them visible before its own p_full.
                if (p.seqlens && (j + 1) * kTN > n) {
                    const uint32_t gr = gring + j;   // K/V ring position of this tile
                    mbar_wait(&v_full[gr % S], (gr / S) & 1, wc);
                    for (int r = n - j * kTN + row_in_tile; r < kTN; r += kTM) {
                        uint8_t* rowp = smem + C::kOffV + (gr % S) * C::kKVBytes + r * 128;
#pragma unroll
                        for (int a = 0; a < C::kAtoms; ++a)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                reinterpret_cast<uint4*>(rowp + a * (kTN * 128))[i] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if constexpr (!kChunkP) {
#pragma unroll
                    for (int c = 0; c < kTN / 64; ++c) tmem_st32(tP + c * 32, pk + c * 32);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[q]);
            }
            // ---- epilogue: O / l, LSE
            if (T > 0) {
                mbar_wait(&o_done[q], (gt - 1) & 1, wc);
                tc_fence_after();
            }
            // The TMEM loads below are warp-collective: every lane executes them; only the stores
            // are predicated on the row existing.
            gring += max(tile_count<CAUSAL, C::kTN>(p, pair, 0, n), tile_count<CAUSAL, C::kTN>(p, pair, 1, n));
            const bool store = row < p.R && !aborted(wc);
            const size_t orow = static_cast<size_t>(u) * p.R + (row < p.R ? row : 0);
            const bool none = !(l > 0.f);   // no visible key: O = 0, LSE = -inf
            const float inv_l = none ? 0.f : 1.f / l;
            float amax = 0.f;
            __syncwarp();
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t o[32];
                if (T > 0) {
                    tmem_ld32p(tO + c4 * 32, o);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv_l;
                if (store) {
                    if (p.o_stage) {
                        float4* dst = reinterpret_cast<float4*>(p.o_stage + orow * D + c4 * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                    if (p.amax_bits) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                    }
                    if constexpr (RING) {
                        if (p.nv_codes) {
                            // single-pass NVFP4: this thread holds the whole row, two 16-value blocks per chunk
#pragma unroll
                            for (int b = 0; b < 2; ++b) {
                                uint32_t lo, hi;
                                const uint32_t sc = nvfp4_encode16(v + 16 * b, nv_sg, lo, hi);
                                reinterpret_cast<uint2*>(p.nv_codes + orow * (D / 2) + c4 * 16)[b] = make_uint2(lo, hi);
                                p.nv_scales[orow * (D / 16) + c4 * 2 + b] = static_cast<uint8_t>(sc);
                            }
                        }
                    }
                    if (p.out) {
                        if (p.out_f32) {
                            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + c4 * 32);
#pragma unroll
                            for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * D + c4 * 32);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                                    pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                        }
                    }
                }
            }
            if (store && p.lse) p.lse[orow] = none ? -INFINITY : (m_run + __log2f(l)) * kLn2P;
            if (store && p.amax_bits && amax > 0.f) atomicMax(p.amax_bits, __float_as_uint(amax));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// ---- host side ------------------------------------------------------------------------------------
constexpr size_t kSchedBytes = 256;

// Work-item counter: causal or ragged problems (items of different sizes) when a workspace is in use.
bool prefill_dynamic(const AttnArgs& a, int sched_mode) { return sched_mode != 1 && (a.causal || a.seqlens); }

// The ring kernel: balanced (counter) order, single-pass NVFP4 output (its epilogue encoder needs
// the softmax warps' larger register budget; in the compact kernel it slowed dense problems), and
// every D = 128 problem (a row of 128 scores with P and O needs that budget too).
bool prefill_ring(const AttnArgs& a, int sched_mode) { return prefill_dynamic(a, sched_mode) || a.nv_sg || a.D == 128; }

size_t stage_bytes(const AttnArgs& a)
{
    // NVFP4 output without a caller-provided FP32 buffer: FP32 staging of O (last in the scratch)
    if (a.out_kind == FMHA_OUT_NVFP4 && !a.out_f32 && !a.nv_sg)
        return (static_cast<size_t>(a.B) * a.Hq * a.Sq * a.D * 4 + 255) & ~size_t(255);
    return 0;
}

template <int D, bool CAUSAL, bool RING>
int run_prefill(const AttnArgs& a, bool dynamic, void* ws, cudaStream_t st)
{
    using C = PrefillCfg<D>;
    const int nsm = num_sms();
    if (nsm <= 0) return set_error(FMHA_ERR_CUDA, "cannot query the SM count");
    const int U = a.B * a.Hkv;
    const int R = (a.Hq / a.Hkv) * a.Sq;
    CUtensorMap qmap, kmap, vmap;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(R), static_cast<uint64_t>(U)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(R) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(kTM), 1};
        int rc = make_tmap_bf16(&qmap, a.q, 3, dims, strides, box);
        if (rc) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Skv), static_cast<uint64_t>(U)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Skv) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(C::kTN), 1};
        int rc = make_tmap_bf16(&kmap, a.k, 3, dims, strides, box);
        if (rc) return rc;
        rc = make_tmap_bf16(&vmap, a.v, 3, dims, strides, box);
        if (rc) return rc;
    }
    PrefillParams p{};
    p.U = U;
    p.Hkv = a.Hkv;
    p.R = R;
    p.Skv = a.Skv;
    p.pairs = (R + 2 * kTM - 1) / (2 * kTM);
    p.Sq = a.Sq > 0 ? a.Sq : 1;
    // causal item groups: as many units as keep their K and V within 32 MiB of L2
    const size_t unit_kv = static_cast<size_t>(a.Skv) * D * 2 * 2;
    const size_t g = (size_t(32) << 20) / (unit_kv ? unit_kv : 1);
    p.group = static_cast<int>(g < 1 ? 1 : (g > static_cast<size_t>(U) ? U : g));
    p.sched = dynamic ? static_cast<int*>(ws) : nullptr;
    p.c = a.scale * kLog2eP;
    p.seqlens = a.seqlens;
    const bool nvfp4 = a.out_kind == FMHA_OUT_NVFP4;
    p.out = nvfp4 ? nullptr : a.out;
    p.out_f32 = a.out_kind == FMHA_OUT_F32 ? 1 : 0;
    p.lse = a.lse;
    float* stage = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + (dynamic ? kSchedBytes : 0));
    p.o_stage = nvfp4 ? (a.out_f32 ? a.out_f32 : (a.nv_sg ? nullptr : stage)) : nullptr;
    p.amax_bits = nvfp4 ? reinterpret_cast<unsigned*>(a.amax_slot) : nullptr;
    p.nv_sg = a.nv_sg;
    p.nv_codes = a.nv_codes;
    p.nv_scales = a.nv_scales;
    p.nv_ts = a.nv_ts;
    p.status = device_status_ptr();
    p.limit = wait_limit();
    const long long items = static_cast<long long>(U) * p.pairs;
    const int grid = static_cast<int>(items < nsm ? items : nsm);
    FMHA_CHECK_CUDA(set_smem_limit_once(reinterpret_cast<const void*>(prefill_kernel<D, CAUSAL, RING>), C::kSmemBytes));
    if (grid > 0) {
        if (dynamic) FMHA_CHECK_CUDA(cudaMemsetAsync(p.sched, 0, sizeof(int), st));
        timing_mark_begin(st);
        const cudaError_t e = launch_pdl(prefill_kernel<D, CAUSAL, RING>, dim3(static_cast<unsigned>(grid)),
                                         dim3(prefill_threads<RING>()), C::kSmemBytes, st, qmap, kmap, vmap, p);
        timing_mark_end(st);
        FMHA_CHECK_CUDA(e);
        count_launch();
    }
    return FMHA_OK;
}

template <int D>
int run_prefill_d(const AttnArgs& a, int sched_mode, void* ws, cudaStream_t st)
{
    const bool dyn = prefill_dynamic(a, sched_mode);
    if constexpr (PrefillCfg<D>::kSharedS) {   // always the ring kernel (prefill_ring)
        return a.causal ? run_prefill<D, true, true>(a, dyn, ws, st) : run_prefill<D, false, true>(a, dyn, ws, st);
    } else {
        const bool ring = prefill_ring(a, sched_mode);
        if (a.causal) return ring ? run_prefill<D, true, true>(a, dyn, ws, st) : run_prefill<D, true, false>(a, dyn, ws, st);
        return ring ? run_prefill<D, false, true>(a, dyn, ws, st) : run_prefill<D, false, false>(a, dyn, ws, st);
    }
}

}  // namespace

size_t prefill_workspace_bytes(const AttnArgs& a, int sched_mode)
{
    return (prefill_dynamic(a, sched_mode) ? kSchedBytes : 0) + stage_bytes(a);
}

int launch_prefill(const AttnArgs& a, int sched_mode, void* ws, size_t ws_bytes, cudaStream_t st)
{
    if (ws_bytes < prefill_workspace_bytes(a, sched_mode)) return set_error(FMHA_ERR_WORKSPACE, "row-tile path: workspace too small");
    switch (a.D) {
        case 64: return run_prefill_d<64>(a, sched_mode, ws, st);
        case 128: return run_prefill_d<128>(a, sched_mode, ws, st);
        default: return set_error(FMHA_ERR_UNSUPPORTED, "row-tile path: D must be 64 or 128");
    }
}

}  // namespace atc_gb300
