// Decode attention (few query rows per key/value head): split-KV over a persistent grid, plus
// the combine of the partial results.
//
// Follows the kernel plan of "NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md" (nvfp4-megamoe-kernel): TMA
// loads of Q/K/V, the QK product on tcgen05 with the accumulator in Tensor Memory, softmax warps
// reading S back with tcgen05.ld, the running max / sum with O rescale over several KV tiles
// ("in-kernel softmax with O rescale", "multi-KV-tile support"), then the PV product.  The
// GB300 design around it is this file's own:
//
//  * Swap-AB.  With G <= 16 query rows per key/value head (G = (Hq/Hkv) * Sq), the products are
//    taken transposed so that the 128 keys of a tile fill the MMA's M dimension:
//      S^T[kv][q] = K[kv][:] . Q[q][:]      (A = K tile, K-major; B = Q rows, K-major; N = 16)
//      O^T[d][q]  = V^T[d][kv] . P^T[kv][q]  (A = V tile read MN-major; B = P, K-major; N = 16)
//    Thread t of the softmax warpgroup owns TMEM lane t: key t of the tile for S, feature d = t
//    for O.  Reductions over keys are warp shuffles plus a 4-warp shared-memory step.
//  * The per-tile PV product goes to a fresh TMEM buffer (no accumulate) and the softmax threads
//    fold it into register accumulators with the rescale factor: acc = alpha * acc + O_tile.
//    O is never read-modify-written in TMEM, so there is no ordering hazard between the rescale
//    and the next MMA.
//  * Work split ("stream-K" over keys): the key tiles of all units (b, kv-head) are laid end to
//    end and CTA c of P takes tiles [c*T/P, (c+1)*T/P).  Each maximal run inside one unit is a
//    work item; an item that covers a whole unit writes the final O and LSE, otherwise it writes
//    a normalised partial (O_i, lse_i) to slot u + c of the workspace and the combine kernel
//    merges them: lse = log sum_i exp(lse_i), O = sum_i exp(lse_i - lse) O_i.  Ragged batches
//    balance by construction.  With num_splits == 1 each CTA takes whole units instead.
//  * Roles (decode_kernel<D, CAUSAL, EPI>): warps 0-3 softmax.  EPI (units of several query
//    columns): warps 4-7 epilogue, warp 8 TMA producer, warp 9 MMA issuer, warps 10-11 only complete
//    their warpgroup; at the end of a work item the softmax warps hand its accumulators to the
//    epilogue warps (Tensor Memory, two buffers) and go on with the next item while the epilogue
//    normalises, stores and merges.  !EPI (one column): warp 4 producer, warp 5 MMA, and the softmax
//    warps run each item's short epilogue themselves.  Every wait is bounded; a timeout flips the
//    CTA into a drain mode (no new TMA/MMA, loops run out) and sets the device status word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>

#include "internal.h"
#include "nvfp4_dev.cuh"
#include "ptx.cuh"

namespace atc_gb300 {
namespace {

constexpr int kTileKV = 128;    // keys per tile = MMA M
constexpr int kN = 16;          // query rows per unit, padded (MMA N)
// EPI: softmax, epilogue and control warpgroups (warps 0-3, 4-7, 8-11: producer 8, MMA 9); else the
// softmax warps run each item's epilogue themselves and warps 4 and 5 are the producer and the MMA.
template <bool EPI>
constexpr int decode_threads() { return EPI ? 384 : 192; }
template <bool EPI>
constexpr int tma_warp() { return EPI ? 8 : 4; }
template <bool EPI>
constexpr int mma_warp() { return EPI ? 9 : 5; }
// setmaxnreg split of the launch's 168 registers a thread: on each SM quarter one warp of each
// warpgroup, 232 + 184 + 88 = 504 of its 512, and 128 * 504 = 384 * 168 in all
constexpr uint32_t kRegsSm = 232, kRegsEpi = 184, kRegsCtl = 88;
static_assert(128 * (kRegsSm + kRegsEpi + kRegsCtl) <= decode_threads<true>() * 168, "register split exceeds the launch allocation");
static_assert(kRegsSm + kRegsEpi + kRegsCtl <= 512, "register split exceeds an SM quarter");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleD = 8.0f;   // log2 units: a column's reference max moves only when exceeded by more

template <int D>
struct DecodeCfg {
    static constexpr int kAtoms = D / 64;                  // 64-column swizzle atoms per row
    static constexpr int kStages = (D == 64) ? 4 : 3;      // K and V ring depth
    static constexpr int kQBytes = kAtoms * kN * 128;      // one Q buffer
    static constexpr int kKVBytes = kAtoms * kTileKV * 128;
    static constexpr int kPBytes = 2 * kN * 128;           // P^T: 16 rows x 128 keys
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kSmemBytes = kOffP + 2 * kPBytes + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = 128;             // S[2] x 16, O[2] x 16, handoff[2] x 32
};

struct DecodeParams {
    int U;              // units = B * Hkv
    int Hkv;
    int G;              // real query rows per unit
    int Skv;
    int D;
    int Sq;             // query rows per head (column q of a unit is query q % Sq)
    float c;            // scale * log2(e)
    const int32_t* seqlens;
    const int32_t* prefix;   // [U+1] tile prefix (ragged split mode), else NULL
    int tiles_uniform;       // tiles per unit when prefix == NULL
    int split;               // 1 = stream-K partition, 0 = whole units per CTA
    // outputs
    void* out;               // BF16 or F32 [U*G][D] (NULL when writing FP32 staging only)
    int out_f32;             // 1: `out` is FP32
    float* lse;              // [U*G] or NULL
    float* o_stage;          // FP32 [U*G][D] copy for NVFP4, else NULL
    unsigned* amax_bits;     // NVFP4: running max |O| (FP32 bits), else NULL
    const float* nv_sg;      // single-pass NVFP4: given s_g; codes/scales written here, else NULL
    uint8_t* nv_codes;
    uint8_t* nv_scales;
    float* nv_ts;
    float* part_o;           // [slots][16][D]
    float* part_lse;         // [slots][16]
    int fixup;               // split mode: the CTA completing a unit merges its partials (no combine kernel)
    unsigned long long gen;  // this call's tag for the arrival counters (48 bits)
    unsigned long long* unit_ctr;   // [U] arrival counters: (gen << 16) | arrivals
    int* status;
    long long limit;
};

// ---- work items ----------------------------------------------------------------------------------
struct Item {
    int u, t0, t1;   // unit and its tile range [t0, t1)
    int n;           // valid keys of the unit
    bool whole;      // covers every tile of the unit
    int slot;        // partial slot (u + cta)
};

struct Sched {
    const DecodeParams* p;
    long long g, g1;    // split mode: current / end global tile
    int u;              // whole-unit mode: next unit
    int cta, nctas;

    __device__ int unit_tiles(int u) const
    {
        if (p->prefix) return p->prefix[u + 1] - p->prefix[u];
        if (p->seqlens) return (p->seqlens[u / p->Hkv] + kTileKV - 1) / kTileKV;
        return p->tiles_uniform;
    }
    __device__ long long unit_start(int u) const
    {
        return p->prefix ? static_cast<long long>(p->prefix[u]) : static_cast<long long>(u) * p->tiles_uniform;
    }
    __device__ int unit_keys(int u) const { return p->seqlens ? p->seqlens[u / p->Hkv] : p->Skv; }

    __device__ void init(const DecodeParams* pp, int c, int n)
    {
        p = pp;
        cta = c;
        nctas = n;
        if (p->split) {
            const long long T = p->prefix ? p->prefix[p->U] : static_cast<long long>(p->U) * p->tiles_uniform;
            g = (static_cast<long long>(c) * T) / n;
            g1 = (static_cast<long long>(c + 1) * T) / n;
        } else {
            u = c;
        }
    }

    __device__ bool next(Item& it)
    {
        if (p->split) {
            if (g >= g1) return false;
            int uu;
            if (p->prefix) {   // last unit whose start <= g (prefix is non-decreasing)
                int lo = 0, hi = p->U - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (p->prefix[mid] <= g) lo = mid; else hi = mid - 1;
                }
                uu = lo;
                while (uu + 1 < p->U && p->prefix[uu + 1] <= g) ++uu;   // skip empty units
            } else {
                uu = static_cast<int>(g / p->tiles_uniform);
            }
            const long long s = unit_start(uu);
            const int nt = unit_tiles(uu);
            it.u = uu;
            it.t0 = static_cast<int>(g - s);
            it.t1 = static_cast<int>(min(static_cast<long long>(nt), g1 - s));
            it.n = unit_keys(uu);
            it.whole = (it.t0 == 0 && it.t1 == nt);
            it.slot = uu + cta;
            g = s + it.t1;
            return true;
        }
        if (u >= p->U) return false;
        it.u = u;
        it.t0 = 0;
        it.t1 = unit_tiles(u);
        it.n = unit_keys(u);
        it.whole = true;
        it.slot = 0;
        u += nctas;
        return true;
    }
};

// Byte offset of element (row r, column k) of a K-major operand made of 128-byte-swizzled
// atoms of 64 columns, `atom_bytes` apart.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k, uint32_t atom_bytes)
{
    const int a = k >> 6, kk = k & 63;
    return a * atom_bytes + r * 128 + ((((kk >> 3) ^ (r & 7)) & 7) << 4) + ((kk & 7) << 1);
}


// Bounded wait that ignores the abort flag: used at teardown so nothing is still in flight.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, long long limit)
{
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

struct Ring {
    uint32_t idx = 0, phase = 0;
    int n;
    __device__ explicit Ring(int stages) : n(stages) {}
    __device__ void advance()
    {
        if (++idx == static_cast<uint32_t>(n)) {
            idx = 0;
            phase ^= 1;
        }
    }
};

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Stream-K: the CTAs holding partials of unit u are c0..c1 of P, skipping CTAs whose tile range is
// empty (possible when there are fewer tiles than CTAs).  Fills slots[] (partial slots u + c, at
// most cap) and returns how many there are; 0 for a unit without tiles.
__device__ int unit_partial_slots(const DecodeParams& p, int u, int P, int* slots, int cap)
{
    int tiles;
    long long Tu, T;
    if (p.prefix) {
        tiles = p.prefix[u + 1] - p.prefix[u];
        Tu = p.prefix[u];
        T = p.prefix[p.U];
    } else {
        tiles = p.tiles_uniform;
        Tu = static_cast<long long>(u) * tiles;
        T = static_cast<long long>(p.U) * tiles;
    }
    if (tiles <= 0) return 0;
    const int c0 = static_cast<int>(min((((Tu + 1) * P) - 1) / T, static_cast<long long>(P - 1)));
    const int c1 = static_cast<int>(min((((Tu + tiles) * P) - 1) / T, static_cast<long long>(P - 1)));
    int n = 0;
    for (int c = c0; c <= c1 && n < cap; ++c)
        if ((static_cast<long long>(c) * T) / P != (static_cast<long long>(c + 1) * T) / P) slots[n++] = u + c;
    return n;
}

constexpr int kMaxFixSlots = 512;

template <int D, bool CAUSAL, bool EPI>
__global__ void __launch_bounds__(decode_threads<EPI>(), 1)
    decode_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeParams p)
{
    using C = DecodeCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ uint64_t q_full[2], q_empty[2], k_full[S], k_empty[S], v_full[S], v_empty[S];
    __shared__ uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2], mma_done;
    __shared__ uint64_t ep_full[2], ep_empty[2];   // softmax -> epilogue handoff
    __shared__ float ep_m[2][kN];                  // the columns' reference maxima
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float red_max[2][4][kN];
    __shared__ uint32_t red_need[2][4];   // per warp: columns whose scores passed the reference + kRescaleD
    __shared__ float red_sum[4][kN];
    __shared__ float col_inv[kN], col_lse[kN];   // per query column: 1 / L and the LSE of this range
    __shared__ int ep_abort, fx_last;          // softmax warps: abort snapshot, "this CTA merges"
    __shared__ int fx_n;
    __shared__ int fx_slot[kMaxFixSlots];
    __shared__ float fx_w[kN][4], fx_lse[kN];   // merge: per column, the partials' weights and the merged LSE

    const int warp = threadIdx.x / 32;
    griddep_launch_dependents();
    const WaitCtl wc{&abort_flag, p.status, p.limit};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 128);
            mbar_init(&p_full[i], 128);
            mbar_init(&p_empty[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 128);
            mbar_init(&ep_full[i], 128);
            mbar_init(&ep_empty[i], 128);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(&mma_done, 1);
        fence_barrier_init();
    }
    if (warp == mma_warp<EPI>()) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;   // S buffers at columns 0/16, O buffers at 32/48, handoff at 64/96
    griddep_wait();   // the previous kernel of the stream has completed: global memory from here on
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.nv_ts) *p.nv_ts = *p.nv_sg;   // single-pass NVFP4: report s_g

    Sched sched;
    sched.init(&p, blockIdx.x, gridDim.x);
    Item it;

    // The epilogue of one item, run by 128 threads: the epilogue warpgroup (named barrier 2) when a
    // unit has several query columns, else the softmax warps themselves (barrier 1), for which the
    // epilogue is short and an extra warpgroup's handoff measured slower.  tid: O^T row (Tensor
    // Memory lane) and output column, ew: warp within the group.
    // slots_ready: fx_n / fx_slot already hold this item's partial slots (the epilogue warpgroup finds
    // them while it waits for the item)
    auto run_epilogue = [&](const Item& it, bool empty, const float (&m)[kN], const float (&l)[kN],
                            const float (&acc)[kN], int tid, int ew, int bar, bool slots_ready) {
        const int lane = static_cast<int>(lane_id());
        const int G = p.G;
        const float nv_sg = p.nv_sg ? *p.nv_sg : 0.f;
        // final output of one row at column tid (tid < D); the |O| max goes to amax_acc
        auto write_final = [&](size_t row, float o, float lse_v, float& amax_acc) {
            if (p.o_stage) p.o_stage[row * D + tid] = o;
            if (p.amax_bits) amax_acc = fmaxf(amax_acc, fabsf(o));
            if (p.out) {
                if (p.out_f32)
                    static_cast<float*>(p.out)[row * D + tid] = o;
                else
                    static_cast<uint16_t*>(p.out)[row * D + tid] = float_to_bf16_bits(o);
            }
            if (tid == 0 && p.lse) p.lse[row] = lse_v;
        };
        // ---- epilogue: L = sum over the 128 key lanes, O = acc · (1 / L), lse = ln2 * (m + log2 L)
        if (!empty) {
            if (G == 1) {
                const float s = warp_sum(l[0]);
                if (lane == 0) red_sum[ew][0] = s;
            } else {
                // all columns' butterflies interleaved: five rounds of independent shuffles
                float v[kN];
#pragma unroll
                for (int q = 0; q < kN; ++q) v[q] = q < G ? l[q] : 0.f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int q = 0; q < kN; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                if (lane == 0)
#pragma unroll
                    for (int q = 0; q < kN; ++q)
                        if (q < G) red_sum[ew][q] = v[q];
            }
        }
        // red_sum is complete, and every thread is past its reads of the previous item's
        // col_inv / col_lse (an empty item has no tile barriers in between)
        named_bar_sync(bar, 128);
        // one thread per column: L, then 1 / L and the LSE for every thread of the CTA
        if (tid < G) {
            const float Lq = empty ? 0.f : (red_sum[0][tid] + red_sum[1][tid]) + (red_sum[2][tid] + red_sum[3][tid]);
            float mq = m[0];
#pragma unroll
            for (int q = 1; q < kN; ++q)
                if (q == tid) mq = m[q];
            const bool none = !(Lq > 0.f);   // no visible key in this range
            col_inv[tid] = none ? 0.f : 1.f / Lq;
            col_lse[tid] = none ? -INFINITY : (mq + __log2f(Lq)) * kLn2;
        }
        // one abort decision for all four warps (named barriers and shuffles below)
        if (tid == 0) ep_abort = aborted(wc) ? 1 : 0;
        named_bar_sync(bar, 128);
        if (ep_abort) return;
        // single-pass NVFP4 in split mode: whole units also go through the combine, which
        // encodes every row in parallel (encoding here would lengthen the CTAs holding many
        // short units)
        const bool final_here = it.whole && !(p.split && p.nv_codes);
        float local_amax = 0.f;
        if (tid < D) {
#pragma unroll
            for (int q = 0; q < kN; ++q) {
                if (q >= G) break;
                const float o = col_inv[q] > 0.f ? acc[q] * col_inv[q] : 0.f;   // 0: no visible key in this range
                const float lse_v = col_lse[q];
                const size_t row = static_cast<size_t>(it.u) * G + q;
                if (final_here) {
                    write_final(row, o, lse_v, local_amax);
                    // single-pass NVFP4: a warp holds 32 consecutive columns of the row
                    if (p.nv_codes) nvfp4_encode_lanes(o, nv_sg, tid, p.nv_codes + row * (D / 2), p.nv_scales + row * (D / 16));
                } else {
                    p.part_o[(static_cast<size_t>(it.slot) * kN + q) * D + tid] = o;
                    if (tid == 0) p.part_lse[static_cast<size_t>(it.slot) * kN + q] = lse_v;
                }
            }
        }
        if (p.amax_bits && final_here) {
            const float wm = warp_max(local_amax);
            if (lane == 0 && wm > 0.f) atomicMax(p.amax_bits, __float_as_uint(wm));
        }
        if (p.fixup && !final_here) {
            // stream-K fixup: publish this partial, count the unit's arrivals, and let the CTA
            // that completes the unit merge it (O = sum exp(lse_i - lse) O_i, as the combine).
            // The CTA barrier orders every thread's partial stores before thread 0's device-scope
            // fence, which releases them all (release is cumulative) ahead of its arrival: one
            // fence waits for the stores instead of 128.
            named_bar_sync(bar, 128);
            if (tid == 0) {
                const int n = slots_ready ? fx_n : unit_partial_slots(p, it.u, static_cast<int>(gridDim.x), fx_slot, kMaxFixSlots);
                fx_n = n;
                __threadfence();
                const int arrived = n > 0 ? arrive_unit(p.unit_ctr + it.u, p.gen, n) : 0;
                // -1: the counter kept changing under us (another call on this workspace):
                // the unit may stay unmerged, so say so instead of failing silently
                if (arrived < 0) atomicExch(p.status, kDevMergeLost);
                fx_last = (arrived == n && n > 0) ? 1 : 0;
                // every arrival of this call is in: clear the counter for the next call.  A CUDA graph
                // replays a call with the same tag, so its arrivals must not be left over (0 carries
                // no call's tag: tags are never 0).
                if (fx_last) atomicExch(p.unit_ctr + it.u, 0ull);
            }
            named_bar_sync(bar, 128);
            if (fx_last) {
                __threadfence();
                const int ns = fx_n;
                float amax_m = 0.f;
                if (ns <= 4) {
                    // the usual case: this thread's element of every partial O of every column, and
                    // (threads q < G) column q's partial LSEs, all in flight at once, so the merge
                    // costs one L2 round trip whatever the number of columns (a round per few
                    // columns was one dependent trip each, slow while the other CTAs stream)
                    float ov[kN][4];
#pragma unroll
                    for (int q = 0; q < kN; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const bool use = q < G && i < ns && tid < D;
                            ov[q][i] = use ? __ldcg(p.part_o + (static_cast<size_t>(fx_slot[i < ns ? i : 0]) * kN + q) * D + tid) : 0.f;
                        }
                    if (tid < G) {
                        float lv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            lv[i] = i < ns ? __ldcg(p.part_lse + static_cast<size_t>(fx_slot[i]) * kN + tid) : -INFINITY;
                        const float mx = fmaxf(fmaxf(lv[0], lv[1]), fmaxf(lv[2], lv[3]));
                        const bool any = mx > -INFINITY;   // partials without a visible key carry -inf
                        float sum = 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) sum += (any && i < ns) ? __expf(lv[i] - mx) : 0.f;
                        const float lse_all = any ? mx + __logf(sum) : -INFINITY;
#pragma unroll
                        for (int i = 0; i < 4; ++i) fx_w[tid][i] = (any && i < ns) ? __expf(lv[i] - lse_all) : 0.f;
                        fx_lse[tid] = lse_all;
                    }
                    named_bar_sync(bar, 128);
#pragma unroll
                    for (int q = 0; q < kN; ++q) {
                        if (q >= G) break;
                        float o = 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) o = fmaf(fx_w[q][i], ov[q][i], o);
                        if (tid < D) write_final(static_cast<size_t>(it.u) * G + q, o, fx_lse[q], amax_m);
                    }
                } else {
                    for (int q = 0; q < G; ++q) {
                        float mx = -INFINITY;
                        for (int i = 0; i < ns; ++i) mx = fmaxf(mx, __ldcg(p.part_lse + static_cast<size_t>(fx_slot[i]) * kN + q));
                        // partials without a visible key carry lse = -inf and weigh 0; all of them -> empty row
                        const bool any = mx > -INFINITY;
                        float sum = 0.f;
                        if (any)
                            for (int i = 0; i < ns; ++i) sum += __expf(__ldcg(p.part_lse + static_cast<size_t>(fx_slot[i]) * kN + q) - mx);
                        const float lse_all = (ns > 0 && any) ? mx + __logf(sum) : -INFINITY;
                        if (tid < D) {
                            float o = 0.f;
                            if (any)
                                for (int i = 0; i < ns; ++i) {
                                    const size_t sl = static_cast<size_t>(fx_slot[i]) * kN + q;
                                    o = fmaf(__expf(__ldcg(p.part_lse + sl) - lse_all), __ldcg(p.part_o + sl * D + tid), o);
                                }
                            write_final(static_cast<size_t>(it.u) * G + q, o, lse_all, amax_m);
                        }
                    }
                }
                if (p.amax_bits) {
                    const float wm = warp_max(amax_m);
                    if (lane == 0 && wm > 0.f) atomicMax(p.amax_bits, __float_as_uint(wm));
                }
                named_bar_sync(bar, 128);   // every read of fx_slot is done before thread 0 refills it
            }
        }
    };

    // Each setmaxnreg dominates only its own role's code and is executed by whole warpgroups.
    if (warp >= tma_warp<EPI>()) {
        if constexpr (EPI) setmaxnreg_dec<kRegsCtl>();
      if (warp == tma_warp<EPI>()) {
        // ------------------------------------------------ TMA producer
        if (lane_id() == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            const uint64_t pol = policy_evict_first();
            Ring qr(2), kr(S), vr(S);
            uint32_t kcnt[S], vcnt[S], qcnt[2] = {0, 0};
            for (int i = 0; i < S; ++i) kcnt[i] = vcnt[i] = 0;
            while (sched.next(it)) {
                if (it.t1 <= it.t0) continue;
                mbar_wait(&q_empty[qr.idx], qr.phase ^ 1, wc);
                if (!aborted(wc)) {
                    uint8_t* dst = smem + C::kOffQ + qr.idx * C::kQBytes;
                    mbar_arrive_expect_tx(&q_full[qr.idx], C::kQBytes);
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d(dst + a * (kN * 128), &qmap, &q_full[qr.idx], a * 64, 0, it.u);
                    ++qcnt[qr.idx];
                }
                qr.advance();
                for (int t = it.t0; t < it.t1; ++t) {
                    mbar_wait(&k_empty[kr.idx], kr.phase ^ 1, wc);
                    if (!aborted(wc)) {
                        uint8_t* dst = smem + C::kOffK + kr.idx * C::kKVBytes;
                        mbar_arrive_expect_tx(&k_full[kr.idx], C::kKVBytes);
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_load_3d_hint(dst + a * (kTileKV * 128), &kmap, &k_full[kr.idx], a * 64, t * kTileKV,
                                             it.u, pol);
                        ++kcnt[kr.idx];
                    }
                    kr.advance();
                    mbar_wait(&v_empty[vr.idx], vr.phase ^ 1, wc);
                    if (!aborted(wc)) {
                        uint8_t* dst = smem + C::kOffV + vr.idx * C::kKVBytes;
                        mbar_arrive_expect_tx(&v_full[vr.idx], C::kKVBytes);
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_load_3d_hint(dst + a * (kTileKV * 128), &vmap, &v_full[vr.idx], a * 64, t * kTileKV,
                                             it.u, pol);
                        ++vcnt[vr.idx];
                    }
                    vr.advance();
                }
            }
            // nothing may still be landing in shared memory when the CTA exits
            for (int i = 0; i < S; ++i) {
                if (kcnt[i]) drain_wait(&k_full[i], (kcnt[i] - 1) & 1, kDrainLimit);
                if (vcnt[i]) drain_wait(&v_full[i], (vcnt[i] - 1) & 1, kDrainLimit);
            }
            for (int i = 0; i < 2; ++i)
                if (qcnt[i]) drain_wait(&q_full[i], (qcnt[i] - 1) & 1, kDrainLimit);
        }
      } else if (warp == mma_warp<EPI>()) {
        // ------------------------------------------------ MMA issuer
        if (lane_id() == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kN, true, false);
            constexpr uint32_t lbo_v = (D >= 128) ? 16384u : 0u;   // D = 64: M rows 64..127 repeat 0..63
            Ring qr(2), kr(S), vr(S), sr(2), pr(2), orr(2);
            auto pv = [&]() {
                mbar_wait(&p_full[pr.idx], pr.phase, wc);
                mbar_wait(&v_full[vr.idx], vr.phase, wc);
                mbar_wait(&o_empty[orr.idx], orr.phase ^ 1, wc);
                tc_fence_after();
                if (!aborted(wc)) {
                    const uint32_t sV = smem_u32(smem + C::kOffV + vr.idx * C::kKVBytes);
                    const uint32_t sP = smem_u32(smem + C::kOffP + pr.idx * C::kPBytes);
                    const uint32_t dO = tmem + 32 + orr.idx * 16;
#pragma unroll
                    for (int ks = 0; ks < kTileKV / 16; ++ks) {
                        const uint64_t da = sdesc_sw128(sV + ks * 2048, lbo_v, 1024);
                        const uint64_t db = sdesc_sw128(sP + (ks >> 2) * (kN * 128) + (ks & 3) * 32, 16, 1024);
                        mma_ss(dO, da, db, idesc_pv, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&o_full[orr.idx]);
                    mma_commit(&v_empty[vr.idx]);
                    mma_commit(&p_empty[pr.idx]);
                }
                pr.advance();
                vr.advance();
                orr.advance();
            };
            while (sched.next(it)) {
                if (it.t1 <= it.t0) continue;
                mbar_wait(&q_full[qr.idx], qr.phase, wc);
                const uint32_t sQ = smem_u32(smem + C::kOffQ + qr.idx * C::kQBytes);
                for (int t = it.t0; t < it.t1; ++t) {
                    mbar_wait(&k_full[kr.idx], kr.phase, wc);
                    mbar_wait(&s_empty[sr.idx], sr.phase ^ 1, wc);
                    tc_fence_after();
                    if (!aborted(wc)) {
                        const uint32_t sK = smem_u32(smem + C::kOffK + kr.idx * C::kKVBytes);
                        const uint32_t dS = tmem + sr.idx * 16;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t da = sdesc_sw128(sK + (kk >> 2) * (kTileKV * 128) + (kk & 3) * 32, 16, 1024);
                            const uint64_t db = sdesc_sw128(sQ + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
                            mma_ss(dS, da, db, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&s_full[sr.idx]);
                        mma_commit(&k_empty[kr.idx]);
                    }
                    kr.advance();
                    sr.advance();
                    if (t > it.t0) pv();   // PV of the previous tile overlaps this tile's softmax
                }
                pv();
                if (!aborted(wc)) mma_commit(&q_empty[qr.idx]);
                qr.advance();
            }
            mma_commit(&mma_done);
            drain_wait(&mma_done, 0, kDrainLimit);
        }
      }
    } else if (warp < 4) {
        if constexpr (EPI) setmaxnreg_inc<kRegsSm>();
        // ------------------------------------------------ softmax / correction (128 threads)
        const int tid = threadIdx.x;
        const int lane = static_cast<int>(lane_id());
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const int G = p.G;
        Ring sr(2), pr(2), orr(2), vr(S), hr(2);
        uint32_t tile_ctr = 0;
        while (sched.next(it)) {
            float m[kN], l[kN], acc[kN], alpha_prev[kN];
            // keys visible to column q: 0 .. lim[q] - 1 (causal: query q % Sq sees keys up to
            // (q % Sq) + n - Sq; otherwise all n)
            int lim[kN];
#pragma unroll
            for (int q = 0; q < kN; ++q) lim[q] = CAUSAL ? it.n - p.Sq + 1 + (q % p.Sq) : it.n;
#pragma unroll
            for (int q = 0; q < kN; ++q) {
                m[q] = -INFINITY;
                l[q] = 0.f;
                acc[q] = 0.f;
                alpha_prev[q] = 0.f;
            }
            auto consume = [&](const float (&al)[kN]) {
                mbar_wait(&o_full[orr.idx], orr.phase, wc);
                tc_fence_after();
                uint32_t ov[16];
                tmem_ld16(tmem + lane_base + 32 + orr.idx * 16, ov);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&o_empty[orr.idx]);
                orr.advance();
#pragma unroll
                for (int q = 0; q < kN; ++q) acc[q] = fmaf(acc[q], al[q], __uint_as_float(ov[q]));
            };
            for (int t = it.t0; t < it.t1; ++t) {
                mbar_wait(&s_full[sr.idx], sr.phase, wc);
                tc_fence_after();
                uint32_t sv[16];
                tmem_ld16(tmem + lane_base + sr.idx * 16, sv);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&s_empty[sr.idx]);
                sr.advance();

                const int kv = t * kTileKV + tid;
                const bool valid = kv < it.n;
                float x[kN];
#pragma unroll
                for (int q = 0; q < kN; ++q) x[q] = (CAUSAL ? kv < lim[q] : valid) ? __uint_as_float(sv[q]) * p.c : -INFINITY;
                // Lazy column max (as the row-tile kernel's lazy rescale): the reference m[q] moves only
                // when some score of column q exceeds it by more than 2^8, so P <= 256 and the final
                // O = acc / L and LSE = m + log2 L are exact for any reference.  Usually no column
                // moves and no max is reduced: one OR of flags across the four warps decides.
                float(*rb)[kN] = red_max[tile_ctr & 1];
                uint32_t need = 0;
#pragma unroll
                for (int q = 0; q < kN; ++q)
                    if (q < G && x[q] > m[q] + kRescaleD) need |= 1u << q;
                need = __reduce_or_sync(0xffffffffu, need);
                if (lane == 0) red_need[tile_ctr & 1][warp] = need;
                named_bar_sync(1, 128);
                need = red_need[tile_ctr & 1][0] | red_need[tile_ctr & 1][1] | red_need[tile_ctr & 1][2] | red_need[tile_ctr & 1][3];
                if (need) {   // the same value in all four warps
#pragma unroll
                    for (int q = 0; q < kN; ++q)
                        if ((need >> q) & 1u) {
                            const float mx = warp_max(x[q]);
                            if (lane == 0) rb[warp][q] = mx;
                        }
                    named_bar_sync(1, 128);
                }
                ++tile_ctr;
                float alpha[kN], pv[kN];
#pragma unroll
                for (int q = 0; q < kN; ++q) {
                    if (q < G) {
                        alpha[q] = 1.f;
                        if ((need >> q) & 1u) {
                            const float mt = fmaxf(fmaxf(rb[0][q], rb[1][q]), fmaxf(rb[2][q], rb[3][q]));
                            // a column without a finite reference yet has nothing to rescale
                            alpha[q] = m[q] == -INFINITY ? 0.f : ex2_approx(m[q] - mt);
                            m[q] = mt;
                        }
                        // a column with no visible key so far keeps m = -inf (no -inf - -inf)
                        pv[q] = m[q] == -INFINITY ? 0.f : ex2_approx(x[q] - m[q]);
                        l[q] = fmaf(l[q], alpha[q], pv[q]);
                    } else {
                        alpha[q] = 0.f;
                        pv[q] = 0.f;
                    }
                }
                // Keys at or beyond n in a partial tile: their V rows may hold anything (NaN in
                // padded memory) and P = 0 does not cancel NaN in the MMA, so zero those rows.
                // Whole 128-byte rows are zeroed, which the swizzle only permutes within.
                if ((t + 1) * kTileKV > it.n) {
                    mbar_wait(&v_full[vr.idx], vr.phase, wc);
                    if (!valid) {
                        uint8_t* rowp = smem + C::kOffV + vr.idx * C::kKVBytes + tid * 128;
#pragma unroll
                        for (int a = 0; a < C::kAtoms; ++a)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                reinterpret_cast<uint4*>(rowp + a * (kTileKV * 128))[i] = make_uint4(0, 0, 0, 0);
                    }
                }
                vr.advance();
                mbar_wait(&p_empty[pr.idx], pr.phase ^ 1, wc);
                uint8_t* sP = smem + C::kOffP + pr.idx * C::kPBytes;
#pragma unroll
                for (int q = 0; q < kN; ++q)
                    *reinterpret_cast<uint16_t*>(sP + sw128_offset(q, tid, kN * 128)) = float_to_bf16_bits(pv[q]);
                fence_proxy_async_smem();
                mbar_arrive(&p_full[pr.idx]);
                pr.advance();
                if (t > it.t0) consume(alpha_prev);
#pragma unroll
                for (int q = 0; q < kN; ++q) alpha_prev[q] = alpha[q];
            }
            if (it.t1 > it.t0) consume(alpha_prev);

            if constexpr (!EPI) {
                run_epilogue(it, it.t1 <= it.t0, m, l, acc, tid, warp, 1, false);
                continue;
            }
            // ---- hand the item to the epilogue warpgroup: acc and the partial column sums l through
            // Tensor Memory (lane tid), the reference maxima through shared memory; the softmax goes
            // on with the next item meanwhile.  Both sides walk the same item sequence and take part
            // in every handoff whatever their waits return (a timeout only drains).
            {
                mbar_wait(&ep_empty[hr.idx], hr.phase ^ 1, wc);
                tc_fence_after();
                __syncwarp();   // tcgen05.st is warp-collective
                uint32_t hv[32];
#pragma unroll
                for (int q = 0; q < kN; ++q) {
                    hv[q] = __float_as_uint(acc[q]);
                    hv[kN + q] = __float_as_uint(l[q]);
                }
                tmem_st32(tmem + lane_base + 64 + hr.idx * 32, hv);
                tmem_st_wait();
                if (tid == 0)
#pragma unroll
                    for (int q = 0; q < kN; ++q) ep_m[hr.idx][q] = m[q];
                tc_fence_before();
                mbar_arrive(&ep_full[hr.idx]);
            }
            hr.advance();
        }
    } else {
      if constexpr (EPI) {
        setmaxnreg_inc<kRegsEpi>();
        // ------------------------------------------------ epilogue (128 threads): the items the softmax
        // warpgroup hands over, in order; thread tid owns O^T row tid (Tensor Memory lane tid)
        const int tid = threadIdx.x - 128;
        const int ew = warp - 4;
        const uint32_t lane_base = static_cast<uint32_t>(ew * 32) << 16;
        Ring hr(2);
        while (sched.next(it)) {   // the softmax warpgroup's sequence of items
            // a partial's slots (64-bit divisions) while the softmax warps still stream the item, off
            // the path from its last tile to its arrival count
            const bool pre = p.fixup && !(it.whole && !(p.split && p.nv_codes)) && it.t1 > it.t0;
            if (pre && tid == 0) fx_n = unit_partial_slots(p, it.u, static_cast<int>(gridDim.x), fx_slot, kMaxFixSlots);
            mbar_wait(&ep_full[hr.idx], hr.phase, wc);
            tc_fence_after();
            __syncwarp();   // tcgen05.ld is warp-collective
            const bool empty = it.t1 <= it.t0;
            float m[kN], l[kN], acc[kN];
            {
                uint32_t hv[32];
                tmem_ld32(tmem + lane_base + 64 + hr.idx * 32, hv);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < kN; ++q) {
                    acc[q] = __uint_as_float(hv[q]);
                    l[q] = __uint_as_float(hv[kN + q]);
                    m[q] = ep_m[hr.idx][q];
                }
            }
            tc_fence_before();
            mbar_arrive(&ep_empty[hr.idx]);
            hr.advance();

            run_epilogue(it, empty, m, l, acc, tid, ew, 2, pre);
        }
      }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == mma_warp<EPI>()) tmem_dealloc(tmem, C::kTmemCols);
}

// Exclusive prefix of per-unit tile counts (ragged keys), one block.
__global__ void __launch_bounds__(1024) tile_prefix_kernel(const int32_t* seqlens, int Hkv, int U, int32_t* prefix)
{
    griddep_launch_dependents();
    griddep_wait();
    __shared__ int part[1024];
    const int per = (U + 1023) / 1024;
    const int b0 = threadIdx.x * per;
    int s = 0;
    for (int u = b0; u < min(U, b0 + per); ++u) s += (seqlens[u / Hkv] + kTileKV - 1) / kTileKV;
    part[threadIdx.x] = s;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int u = b0; u < min(U, b0 + per); ++u) {
        prefix[u] = run;
        run += (seqlens[u / Hkv] + kTileKV - 1) / kTileKV;
    }
    if (threadIdx.x == 1023) prefix[U] = part[1023];
}

// Merges the partial results of units whose tiles were split over several CTAs, and writes the
// result of units without keys (O = 0, LSE = -inf).  One block of D threads per query row; warp 0
// finds the CTAs holding partials of the unit once per block (64-bit divisions).
constexpr int kMaxPartsD = 512;

__global__ void combine_kernel(const __grid_constant__ DecodeParams p, int nctas)
{
    __shared__ int slots[kMaxPartsD];
    __shared__ float weights[kMaxPartsD];
    __shared__ int nslots;
    __shared__ float lse_sh;
    griddep_launch_dependents();
    griddep_wait();
    const int row = blockIdx.x;
    const int u = row / p.G;
    const int q = row % p.G;
    const int d = threadIdx.x;
    const int D = p.D;
    if (threadIdx.x < 32) {
        int tiles;
        long long Tu, T;
        if (p.prefix) {
            tiles = p.prefix[u + 1] - p.prefix[u];
            Tu = p.prefix[u];
            T = p.prefix[p.U];
        } else {
            tiles = p.tiles_uniform;
            Tu = static_cast<long long>(u) * tiles;
            T = static_cast<long long>(p.U) * tiles;
        }
        int cnt = 0;
        if (tiles > 0) {
            const long long P = nctas;
            const int c0 = static_cast<int>(min((((Tu + 1) * P) - 1) / T, P - 1));
            const int c1 = static_cast<int>(min((((Tu + tiles) * P) - 1) / T, P - 1));
            if (c0 == c1 && !p.nv_codes) {
                cnt = -1;   // one CTA held the whole unit and wrote it
            } else {
                for (int cw = c0; cw <= c1; cw += 32) {
                    const int c = cw + static_cast<int>(threadIdx.x);
                    // CTAs with an empty tile range (possible when T < P) hold no partial
                    const bool ok = c <= c1 && (c * T) / P != ((c + 1) * T) / P;
                    const unsigned m = __ballot_sync(0xffffffffu, ok);
                    if (ok) {
                        const int idx = cnt + __popc(m & ((1u << threadIdx.x) - 1u));
                        if (idx < kMaxPartsD) slots[idx] = u + c;
                    }
                    cnt += __popc(m);
                }
                cnt = min(cnt, kMaxPartsD);
            }
        }
        __syncwarp();
        // LSE of the merged row and each partial's weight exp(lse_i - lse), once per block
        float mx = -INFINITY;
        for (int i = static_cast<int>(threadIdx.x); i < cnt; i += 32) mx = fmaxf(mx, p.part_lse[static_cast<size_t>(slots[i]) * kN + q]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // partials without a visible key carry lse = -inf and weigh 0; all of them -> empty row
        const bool any = mx > -INFINITY;
        float sum = 0.f;
        if (any)
            for (int i = static_cast<int>(threadIdx.x); i < cnt; i += 32) sum += __expf(p.part_lse[static_cast<size_t>(slots[i]) * kN + q] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float lse_all = (cnt > 0 && any) ? mx + __logf(sum) : -INFINITY;
        for (int i = static_cast<int>(threadIdx.x); i < cnt; i += 32)
            weights[i] = any ? __expf(p.part_lse[static_cast<size_t>(slots[i]) * kN + q] - lse_all) : 0.f;
        if (threadIdx.x == 0) {
            nslots = cnt;
            lse_sh = lse_all;
        }
    }
    __syncthreads();
    const int ns = nslots;
    if (ns < 0) return;
    float o = 0.f;
    const float lse_v = lse_sh;
#pragma unroll 4
    for (int i = 0; i < ns; ++i) o = fmaf(weights[i], p.part_o[(static_cast<size_t>(slots[i]) * kN + q) * D + d], o);
    const size_t r = static_cast<size_t>(row);
    if (p.o_stage) p.o_stage[r * D + d] = o;
    if (p.out) {
        if (p.out_f32)
            static_cast<float*>(p.out)[r * D + d] = o;
        else
            static_cast<uint16_t*>(p.out)[r * D + d] = float_to_bf16_bits(o);
    }
    if (d == 0 && p.lse) p.lse[r] = lse_v;
    if (p.nv_codes) nvfp4_encode_lanes(o, *p.nv_sg, d, p.nv_codes + r * (D / 2), p.nv_scales + r * (D / 16));
    if (p.amax_bits) {
        const float wm = warp_max(fabsf(o));
        if ((threadIdx.x & 31) == 0 && wm > 0.f) atomicMax(p.amax_bits, __float_as_uint(wm));
    }
}

}  // namespace

// ---- host side ------------------------------------------------------------------------------------
namespace {

struct DecodeWs {
    size_t prefix_off, ctr_off, lse_off, o_off, stage_off, total;
};

DecodeWs decode_ws_layout(const AttnArgs& a, bool split, int nsm)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t U = static_cast<size_t>(a.B) * a.Hkv;
    const size_t slots = split ? U + nsm : 0;
    DecodeWs w{};
    size_t off = 0;
    w.prefix_off = off;
    off += (split && a.seqlens) ? al((U + 1) * 4) : 0;
    w.ctr_off = off;
    off += split ? al(U * 8) : 0;   // fixup arrival counters
    w.lse_off = off;
    off += al(slots * kN * 4);
    w.o_off = off;
    off += al(slots * kN * a.D * 4);
    w.stage_off = off;
    const bool stage = (a.out_kind == FMHA_OUT_NVFP4) && !a.out_f32 && !a.nv_sg;
    off += stage ? al(static_cast<size_t>(a.B) * a.Hq * a.Sq * a.D * 4) : 0;
    w.total = off;
    return w;
}

template <int D, bool CAUSAL>
int run_decode(const AttnArgs& a, bool split, void* ws, cudaStream_t st)
{
    using C = DecodeCfg<D>;
    const int nsm = num_sms();
    if (nsm <= 0) return set_error(FMHA_ERR_CUDA, "cannot query the SM count");
    const int U = a.B * a.Hkv;
    const int G = (a.Hq / a.Hkv) * a.Sq;
    const DecodeWs w = decode_ws_layout(a, split, nsm);
    uint8_t* base = static_cast<uint8_t*>(ws);

    CUtensorMap qmap, kmap, vmap;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(G), static_cast<uint64_t>(U)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(G) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(kN), 1};
        int rc = make_tmap_bf16(&qmap, a.q, 3, dims, strides, box);
        if (rc) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Skv), static_cast<uint64_t>(U)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Skv) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(kTileKV), 1};
        int rc = make_tmap_bf16(&kmap, a.k, 3, dims, strides, box);
        if (rc) return rc;
        rc = make_tmap_bf16(&vmap, a.v, 3, dims, strides, box);
        if (rc) return rc;
    }

    DecodeParams p{};
    p.U = U;
    p.Hkv = a.Hkv;
    p.G = G;
    p.Skv = a.Skv;
    p.D = D;
    p.Sq = a.Sq > 0 ? a.Sq : 1;
    p.c = a.scale * kLog2e;
    p.seqlens = a.seqlens;
    p.tiles_uniform = (a.Skv + kTileKV - 1) / kTileKV;
    p.split = split ? 1 : 0;
    p.prefix = (split && a.seqlens) ? reinterpret_cast<const int32_t*>(base + w.prefix_off) : nullptr;
    const bool nvfp4 = a.out_kind == FMHA_OUT_NVFP4;
    p.out = nvfp4 ? nullptr : a.out;
    p.out_f32 = a.out_kind == FMHA_OUT_F32 ? 1 : 0;
    p.lse = a.lse;
    p.o_stage = nvfp4 ? (a.out_f32 ? a.out_f32 : (a.nv_sg ? nullptr : reinterpret_cast<float*>(base + w.stage_off))) : nullptr;
    p.amax_bits = nvfp4 ? reinterpret_cast<unsigned*>(a.amax_slot) : nullptr;
    p.nv_sg = a.nv_sg;
    p.nv_codes = a.nv_codes;
    p.nv_scales = a.nv_scales;
    p.nv_ts = a.nv_ts;
    p.part_lse = split ? reinterpret_cast<float*>(base + w.lse_off) : nullptr;
    p.part_o = split ? reinterpret_cast<float*>(base + w.o_off) : nullptr;
    // Split units are merged in the kernel by the CTA completing them (a unit's last partial lands
    // at the end of a CTA's range, so the merge costs a few microseconds of tail instead of the
    // combine launch).  Measured slower for ragged batches, which keep the combine kernel (it also
    // writes units without keys); single-pass NVFP4 keeps it too (one block per row encodes).
    p.fixup = (split && !a.nv_sg && !a.seqlens && nsm <= kMaxFixSlots) ? 1 : 0;
    p.unit_ctr = split ? reinterpret_cast<unsigned long long*>(base + w.ctr_off) : nullptr;
    p.gen = next_call_tag();
    p.status = device_status_ptr();
    p.limit = wait_limit();

    if (p.prefix) {
        FMHA_CHECK_CUDA(launch_pdl(tile_prefix_kernel, dim3(1), dim3(1024), 0, st, a.seqlens, a.Hkv, U,
                                   const_cast<int32_t*>(p.prefix)));
        count_launch();
    }
    // The epilogue warpgroup takes each item's epilogue off the softmax warps when a unit has several
    // query columns (publishing a 16-column partial costs several tiles' streaming time); with one
    // column the epilogue is short and the six-warp kernel, whose softmax warps run it, measured faster.
    const bool epi = G > 1;
    const void* fn = epi ? reinterpret_cast<const void*>(decode_kernel<D, CAUSAL, true>)
                         : reinterpret_cast<const void*>(decode_kernel<D, CAUSAL, false>);
    FMHA_CHECK_CUDA(set_smem_limit_once(fn, C::kSmemBytes));
    // one CTA per SM, or one per key tile when a uniform-length problem has fewer tiles than SMs (a
    // small problem then launches only the CTAs that have work)
    int grid = split ? nsm : (U < nsm ? U : nsm);
    if (split && !p.prefix) {
        const long long tiles = static_cast<long long>(U) * p.tiles_uniform;
        if (tiles < grid) {
            grid = static_cast<int>(tiles);
        } else {
            // When the units divide evenly over at least 5/6 of the SMs, each CTA streams the same
            // number of whole units: no partial to publish or merge, and that many SMs still keep
            // HBM busy (B8 H32 Skv4096: 128 CTAs of two units 87.3 us, 152 CTAs of 53.9 tiles 88.6)
            for (int g = grid; 6 * g >= 5 * nsm; --g)
                if (U % g == 0) {
                    grid = g;
                    break;
                }
        }
    }
    if (grid > 0) {
        timing_mark_begin(st);
        const cudaError_t e = epi ? launch_pdl(decode_kernel<D, CAUSAL, true>, dim3(static_cast<unsigned>(grid)),
                                               dim3(decode_threads<true>()), C::kSmemBytes, st, qmap, kmap, vmap, p)
                                  : launch_pdl(decode_kernel<D, CAUSAL, false>, dim3(static_cast<unsigned>(grid)),
                                               dim3(decode_threads<false>()), C::kSmemBytes, st, qmap, kmap, vmap, p);
        timing_mark_end(st);
        FMHA_CHECK_CUDA(e);
        count_launch();
    }
    if (split && !p.fixup && U * G > 0) {
        FMHA_CHECK_CUDA(launch_pdl(combine_kernel, dim3(static_cast<unsigned>(U * G)), dim3(static_cast<unsigned>(D)), 0,
                                   st, p, grid));
        count_launch();
    }
    return FMHA_OK;
}

}  // namespace

size_t decode_workspace_bytes(const AttnArgs& a, int num_splits)
{
    const int nsm = num_sms() > 0 ? num_sms() : 256;   // sized for the largest plausible SM count
    const bool split = num_splits != 1;
    return decode_ws_layout(a, split, nsm).total;
}

int launch_decode(const AttnArgs& a, int num_splits, void* ws, size_t ws_bytes, cudaStream_t st)
{
    const bool split = num_splits != 1 && ws != nullptr;
    const int nsm = num_sms();
    const DecodeWs w = decode_ws_layout(a, split, nsm);
    if (w.total > 0 && (!ws || ws_bytes < w.total)) return set_error(FMHA_ERR_WORKSPACE, "decode: workspace too small");
    switch (a.D) {
        case 64: return a.causal ? run_decode<64, true>(a, split, ws, st) : run_decode<64, false>(a, split, ws, st);
        case 128: return a.causal ? run_decode<128, true>(a, split, ws, st) : run_decode<128, false>(a, split, ws, st);
        default: return set_error(FMHA_ERR_UNSUPPORTED, "decode path: D must be 64 or 128");
    }
}

}  // namespace atc_gb300

// ================================================================================================
// Split-KV decode without any device allocation by the caller or the library.
//
// Some callers cannot provide the workspace that fmha_fwd_ex's split-KV path needs: plug-ins and
// foreign-language bindings that are handed only tensor pointers and have no allocator to ask,
// and latency-critical loops that must not call cudaMalloc (it can synchronise the device and
// its latency is unbounded).  For them the split partials and the tile prefix live in the fixed
// array below, which every GPU that loads this library holds until the process exits.
//
// The array is shared by every call on a device and keeps the contents of the last call.  No
// part of it needs to start at zero: each byte a call reads (tile prefix, partial O and LSE) is
// written earlier in the same call.  Calls that overlap on the GPU (different streams, or
// different host threads, without ordering between them) race on it.
// ================================================================================================
static __device__ __align__(256) unsigned char g_fmha_decode_scratch[FMHA_NOALLOC_SCRATCH_BYTES];

namespace atc_gb300 {
namespace {

constexpr int kMaxScratchDevices = 64;
std::atomic<void*> g_decode_scratch_addr[kMaxScratchDevices];

// Device address of the scratch array on the current device, looked up once per device (with
// that device current) and cached.
int decode_scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxScratchDevices) return set_error(FMHA_ERR_UNSUPPORTED, "device index out of range");
    void* p = g_decode_scratch_addr[dev].load();
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_fmha_decode_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(decode scratch)");
        g_decode_scratch_addr[dev].store(p);
    }
    *out = p;
    return FMHA_OK;
}

}  // namespace
}  // namespace atc_gb300

extern "C" int fmha_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                       int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                                       const int32_t* seqlens_k, fmha_stream_t stream)
{
    using namespace atc_gb300;
    if (!q || !k || !v || !out) return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: NULL q/k/v/out");
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0 || Hq % Hkv != 0)
        return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: need B >= 0, Sq >= 0, Skv >= 1, Hq % Hkv == 0");
    if (D != 64 && D != 128) return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: D must be 64 or 128");
    if (!(scale > 0.f) || !(scale < INFINITY))
        return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: scale must be a positive finite number");
    if (static_cast<long long>(Hq / Hkv) * Sq > 16)
        return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: at most 16 query rows per key/value head");
    auto mis = [](const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & m) != 0; };
    if (mis(q, 15) || mis(k, 15) || mis(v, 15) || mis(out, 15) || mis(lse, 3) || mis(seqlens_k, 3))
        return set_error(FMHA_ERR_INVALID, "fmha_fwd_decode_noalloc: q/k/v/out 16-byte, lse/seqlens 4-byte aligned");
    if (static_cast<long long>(B) * Hkv * Skv >= (1LL << 31))
        return set_error(FMHA_ERR_UNSUPPORTED, "fmha_fwd_decode_noalloc: more than 2^31 key rows");
    if (static_cast<long long>(B) * Hq * Sq == 0) return FMHA_OK;
    if (!device_status_ptr()) return set_error(FMHA_ERR_CUDA, "no CUDA device");

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
    a.seqlens = seqlens_k;
    a.out_kind = FMHA_OUT_BF16;
    const size_t need = decode_workspace_bytes(a, 0);
    if (need > FMHA_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "fmha_fwd_decode_noalloc: this problem needs %zu bytes of split-KV scratch, the static area holds %zu "
                 "(B*Hkv and the SM count set the size)",
                 need, static_cast<size_t>(FMHA_NOALLOC_SCRATCH_BYTES));
        return set_error(FMHA_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    int rc = decode_scratch_address(&scratch);
    if (rc) return rc;
    return launch_decode(a, 0, scratch, FMHA_NOALLOC_SCRATCH_BYTES, reinterpret_cast<cudaStream_t>(stream));
}

