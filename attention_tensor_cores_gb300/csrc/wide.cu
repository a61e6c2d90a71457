// Wide-head attention (D = 512 for K and V), e.g. 128 query heads sharing one key/value head.
//
// Same computation as the other paths ("NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md", nvfp4-megamoe-kernel,
// kernel plan: TMA loads, tcgen05 QK and PV with Tensor Memory accumulators, in-kernel softmax with O
// rescale, multi-KV-tile, and the pages' goal of head dims up to 512).  What D = 512 changes on
// GB300: an FP32 O tile of 128 rows x 512 columns is all 512 Tensor Memory columns, and the 128 x 512
// BF16 Q tile alone is 128 KB of shared memory.  The design:
//
//  * CTA pairs split the value dimension: CTA h of a pair accumulates O[:, 256h : 256h + 256] (256
//    TMEM columns).  Both CTAs of the pair compute the full S = Q K^T, so each holds all of Q.
//  * 128-key tiles: the QK MMA is M = 128 query rows by N = 128 keys, so each K = 16 step reads a
//    4 KB slice of Q for 256K MACs (with 32-key tiles the Q re-reads made the tensor core's
//    shared-memory operand path the limiter).  A 128-key K tile (128 KB) and Q (128 KB) do not fit
//    together, so K and V stream through one ring of 16 KB chunks: a K chunk is 64 of the 512
//    contraction columns of the tile's 128 keys, a V chunk is 32 keys by this CTA's 256 columns.
//    Chunks go through the ring in the order the MMAs use them: K(0); K(j), V(j-1) for each later
//    tile j; then V of the last tile.
//  * Tensor Memory: S (128 columns), P (64 columns of BF16 pairs), O half (256 columns).  QK(j+1)
//    only needs the softmax to have read S(j), so it runs while the softmax of j works; PV(j) needs
//    P(j).  The tensor pipe then alternates QK(j+1), PV(j) without waiting on the softmax.
//  * Stream-K over keys: the tiles of all units (b, kv-head, 128-row block) are laid end to end and
//    pair p of P takes [p*T/P, (p+1)*T/P); a run that covers a whole unit writes O and LSE,
//    otherwise a normalised partial goes to slot unit + p and the combine kernel merges them.  With
//    uniform lengths the CTA-pair variant leaves empty positions after each unit on that line.
//    Without a workspace (no split), pair p takes whole units p, p + P, ... and writes them itself:
//    no partials, no combine launch.
//  * Roles: warps 0-3 softmax (one query row per thread, lazy rescale as in the row-tile kernel),
//    warp 4 loads Q, K and V, warp 5 issues the MMAs in order.  All waits are bounded.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"
#include "nvfp4_dev.cuh"
#include "ptx.cuh"

namespace atc_gb300 {
namespace {

constexpr int kWD = 512;            // head dim of Q/K/V
constexpr int kWHalf = 256;         // value columns per CTA
constexpr int kWRows = 128;         // query rows per unit (MMA M)
constexpr int kWKeys = 128;         // keys per tile (QK N, PV K)
constexpr int kWKChunks = 8;        // K chunks per tile: 64 contraction columns each
constexpr int kWVKeys = 32;         // keys per V chunk
constexpr int kWThreads = 192;      // 4 softmax warps, producer, MMA issuer
constexpr float kLog2eW = 1.4426950408889634f;
constexpr float kLn2W = 0.6931471805599453f;
constexpr float kRescaleW = 8.0f;

constexpr int kWQBytes = 8 * kWRows * 128;          // 8 atoms of 128 rows x 128 B = 128 KB
constexpr int kWOffQ = 0;
constexpr int kWOffRing = kWOffQ + kWQBytes;

// Chunk geometry of the two variants.
//  * Independent CTAs (PAIR = false): a K chunk is 64 contraction columns of the tile's 128 keys
//    (16 KB), a V chunk 32 keys by this CTA's 256 value columns (4 atoms, 16 KB); 6 ring slots.
//  * CTA-pair MMA (PAIR = true): a K chunk is 64 columns of this CTA's 64 keys of the tile (8 KB), a
//    V chunk 32 keys by 128 value columns (2 atoms, 8 KB), the lower part (value columns 128h..) and
//    then the upper part (256 + 128h..) of CTA h; 12 ring slots.
template <bool PAIR>
struct WCfg {
    static constexpr int kKRows = PAIR ? 64 : 128;          // keys of one K chunk held by this CTA
    static constexpr int kVAtoms = PAIR ? 2 : 4;            // 64-column atoms of a V chunk
    static constexpr int kVChunks = PAIR ? 8 : 4;           // V chunks per tile
    static constexpr int kChunkBytes = PAIR ? 8192 : 16384;
    static constexpr int kSlots = PAIR ? 12 : 6;
    static constexpr int kPeriod = kWKChunks + kVChunks;    // chunks per tile
    static constexpr int kSmem = kWOffRing + kSlots * kChunkBytes + 1024;
    static_assert(kKRows * 128 == kChunkBytes && kVAtoms * kWVKeys * 128 == kChunkBytes, "chunk layouts");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};
// TMEM columns: S 0..127, P 128..191 (BF16 pairs of 128 keys; the pair variant uses 128..255, see the
// kernel), O half 256..511.
constexpr uint32_t kWColS = 0, kWColP = 128, kWColO = 256;
// A pair that ends one unit and starts the next pays one more epilogue (a partial) and one more Q load
// than a pair inside a unit.  With uniform lengths each unit can be followed by empty positions on the
// stream-K split line, so that such pairs get fewer tiles.  Measured on B32 Hq128 Skv16384 (one GB300,
// gaps 0-4): the CTA-pair kernel's step 232.3-233.0 -> 229.4-230.0 us with 2; the independent kernel
// flat from 0 to 2 and slower beyond, so it keeps none.
constexpr int kWSplitGapPair = 2;

// Position of chunk c of V(j) in an item's chunk sequence K(0); K(1), V(0); ...; K(T-1), V(T-2); V(T-1).
template <bool PAIR>
__device__ __forceinline__ uint32_t wv_chunk_pos(int j, int T, int c)
{
    constexpr int P = WCfg<PAIR>::kPeriod;
    return static_cast<uint32_t>(j < T - 1 ? P * j + 2 * kWKChunks + c : P * j + kWKChunks + c);
}

struct WideParams {
    int U;          // units = B * Hkv * row_tiles
    int row_tiles;  // ceil(R / 128)
    int Hkv;
    int R;          // query rows per (b, kv-head) = (Hq / Hkv) * Sq
    int Skv;
    int Sq;         // query rows per head: row r of a (b, kv-head) is query r % Sq
    int causal;     // bottom-right aligned causal mask
    float c;
    const int32_t* seqlens;
    const int32_t* prefix;   // [U+1] tile prefix (ragged), else NULL
    int tiles_uniform;
    int gap;            // split with uniform lengths: empty positions after each unit on the split line
    int whole_units;    // 1: no split, pair p handles units p, p + P, ... whole (no workspace)
    void* out;
    int out_f32;
    float* lse;
    float* o_stage;
    unsigned* amax_bits;
    const float* nv_sg;      // single-pass NVFP4: given s_g; codes/scales written here, else NULL
    uint8_t* nv_codes;
    uint8_t* nv_scales;
    float* nv_ts;
    float* part_o;      // [slots][64 column groups of 8][128 rows][8], see wpart_index
    float* part_lse;    // [slots][128]
    int* status;
    long long limit;
};

// Offset of partial O element (slot, row, col).  Each 8-column group keeps its 128 rows side by
// side, so a warp storing 8 columns of 32 consecutive rows writes 1 KB of contiguous memory, and
// a row's 8 columns are one 32-byte sector.
__host__ __device__ __forceinline__ size_t wpart_index(size_t slot, int row, int col)
{
    return ((slot * (kWD / 8) + static_cast<size_t>(col >> 3)) * kWRows + row) * 8 + (col & 7);
}

struct WItem {
    int u, t0, t1, n;
    bool whole;
    int slot;
};

// Unit u -> (b*Hkv + kvh, 128-row block).
__device__ __forceinline__ int wunit_head(const WideParams& p, int u) { return u / p.row_tiles; }
__device__ __forceinline__ int wunit_keys(const WideParams& p, int u)
{
    return p.seqlens ? p.seqlens[wunit_head(p, u) / p.Hkv] : p.Skv;
}
__device__ __forceinline__ int wunit_tiles(const WideParams& p, int u)
{
    if (p.prefix) return p.prefix[u + 1] - p.prefix[u];
    return (wunit_keys(p, u) + kWKeys - 1) / kWKeys;
}
// Start of unit u on the stream-K split line: its tiles, then (uniform lengths) p.gap empty positions.
__device__ __forceinline__ long long wunit_start(const WideParams& p, int u)
{
    return p.prefix ? static_cast<long long>(p.prefix[u]) : static_cast<long long>(u) * (p.tiles_uniform + p.gap);
}
__device__ __forceinline__ long long wsplit_total(const WideParams& p)
{
    return p.prefix ? static_cast<long long>(p.prefix[p.U]) : static_cast<long long>(p.U) * (p.tiles_uniform + p.gap);
}

struct WSched {
    const WideParams* p;
    long long g, g1;
    int pair, step;
    __device__ void init(const WideParams* pp, int pr, int npairs)
    {
        p = pp;
        pair = pr;
        step = npairs;
        if (p->whole_units) {
            g = pr;
            g1 = p->U;
            return;
        }
        const long long T = wsplit_total(*p);
        g = (static_cast<long long>(pr) * T) / npairs;
        g1 = (static_cast<long long>(pr + 1) * T) / npairs;
    }
    __device__ bool next(WItem& it)
    {
        if (g >= g1) return false;
        if (p->whole_units) {
            const int uu = static_cast<int>(g);
            it.u = uu;
            it.t0 = 0;
            it.t1 = wunit_tiles(*p, uu);
            it.n = wunit_keys(*p, uu);
            it.whole = true;
            it.slot = 0;
            g += step;
            return true;
        }
        int uu;
        if (p->prefix) {
            int lo = 0, hi = p->U - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p->prefix[mid] <= g) lo = mid; else hi = mid - 1;
            }
            uu = lo;
        } else {
            const long long len = p->tiles_uniform + p->gap;
            uu = static_cast<int>(g / len);
            if (g - uu * len >= p->tiles_uniform) {   // in the empty positions after unit uu
                g = (uu + 1) * len;
                if (g >= g1) return false;
                ++uu;
            }
        }
        const long long s = wunit_start(*p, uu);
        const int nt = wunit_tiles(*p, uu);
        it.u = uu;
        it.t0 = static_cast<int>(g - s);
        it.t1 = static_cast<int>(min(static_cast<long long>(nt), g1 - s));
        it.n = wunit_keys(*p, uu);
        it.whole = (it.t0 == 0 && it.t1 == nt);
        it.slot = uu + pair;
        g = s + it.t1;
        return true;
    }
};

__device__ __forceinline__ void wdrain(uint64_t* bar, uint32_t parity, long long limit)
{
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

struct WRing {
    uint32_t idx = 0, phase = 0;
    int n;
    __device__ explicit WRing(int stages) : n(stages) {}
    __device__ void advance()
    {
        if (++idx == static_cast<uint32_t>(n)) {
            idx = 0;
            phase ^= 1;
        }
    }
};

// PAIR = false: the two CTAs of a pair run independently (each loads every K chunk, each computes
// the full S).  PAIR = true: the pair is a cluster of two CTAs and both products are pair MMAs
// (tcgen05 cta_group::2, issued by the even CTA): CTA h loads only keys 64h..64h+63 of each K tile,
// and the QK MMA (M = 256 with Q in both CTAs, N = the tile's 128 keys, half from each CTA's shared
// memory) leaves the full S in both CTAs' Tensor Memory.  The PV MMA then has to produce different
// value columns in the two CTAs from one shared B operand, so it runs over a doubled contraction:
// CTA h's A operand is [P, 0] (h = 0) or [0, P] (h = 1), 256 BF16 columns of Tensor Memory, and B
// stacks the lower and upper value halves, B[k][n] = V[k][n] for k < 128 and V[k - 128][256 + n]
// above, its 256 columns split 128/128 between the CTAs.  D = P V[:, 256h : 256h + 256] in CTA h, the
// same output split as the independent variant.  Half of the PV work multiplies zeros; in exchange
// every K and V byte is read into shared memory once per pair.  Dense keys only (the ragged tail
// clears V rows in the CTA's own ring, which needs the CTA's own copy-completion barrier).
template <bool PAIR>
__global__ void __launch_bounds__(kWThreads, 1)
    wide_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const __grid_constant__ WideParams p)
{
    using C = WCfg<PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full[8], q_empty, c_full[C::kSlots], c_empty[C::kSlots];   // q_full: one per Q atom
    __shared__ uint64_t s_full, s_empty, p_full, o_done, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x / 32;
    griddep_launch_dependents();
    // this CTA's half of the value columns (PAIR: its rank in the cluster); the even CTA leads a pair
    const int half = PAIR ? static_cast<int>(cluster_ctarank()) : static_cast<int>(blockIdx.x & 1);
    const bool leader = !PAIR || half == 0;
    const WaitCtl wc{&abort_flag, p.status, p.limit};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int a = 0; a < 8; ++a) mbar_init(&q_full[a], 1);
        mbar_init(&q_empty, 1);
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&c_full[i], 1);
            mbar_init(&c_empty[i], 1);
        }
        mbar_init(&s_full, 1);
        // PAIR: one arrival per softmax warp of both CTAs (a cluster-scope release per thread would put a
        // memory barrier on every softmax thread's path twice per tile)
        mbar_init(&s_empty, PAIR ? 8 : 128);
        mbar_init(&p_full, PAIR ? 8 : 128);
        mbar_init(&o_done, 1);
        mbar_init(&mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&tmem_slot, 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tmem_slot, 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    griddep_wait();   // the previous kernel of the stream has completed: global memory from here on
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.nv_ts) *p.nv_ts = *p.nv_sg;   // single-pass NVFP4: report s_g
    // waits on the barriers the other CTA's softmax threads arrive on (cluster-scope acquire); copy and
    // MMA completions aimed at a barrier are waited for with the ordinary wait
    auto wait_x = [&](uint64_t* b, uint32_t parity) -> bool {
        if constexpr (PAIR) return mbar_wait_cluster(b, parity, wc);
        return mbar_wait(b, parity, wc);
    };
    // shared::cluster address of barrier b in the leading CTA / in the other CTA of the pair
    auto lead_bar = [&](uint64_t* b) -> uint32_t { return mapa_shared(smem_u32(b), 0); };
    auto other_bar = [&](uint64_t* b) -> uint32_t { return mapa_shared(smem_u32(b), static_cast<uint32_t>(half ^ 1)); };
    WSched sched;
    sched.init(&p, blockIdx.x >> 1, gridDim.x >> 1);
    WItem it;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer: Q per item, then the chunk sequence
        if (lane_id() == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            WRing cr(C::kSlots);
            uint32_t qn = 0, ccnt[C::kSlots], qcnt[8];   // items, and copies per ring slot / Q atom
            for (int i = 0; i < C::kSlots; ++i) ccnt[i] = 0;
            for (int a = 0; a < 8; ++a) qcnt[a] = 0;
            // a copy into this CTA's shared memory, completing on the current slot's barrier; with PAIR
            // the leader's barrier counts both CTAs' bytes
            auto load = [&](uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
                if constexpr (PAIR) {
                    if (!leader) {
                        tma_load_3d_pair(dst, m, lead_bar(bar), x, y, z);
                        return;
                    }
                }
                tma_load_3d(dst, m, bar, x, y, z);
            };
            // wait until this CTA's copy of the slot is free (the leader's MMA thread releases both)
            auto begin_chunk = [&]() -> bool {
                mbar_wait(&c_empty[cr.idx], cr.phase ^ 1, wc);
                if (aborted(wc)) return false;
                if (leader) mbar_arrive_expect_tx(&c_full[cr.idx], PAIR ? 2 * C::kChunkBytes : C::kChunkBytes);
                ++ccnt[cr.idx];
                return true;
            };
            // K chunks of tile t; with q_rt >= 0 (an item's first tile) each Q atom goes right before the K
            // chunk it multiplies, so the first MMAs wait for 32 KB instead of the whole 128 KB of Q
            auto load_k = [&](int hu, int t, int q_rt) {
                for (int a = 0; a < kWKChunks; ++a) {
                    if (q_rt >= 0 && !aborted(wc)) {
                        if (leader) mbar_arrive_expect_tx(&q_full[a], PAIR ? 2 * (kWRows * 128) : kWRows * 128);
                        load(smem + kWOffQ + a * (kWRows * 128), &qmap, &q_full[a], a * 64, q_rt * kWRows, hu);
                        ++qcnt[a];
                    }
                    if (begin_chunk())
                        load(smem + kWOffRing + cr.idx * C::kChunkBytes, &kmap, &c_full[cr.idx], a * 64,
                             t * kWKeys + (PAIR ? 64 * half : 0), hu);
                    cr.advance();
                }
            };
            auto load_v = [&](int hu, int t) {
                for (int c = 0; c < C::kVChunks; ++c) {
                    if (begin_chunk()) {
                        uint8_t* dst = smem + kWOffRing + cr.idx * C::kChunkBytes;
                        const int part = PAIR ? c / 4 : 0, cc = PAIR ? c % 4 : c;
                        const int x0 = PAIR ? part * 256 + half * 128 : half * kWHalf;
                        for (int a = 0; a < C::kVAtoms; ++a)
                            load(dst + a * (kWVKeys * 128), &vmap, &c_full[cr.idx], x0 + a * 64, t * kWKeys + cc * kWVKeys, hu);
                    }
                    cr.advance();
                }
            };
            while (sched.next(it)) {
                if (it.t1 <= it.t0) continue;   // a unit without keys: no Q either (its O is zero)
                const int hu = wunit_head(p, it.u);
                const int rt = it.u % p.row_tiles;
                mbar_wait(&q_empty, (qn & 1) ^ 1, wc);   // the previous item's MMAs are done with Q
                ++qn;
                load_k(hu, it.t0, rt);
                for (int t = it.t0 + 1; t < it.t1 && !aborted(wc); ++t) {
                    load_k(hu, t, -1);
                    load_v(hu, t - 1);
                }
                load_v(hu, it.t1 - 1);
            }
            // nothing may still be landing in shared memory when the CTA exits: the leader's barriers
            // count every copy of the pair; the other CTA waits for the release of its last chunks
            if (leader) {
                for (int i = 0; i < C::kSlots; ++i)
                    if (ccnt[i]) wdrain(&c_full[i], (ccnt[i] - 1) & 1, kDrainLimit);
                for (int a = 0; a < 8; ++a)
                    if (qcnt[a]) wdrain(&q_full[a], (qcnt[a] - 1) & 1, kDrainLimit);
            } else {
                for (int i = 0; i < C::kSlots; ++i)
                    if (ccnt[i]) wdrain(&c_empty[i], (ccnt[i] - 1) & 1, kDrainLimit);
                if (qn) wdrain(&q_empty, (qn - 1) & 1, kDrainLimit);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer (PAIR: the leading CTA only), in the chunk order
        if (leader && lane_id() == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(PAIR ? 256 : kWRows, kWKeys, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(PAIR ? 256 : kWRows, kWHalf, false, true);
            // a barrier of this CTA that the other CTA of a pair has a copy of: signal both
            auto commit_both = [&](uint64_t* b) {
                if constexpr (PAIR) {
                    mma_commit_pair(smem_u32(b));
                    mma_commit_pair(other_bar(b));
                } else {
                    mma_commit(b);
                }
            };
            WRing cr(C::kSlots);
            uint32_t qn = 0, ns = 0, np = 0;   // items, QKs and PVs so far (kernel life)
            const uint32_t sQ = smem_u32(smem + kWOffQ);
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
            // first_q: the item's first QK, whose Q atoms may still be landing (atom a with K chunk a)
            auto issue_qk = [&](bool first_q) {
                if (ns > 0) wait_x(&s_empty, (ns - 1) & 1);   // the softmax has read S
                for (int a = 0; a < kWKChunks; ++a) {
                    if (first_q) mbar_wait(&q_full[a], (qn - 1) & 1, wc);
                    mbar_wait(&c_full[cr.idx], cr.phase, wc);
                    if (aborted(wc)) return;
                    tc_fence_after();
                    const uint64_t dk = sdesc_sw128(smem_u32(smem + kWOffRing + cr.idx * C::kChunkBytes), 16, 1024);
                    const uint64_t dq = dq0 + ((a * (kWRows * 128)) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (a > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (PAIR)
                            mma_ss_pair(tmem + kWColS, dq + ((kk * 32) >> 4), dk + ((kk * 32) >> 4), idesc_qk, acc);
                        else
                            mma_ss(tmem + kWColS, dq + ((kk * 32) >> 4), dk + ((kk * 32) >> 4), idesc_qk, acc);
                    }
                    commit_both(&c_empty[cr.idx]);
                    cr.advance();
                }
                commit_both(&s_full);
                ++ns;
            };
            auto issue_pv = [&](bool first) {
                wait_x(&p_full, np & 1);
                for (int c = 0; c < C::kVChunks; ++c) {
                    mbar_wait(&c_full[cr.idx], cr.phase, wc);
                    if (aborted(wc)) return;
                    tc_fence_after();
                    const uint32_t sV = smem_u32(smem + kWOffRing + cr.idx * C::kChunkBytes);
#pragma unroll
                    for (int kq = 0; kq < kWVKeys / 16; ++kq) {
                        const uint64_t db = sdesc_sw128(sV + kq * 2048, kWVKeys * 128, 1024);
                        const uint32_t acc = (!first || c > 0 || kq > 0) ? 1u : 0u;
                        if constexpr (PAIR) {
                            // contraction index: key 32 (c % 4) + 16 kq of the lower (c < 4) or upper half
                            const uint32_t a_col = kWColP + (c / 4) * 64 + (c % 4) * 16 + kq * 8;
                            mma_ts_pair(tmem + kWColO, tmem + a_col, db, idesc_pv, acc);
                        } else {
                            mma_ts(tmem + kWColO, tmem + kWColP + (c * (kWVKeys / 16) + kq) * 8, db, idesc_pv, acc);
                        }
                    }
                    commit_both(&c_empty[cr.idx]);
                    cr.advance();
                }
                commit_both(&o_done);
                ++np;
            };
            while (sched.next(it)) {
                const int T = it.t1 - it.t0;
                if (T <= 0) continue;   // no keys, no Q loaded (the producer skips it too)
                ++qn;
                if (!aborted(wc)) {
                    issue_qk(true);
                    for (int j = 1; j < T && !aborted(wc); ++j) {
                        issue_qk(false);
                        issue_pv(j == 1);
                    }
                    if (!aborted(wc)) issue_pv(T == 1);
                }
                if (!aborted(wc)) commit_both(&q_empty);
            }
            if constexpr (PAIR)
                mma_commit_pair(smem_u32(&mma_done));
            else
                mma_commit(&mma_done);
            wdrain(&mma_done, 0, kDrainLimit);
        }
    } else if (warp < 4) {
        // ------------------------------------------------ softmax / epilogue, one query row per thread
        const int row_in_tile = warp * 32 + static_cast<int>(lane_id());
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        // P columns of this CTA; with PAIR the other CTA's 64 columns of the doubled contraction stay zero
        const uint32_t col_p = kWColP + (PAIR ? 64u * static_cast<uint32_t>(half) : 0u);
        if constexpr (PAIR) {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            const uint32_t col_z = kWColP + 64u * static_cast<uint32_t>(half ^ 1);
            tmem_st32(tmem + lane_base + col_z, z);
            tmem_st32(tmem + lane_base + col_z + 32, z);
            tmem_st_wait();
        }
        // arrive on a barrier of the leading CTA: every thread, or (PAIR) once per warp after all of its
        // lanes are past their Tensor Memory accesses
        auto arrive_lead = [&](uint64_t* b) {
            if constexpr (PAIR) {
                __syncwarp();
                if (lane_id() == 0) {
                    if (leader)
                        mbar_arrive(b);
                    else
                        mbar_arrive_cluster(lead_bar(b));
                }
                return;
            }
            mbar_arrive(b);
        };
        uint32_t g = 0;       // tiles (= S reads = PVs) so far, kernel life
        uint32_t gchunk = 0;  // chunk sequence position of the current item's first chunk
        while (sched.next(it)) {
            const int hu = wunit_head(p, it.u);
            const int row = (it.u % p.row_tiles) * kWRows + row_in_tile;
            const int T = it.t1 - it.t0;
            // keys this row sees: 0 .. lim - 1
            const int lim = p.causal ? min(it.n, (row < p.R ? row : 0) % p.Sq + it.n - p.Sq + 1) : it.n;
            float m_run = -INFINITY, l = 0.f;
            for (int t = it.t0; t < it.t1; ++t, ++g) {
                mbar_wait(&s_full, g & 1, wc);
                tc_fence_after();
                float s[kWKeys];
                uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
                for (int c4 = 0; c4 < kWKeys / 32; ++c4) tmem_ld32p(tmem + lane_base + kWColS + c4 * 32, su + c4 * 32);
                tmem_ld_wait();
                tc_fence_before();
                arrive_lead(&s_empty);
                if ((t + 1) * kWKeys > lim) {
#pragma unroll
                    for (int i = 0; i < kWKeys; ++i)
                        if (t * kWKeys + i >= lim) s[i] = -INFINITY;
                }
                float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int i = 4; i < kWKeys; i += 8) {
                    mx[0] = fmax3(mx[0], s[i], s[i + 1]);
                    mx[1] = fmax3(mx[1], s[i + 2], s[i + 3]);
                    if (i + 4 < kWKeys) {
                        mx[2] = fmax3(mx[2], s[i + 4], s[i + 5]);
                        mx[3] = fmax3(mx[3], s[i + 6], s[i + 7]);
                    }
                }
                const float mt = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * p.c;
                const bool rescale = mt > m_run + kRescaleW;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ex2_approx(m_run - mt);
                    m_run = mt;
                }
                const float mu = m_run == -INFINITY ? 0.f : -m_run;   // a row with no visible key yet
                const uint64_t cc = f32x2(p.c, p.c);
                const uint64_t nm = f32x2(mu, mu);
                uint32_t pk[kWKeys / 2];
                uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int i = 0; i < kWKeys; i += 2) {
                    float x0, x1;
                    f32x2_split(ffma2(f32x2(s[i], s[i + 1]), cc, nm), x0, x1);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    ls[(i >> 1) & 3] = fadd2(ls[(i >> 1) & 3], f32x2(p0, p1));
                    pk[i >> 1] = pack_bf16x2(p0, p1);
                }
                float la, lb;
                f32x2_split(fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3])), la, lb);
                l = fmaf(l, alpha, la + lb);
                // the previous PV must be done: the P buffer is reused and O must be stable
                if (t > it.t0) mbar_wait(&o_done, (g - 1) & 1, wc);
                tc_fence_after();
                // ragged keys: V rows at or beyond n may hold NaN, and P = 0 does not cancel it
                if (!PAIR && p.seqlens && (t + 1) * kWKeys > it.n) {
                    const int j = t - it.t0;
                    for (int c = 0; c < C::kVChunks; ++c) {
                        const int r0 = it.n - (t * kWKeys + c * kWVKeys);   // first row to clear in this chunk
                        if (r0 >= kWVKeys) continue;
                        const uint32_t pos = gchunk + wv_chunk_pos<PAIR>(j, T, c);
                        const uint32_t slot = pos % C::kSlots;
                        mbar_wait(&c_full[slot], (pos / C::kSlots) & 1, wc);
                        // 128 threads clear rows max(r0, 0) .. 31: row = thread / 4, one 64-column atom each
                        const int r = row_in_tile >> 2, a = row_in_tile & 3;
                        if (r >= (r0 > 0 ? r0 : 0)) {
                            uint4* rowp = reinterpret_cast<uint4*>(smem + kWOffRing + slot * C::kChunkBytes + a * (kWVKeys * 128) + r * 128);
#pragma unroll
                            for (int i = 0; i < 8; ++i) rowp[i] = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (__any_sync(0xffffffffu, rescale) && t > it.t0) {
                    for (int c4 = 0; c4 < kWHalf / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld32p(tmem + lane_base + kWColO + c4 * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tmem + lane_base + kWColO + c4 * 32, o);
                    }
                }
                tmem_st32(tmem + lane_base + col_p, pk);
                tmem_st32(tmem + lane_base + col_p + 32, pk + 32);
                tmem_st_wait();
                tc_fence_before();
                arrive_lead(&p_full);
            }
            gchunk += static_cast<uint32_t>(C::kPeriod * T);
            // ---- epilogue
            if (T > 0) {
                mbar_wait(&o_done, (g - 1) & 1, wc);
                tc_fence_after();
            }
            const bool store = row < p.R && !aborted(wc);
            const int rr = row < p.R ? row : 0;
            const bool none = !(l > 0.f);   // no visible key in this range: O = 0, LSE = -inf
            const float inv_l = none ? 0.f : 1.f / l;
            const float lse_v = none ? -INFINITY : (m_run + __log2f(l)) * kLn2W;
            float amax = 0.f;
            __syncwarp();
            for (int c4 = 0; c4 < kWHalf / 32; ++c4) {
                uint32_t o[32];
                if (T > 0) {   // uniform over the CTA; a unit without keys (whole-unit order) gives O = 0
                    tmem_ld32p(tmem + lane_base + kWColO + c4 * 32, o);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (store) {
                    const int col = half * kWHalf + c4 * 32;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv_l;
                    if (it.whole) {
                        const size_t orow = static_cast<size_t>(hu) * p.R + rr;
                        if (p.o_stage) {
                            float4* dst = reinterpret_cast<float4*>(p.o_stage + orow * kWD + col);
#pragma unroll
                            for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        }
                        if (p.amax_bits) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                        }
                        if (p.nv_codes) {
                            // single-pass NVFP4: two 16-value blocks of this thread's row per chunk
                            const float sg = *p.nv_sg;
#pragma unroll
                            for (int b = 0; b < 2; ++b) {
                                uint32_t lo, hi;
                                const uint32_t sc = nvfp4_encode16(v + 16 * b, sg, lo, hi);
                                reinterpret_cast<uint2*>(p.nv_codes + orow * (kWD / 2) + col / 2)[b] = make_uint2(lo, hi);
                                p.nv_scales[orow * (kWD / 16) + col / 16 + b] = static_cast<uint8_t>(sc);
                            }
                        }
                        if (p.out) {
                            if (p.out_f32) {
                                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kWD + col);
#pragma unroll
                                for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                            } else {
                                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * kWD + col);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                                        pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                            }
                        }
                    } else {
                        // the workspace starts on a 256-byte boundary, so every 8-column group of a row is
                        // one aligned 32-byte sector
#pragma unroll
                        for (int i = 0; i < 4; ++i) st_global_v8(p.part_o + wpart_index(it.slot, row_in_tile, col + 8 * i), v + 8 * i);
                    }
                }
            }
            if (store && half == 0) {
                if (it.whole) {
                    if (p.lse) p.lse[static_cast<size_t>(hu) * p.R + rr] = lse_v;
                } else {
                    p.part_lse[static_cast<size_t>(it.slot) * kWRows + row_in_tile] = lse_v;
                }
            }
            if (store && it.whole && p.amax_bits && amax > 0.f) atomicMax(p.amax_bits, __float_as_uint(amax));
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) {
        cluster_sync();   // neither CTA frees Tensor Memory or exits while the other may still signal it
        if (warp == 5) tmem_dealloc_pair(tmem, 512);
    } else {
        if (warp == 5) tmem_dealloc(tmem, 512);
    }
}


// Exclusive prefix of per-unit 32-key tile counts (ragged keys), one block.
__global__ void __launch_bounds__(1024) wide_prefix_kernel(const int32_t* seqlens, int Hkv, int row_tiles, int U,
                                                          int32_t* prefix)
{
    griddep_launch_dependents();
    griddep_wait();
    __shared__ int part[1024];
    const int per = (U + 1023) / 1024;
    const int b0 = threadIdx.x * per;
    auto tiles = [&](int u) { return (seqlens[(u / row_tiles) / Hkv] + kWKeys - 1) / kWKeys; };
    int s = 0;
    for (int u = b0; u < min(U, b0 + per); ++u) s += tiles(u);
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
        run += tiles(u);
    }
    if (threadIdx.x == 1023) prefix[U] = part[1023];
}

// Merges split units (lse = log sum exp lse_i, O = sum exp(lse_i - lse) O_i) and writes units
// without keys (O = 0, LSE = -inf).  A block serves kCombCols of the 512 columns of one unit's 128
// query rows: warp 0 finds the pairs that hold partials of the unit once (64-bit divisions), then
// thread r merges row r, its LSE in registers and its kCombCols columns over the partials.  A warp's
// load of one 8-column group covers 32 consecutive rows, 1 KB of contiguous memory in the partial
// layout.  16 columns a block rather than 32 halve the registers that hold four partials' columns in
// flight, so twice the blocks are resident (B32 Hq128 Skv16384: step 199.6 -> 196.8 us).
constexpr int kMaxParts = 512;
constexpr int kCombCols = 16;
static_assert(kCombCols % 16 == 0, "the single-pass NVFP4 encoder takes whole 16-value blocks of a row");

__global__ void __launch_bounds__(kWRows) wide_combine_kernel(const __grid_constant__ WideParams p, int npairs)
{
    __shared__ int slots[kMaxParts];
    __shared__ int nslots;
    griddep_launch_dependents();
    // with uniform lengths the unit's partial slots follow from the parameters alone, so a block that
    // starts while the wide kernel still runs computes them before the wait; else after it (prefix)
    const bool params_only = !p.prefix && !p.seqlens;
    if (!params_only) griddep_wait();
    const int u = blockIdx.x / (kWD / kCombCols);
    const int col0 = (blockIdx.x % (kWD / kCombCols)) * kCombCols;
    const int r = static_cast<int>(threadIdx.x);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int hu = wunit_head(p, u);
    const int tiles = wunit_tiles(p, u);
    if (threadIdx.x < 32) {
        int cnt = 0;
        if (tiles > 0) {
            const long long Tu = wunit_start(p, u);
            const long long T = wsplit_total(p);
            const long long P = npairs;
            const int c0 = static_cast<int>(min((((Tu + 1) * P) - 1) / T, P - 1));
            const int c1 = static_cast<int>(min((((Tu + tiles) * P) - 1) / T, P - 1));
            if (c0 == c1) {
                cnt = -1;   // one pair held the whole unit and wrote it
            } else {
                for (int cw = c0; cw <= c1; cw += 32) {
                    const int c = cw + lane;
                    // pairs with an empty tile range (possible when T < P) hold no partial
                    const bool ok = c <= c1 && (c * T) / P != ((c + 1) * T) / P;
                    const unsigned m = __ballot_sync(0xffffffffu, ok);
                    if (ok) {
                        const int idx = cnt + __popc(m & ((1u << lane) - 1u));
                        if (idx < kMaxParts) slots[idx] = u + c;
                    }
                    cnt += __popc(m);
                }
                cnt = min(cnt, kMaxParts);
            }
        }
        if (lane == 0) nslots = cnt;
    }
    __syncthreads();
    if (params_only) griddep_wait();
    const int ns = nslots;
    if (ns < 0) return;   // the same for the whole block
    // rows beyond R (a partial row tile) compute on in-bounds workspace rows and store nothing,
    // so that every lane takes part in the warp reduction below
    const int row = (u % p.row_tiles) * kWRows + r;
    const bool live = row < p.R;
    // merged LSE of this row (partials without a visible key carry lse = -inf and weigh 0) and the
    // weighted sum of this row's 32 columns over the partials
    float acc[kCombCols];
#pragma unroll
    for (int k = 0; k < kCombCols; ++k) acc[k] = 0.f;
    float lse_v = -INFINITY;
    if (ns <= 4) {
        // the usual case (a unit cut by the stream-K split into at most four pieces): every partial LSE
        // and every partial column of this row in flight at once, one memory round trip
        float lv[4];
        float4 x[4][kCombCols / 4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const size_t sl = ns > 0 ? static_cast<size_t>(slots[i < ns ? i : 0]) : 0;   // a valid slot even when unused
            lv[i] = i < ns ? p.part_lse[sl * kWRows + r] : -INFINITY;
#pragma unroll
            for (int k = 0; k < kCombCols / 4; ++k)
                x[i][k] = i < ns ? *reinterpret_cast<const float4*>(p.part_o + wpart_index(sl, r, col0 + 4 * k))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float mx = fmaxf(fmaxf(lv[0], lv[1]), fmaxf(lv[2], lv[3]));
        if (mx > -INFINITY) {
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) sum += __expf(lv[i] - mx);   // exp(-inf) = 0 for the unused slots
            lse_v = mx + __logf(sum);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = __expf(lv[i] - lse_v);
#pragma unroll
                for (int k = 0; k < kCombCols / 4; ++k) {
                    acc[4 * k] = fmaf(w, x[i][k].x, acc[4 * k]);
                    acc[4 * k + 1] = fmaf(w, x[i][k].y, acc[4 * k + 1]);
                    acc[4 * k + 2] = fmaf(w, x[i][k].z, acc[4 * k + 2]);
                    acc[4 * k + 3] = fmaf(w, x[i][k].w, acc[4 * k + 3]);
                }
            }
        }
    } else {
        float mx = -INFINITY;
        for (int i = 0; i < ns; ++i) mx = fmaxf(mx, p.part_lse[static_cast<size_t>(slots[i]) * kWRows + r]);
        const bool any = mx > -INFINITY;
        float sum = 0.f;
        if (any)
            for (int i = 0; i < ns; ++i) sum += __expf(p.part_lse[static_cast<size_t>(slots[i]) * kWRows + r] - mx);
        lse_v = any ? mx + __logf(sum) : -INFINITY;
        for (int j = 0; j < ns && any; ++j) {
            const int sl = slots[j];
            const float w = __expf(p.part_lse[static_cast<size_t>(sl) * kWRows + r] - lse_v);
            float4 x[kCombCols / 4];
#pragma unroll
            for (int k = 0; k < kCombCols / 4; ++k) x[k] = *reinterpret_cast<const float4*>(p.part_o + wpart_index(sl, r, col0 + 4 * k));
#pragma unroll
            for (int k = 0; k < kCombCols / 4; ++k) {
                acc[4 * k] = fmaf(w, x[k].x, acc[4 * k]);
                acc[4 * k + 1] = fmaf(w, x[k].y, acc[4 * k + 1]);
                acc[4 * k + 2] = fmaf(w, x[k].z, acc[4 * k + 2]);
                acc[4 * k + 3] = fmaf(w, x[k].w, acc[4 * k + 3]);
            }
        }
    }
    const size_t orow = static_cast<size_t>(hu) * p.R + (live ? row : 0);
    if (live && p.o_stage) {
        float4* dst = reinterpret_cast<float4*>(p.o_stage + orow * kWD + col0);
#pragma unroll
        for (int k = 0; k < kCombCols / 4; ++k) dst[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    }
    if (live && p.out) {
        if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kWD + col0);
#pragma unroll
            for (int k = 0; k < kCombCols / 4; ++k) dst[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * kWD + col0);
#pragma unroll
            for (int k = 0; k < kCombCols / 8; ++k)
                dst[k] = make_uint4(pack_bf16x2(acc[8 * k], acc[8 * k + 1]), pack_bf16x2(acc[8 * k + 2], acc[8 * k + 3]),
                                    pack_bf16x2(acc[8 * k + 4], acc[8 * k + 5]), pack_bf16x2(acc[8 * k + 6], acc[8 * k + 7]));
        }
    }
    if (live && col0 == 0 && p.lse) p.lse[orow] = lse_v;
    if (live && p.nv_codes) {
        // single-pass NVFP4: the thread's columns are whole 16-value blocks of its row
        const float sg = *p.nv_sg;
#pragma unroll
        for (int b = 0; b < kCombCols / 16; ++b) {
            uint32_t lo, hi;
            const uint32_t sc = nvfp4_encode16(acc + 16 * b, sg, lo, hi);
            reinterpret_cast<uint2*>(p.nv_codes + orow * (kWD / 2) + col0 / 2)[b] = make_uint2(lo, hi);
            p.nv_scales[orow * (kWD / 16) + col0 / 16 + b] = static_cast<uint8_t>(sc);
        }
    }
    if (p.amax_bits) {
        float m = 0.f;
        if (live)
#pragma unroll
            for (int k = 0; k < kCombCols; ++k) m = fmaxf(m, fabsf(acc[k]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0 && m > 0.f) atomicMax(p.amax_bits, __float_as_uint(m));
    }
}

struct WideWs {
    size_t prefix_off, lse_off, o_off, stage_off, total;
};

// whole: no split (whole units per pair), which needs no prefix and no partials
WideWs wide_ws_layout(const AttnArgs& a, int npairs, bool whole)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int R = (a.Hq / a.Hkv) * a.Sq;
    const size_t U = static_cast<size_t>(a.B) * a.Hkv * ((R + kWRows - 1) / kWRows);
    const size_t slots = whole ? 0 : U + npairs;
    WideWs w{};
    size_t off = 0;
    w.prefix_off = off;
    off += (a.seqlens && !whole) ? al((U + 1) * 4) : 0;
    w.lse_off = off;
    off += al(slots * kWRows * 4);
    w.o_off = off;
    off += al(slots * kWRows * kWD * 4);
    w.stage_off = off;
    const bool stage = (a.out_kind == FMHA_OUT_NVFP4) && !a.out_f32 && !a.nv_sg;
    off += stage ? al(static_cast<size_t>(a.B) * a.Hq * a.Sq * kWD * 4) : 0;
    w.total = off;
    return w;
}

}  // namespace

size_t wide_workspace_bytes(const AttnArgs& a, int num_splits)
{
    const int nsm = num_sms() > 0 ? num_sms() : 256;
    return wide_ws_layout(a, nsm / 2, num_splits == 1).total;
}

namespace {

constexpr int kMaxWideDevices = 64;
std::atomic<int> g_pair_clusters[kMaxWideDevices];

// How many CTA pairs (clusters of two, one CTA per SM) the device runs at once; cached per device.
int pair_clusters(int nsm)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxWideDevices) return nsm / 2;
    int n = g_pair_clusters[dev].load();
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nsm & ~1), 1, 1);
    cfg.blockDim = dim3(kWThreads, 1, 1);
    cfg.dynamicSmemBytes = WCfg<true>::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, wide_kernel<true>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = nsm / 2;
    }
    n = min(n, nsm / 2);
    g_pair_clusters[dev].store(n);
    return n;
}

}  // namespace

int launch_wide(const AttnArgs& a, int num_splits, void* ws, size_t ws_bytes, cudaStream_t st)
{
    const int nsm = num_sms();
    if (nsm < 2) return set_error(FMHA_ERR_CUDA, "cannot query the SM count");
    const bool whole = num_splits == 1;
    const WideWs w = wide_ws_layout(a, nsm / 2, whole);
    if (w.total > 0 && (!ws || ws_bytes < w.total)) return set_error(FMHA_ERR_WORKSPACE, "wide-head path: workspace too small");
    uint8_t* base = static_cast<uint8_t*>(ws);
    const int Hq_per = a.Hq / a.Hkv;
    const int R = Hq_per * a.Sq;
    const int row_tiles = (R + kWRows - 1) / kWRows;
    const int heads = a.B * a.Hkv;
    // CTA-pair MMA variant: when asked for, and for dense keys only (the ragged tail's V rows are
    // cleared by each CTA in its own ring).  The default is the independent variant, which measured
    // faster on the wide-head decode workload (0.83 against 0.71 of the HBM copy bandwidth).
    const bool pair = !a.seqlens && a.wide_variant == FMHA_WIDE_PAIR;
    if (pair) FMHA_CHECK_CUDA(set_smem_limit_once(reinterpret_cast<const void*>(wide_kernel<true>), WCfg<true>::kSmem));
    const int max_pairs = pair ? pair_clusters(nsm) : nsm / 2;
    // whole units: no more pairs than units (each pair takes units p, p + P, ...); split with uniform
    // lengths: no more pairs than 32-key tiles, so that a small problem launches only pairs with work
    int npairs = whole ? min(max_pairs, heads * row_tiles) : max_pairs;
    if (!whole && !a.seqlens) {
        const long long tiles = static_cast<long long>(heads) * row_tiles * ((a.Skv + kWKeys - 1) / kWKeys);
        if (tiles < npairs) npairs = static_cast<int>(tiles);
    }
    CUtensorMap qmap, kmap, vmap;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(kWD), static_cast<uint64_t>(R), static_cast<uint64_t>(heads)};
        const uint64_t strides[2] = {static_cast<uint64_t>(kWD) * 2, static_cast<uint64_t>(R) * kWD * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(kWRows), 1};
        int rc = make_tmap_bf16(&qmap, a.q, 3, dims, strides, box);
        if (rc) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(kWD), static_cast<uint64_t>(a.Skv), static_cast<uint64_t>(heads)};
        const uint64_t strides[2] = {static_cast<uint64_t>(kWD) * 2, static_cast<uint64_t>(a.Skv) * kWD * 2};
        // K chunk: 64 columns x the tile's 128 keys, or x this CTA's 64 keys of the tile (pair MMA)
        const uint32_t kbox[3] = {64, static_cast<uint32_t>(pair ? WCfg<true>::kKRows : WCfg<false>::kKRows), 1};
        const uint32_t vbox[3] = {64, static_cast<uint32_t>(kWVKeys), 1};   // V chunk atom: 64 columns x 32 keys
        int rc = make_tmap_bf16(&kmap, a.k, 3, dims, strides, kbox);
        if (rc) return rc;
        rc = make_tmap_bf16(&vmap, a.v, 3, dims, strides, vbox);
        if (rc) return rc;
    }
    WideParams p{};
    p.U = heads * row_tiles;
    p.row_tiles = row_tiles;
    p.Hkv = a.Hkv;
    p.R = R;
    p.Skv = a.Skv;
    p.c = a.scale * kLog2eW;
    p.Sq = a.Sq > 0 ? a.Sq : 1;
    p.causal = a.causal;
    p.seqlens = a.seqlens;
    p.prefix = (a.seqlens && !whole) ? reinterpret_cast<const int32_t*>(base + w.prefix_off) : nullptr;
    p.tiles_uniform = (a.Skv + kWKeys - 1) / kWKeys;
    p.gap = (!whole && !a.seqlens && pair) ? kWSplitGapPair : 0;
    p.whole_units = whole ? 1 : 0;
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
    p.part_lse = whole ? nullptr : reinterpret_cast<float*>(base + w.lse_off);
    p.part_o = whole ? nullptr : reinterpret_cast<float*>(base + w.o_off);
    p.status = device_status_ptr();
    p.limit = wait_limit();
    if (p.prefix) {
        FMHA_CHECK_CUDA(launch_pdl(wide_prefix_kernel, dim3(1), dim3(1024), 0, st, a.seqlens, a.Hkv, row_tiles, p.U,
                                   const_cast<int32_t*>(p.prefix)));
        count_launch();
    }
    if (pair) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * npairs), 1, 1);
        cfg.blockDim = dim3(kWThreads, 1, 1);
        cfg.dynamicSmemBytes = WCfg<true>::kSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1 + pdl_attribute(st, &attr[1]);
        timing_mark_begin(st);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, wide_kernel<true>, qmap, kmap, vmap, p);
        timing_mark_end(st);
        if (e != cudaSuccess) return cuda_error(e, "wide_kernel<pair>");
    } else {
        FMHA_CHECK_CUDA(set_smem_limit_once(reinterpret_cast<const void*>(wide_kernel<false>), WCfg<false>::kSmem));
        timing_mark_begin(st);
        const cudaError_t e = launch_pdl(wide_kernel<false>, dim3(static_cast<unsigned>(2 * npairs)), dim3(kWThreads),
                                         WCfg<false>::kSmem, st, qmap, kmap, vmap, p);
        timing_mark_end(st);
        if (e != cudaSuccess) return cuda_error(e, "wide_kernel");
    }
    count_launch();
    if (whole) return FMHA_OK;   // every unit was written by its pair
    FMHA_CHECK_CUDA(launch_pdl(wide_combine_kernel, dim3(static_cast<unsigned>(p.U * (kWD / kCombCols))), dim3(kWRows),
                               0, st, p, npairs));
    count_launch();
    return FMHA_OK;
}

}  // namespace atc_gb300

