// fa_fwd1t_kernel.cuh -- attention forward with one 128-row Q tile per work unit,
// for head dimensions 64, 128 and 256 on sm_103a.
//
// Same method as fa_fwd_kernel.cuh (tiles of Q against K/V blocks, online softmax
// with a lazily moved reference max, P in tensor memory, O divided by l once;
// "ai6s.net/6af30f4d40858c2d8819b6d5" §2.2-§2.5), with one Q tile per unit and three
// S buffers for it instead of two Q tiles with one S buffer each. It serves
//   * d = 256, where two 128-row Q tiles would need 2 x 256 TMEM columns for O alone
//     and 128-key K/V tiles would be 64 KB each;
//   * row spaces of at most 128 rows (decode steps: the few queries of the heads of
//     one K/V head), where the two-tile kernel would run one tile and wait on its own
//     softmax between S(j) and S(j+1);
//   * small unsplit problems, whose 256-row units would fill at most half of the SMs.
// Layout:
//   * a unit is one 128-row Q tile (128 x D, 16-bit);
//   * K/V tiles hold bn(D) keys (128 for d <= 128, 64 at d = 256, where three
//     128-column S buffers and O would not fit the 512 TMEM columns); the K and V rings
//     are as deep as shared memory allows (3 and 2 at d = 256, 3 and 3 at d = 128,
//     6 and 6 at d = 64);
//   * S is formed in one of three bn(D)-column TMEM buffers (two at d = 256), so that
//     the softmax of block j runs while S(j+1) and S(j+2) are computed; O (D
//     columns) stays in TMEM for the unit. MMA order (three buffers):
//     ... O += P(j) V_j | S(j+3) | O += P(j+1) V_{j+1} ...
//   * at d = 256 the Q tile is also copied into TMEM (128 columns of 16-bit pairs) by
//     the softmax warpgroup, and S = Q K^T takes Q from there: with 64-key tiles the
//     shared-memory form would read 6 KB of operands per 32-cycle MMA, more than the
//     SM's 128 bytes per cycle of shared-memory bandwidth, while K alone is 2 KB;
//   * one softmax warpgroup (thread = query row = TMEM lane, bn(D) keys per block); on
//     blocks that every row sees whole, the row maximum comes from the reducing TMEM
//     load (fa_tmem_max.cuh).
// Start-up: the thread that initialises the barriers also requests the CTA's first
// unit's Q tile and first K tiles, and a launch whose grid covers every unit never
// touches the scheduler counters.
// When the reference max of a row moves (rare), the softmax thread rescales its O
// row, after waiting for the product O += P(j-1) V_{j-1} to complete (two
// alternating barriers, one per parity of j, so that a skipped wait never
// confuses phases: a product two blocks later cannot complete first).
//
// As in fa_fwd_kernel.cuh, query i stands at key position i + Nk - Nq (the last
// positions when Nq < Nk), the query heads of one K/V head share a row space when
// they have few queries each, and the keys may be cut into splits whose fp32 partial
// results fa_combine_kernel merges.
//
// Warps (256 threads): 0-3 softmax, 4 scheduler + Q and K producer, 5 MMA issuer,
// 6 V producer, 7 idle. Every wait is bounded; on expiry the CTA records the
// failure, drains its copies and MMAs, frees its tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_mask.cuh"
#include "fa_tmem_max.cuh"
#include "ptx.cuh"

namespace fa {
namespace onetile {

constexpr int kBM = 128;        // query rows per unit
// keys per K/V tile: 128 where three 128-column S buffers and O fit the 512 TMEM
// columns (D <= 128), else 64
__host__ __device__ constexpr int bn(int D) { return D == 256 ? 64 : 128; }
constexpr int kThreads = 256;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kVWarp = 6;
// K and V ring depths: what shared memory holds next to the Q tile (K/V tiles are
// bn(D) x D, 16-bit: 32 KB at d = 256 and 128, 16 KB at d = 64)
__host__ __device__ constexpr int k_stages(int D) { return D == 64 ? 6 : 3; }
__host__ __device__ constexpr int v_stages(int D) { return D == 64 ? 6 : D == 128 ? 3 : 2; }
constexpr int kMaxStages = 6;
constexpr int kSBufs = 3;  // S buffers (barrier slots); s_bufs(D) are used
__host__ __device__ constexpr int s_bufs(int D) { return D == 256 ? 2 : 3; }
// Q read by S = Q K^T from TMEM (d = 256) instead of shared memory
__host__ __device__ constexpr bool q_in_tmem(int D) { return D == 256; }
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units, as in fa_fwd_kernel.cuh
constexpr unsigned kStatusTimeout = 4;
constexpr int kUnitSlots = 2;
constexpr int kUnitConsumers = 6;  // warps 0-3, 5, 6 arrive once each per unit
enum : int { kRoleSoftmax = 1, kRoleTma = 2, kRoleMma = 3 };

struct Params {
    void *O;
    float *LSE;
    float *part_O;       // key split: fp32 partial O / l [split][b*H+h][Nq][d]; null: write O, LSE
    float *part_LSE;     // key split: partial log-sum-exps [split][b*H+h][Nq]
    int Nq, Nk;          // queries and keys per head
    int q_off;           // query i stands at key position i + q_off (Nk - Nq)
    int BH, kv_group;    // query heads B*H; query heads per K/V head
    int hps, R;          // query heads per row space (1, or kv_group when packed); rows hps*Nq
    int n_units, n_qb;   // (row space, 128-row block, key split) units; blocks per space
    int n_splits;        // key splits per block (1: none)
    int split_tiles;     // bn(D)-key K/V tiles per split
    int heavy_first;
    int wl, wr;          // key j visible to query i iff i + q_off - wl <= j <= i + q_off + wr
    float scale_log2;
    unsigned long long wait_budget_ns;
    unsigned int *status;
    unsigned int *sched; // this launch's {next unit, finished CTAs}
    int fault_skip_k;    // test hook: every CTA skips the K load at this ring position (-1: none)
    // Variable-length batches (kernel template flag VARLEN): row space sp = b*H + h
    // holds the queries of sequence b for query head h; the sequence's query tokens
    // are cu_q[b] .. cu_q[b+1]-1 and its keys cu_k[b] .. cu_k[b+1]-1 of token-major
    // tensors (tokens x heads x d), its queries at its last key positions. Offsets
    // are clamped to [0, total], so no stray value addresses memory outside the
    // tensors. Nq and R stand for the longest sequence's query count.
    const int *cu_q, *cu_k;
    int total_q, total_k;
    int H;
};

// Tiles are stored as regions of 64 columns (128 bytes, the 128-byte swizzle).
template <int D>
struct Smem {
    static_assert(D == 64 || D == 128 || D == 256, "head dimension");
    static constexpr int kRegions = D / 64;
    static constexpr int kQRegion = kBM * 128;   // 128 rows x 128 B (64 columns)
    static constexpr int kKVRegion = bn(D) * 128;  // bn(D) rows x 128 B
    static constexpr int kQBytes = kRegions * kQRegion;
    static constexpr int kKVBytes = kRegions * kKVRegion;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kQBytes;
    static constexpr int kV = kK + k_stages(D) * kKVBytes;
    static constexpr int kBar = kV + v_stages(D) * kKVBytes;
    static constexpr int kNumBars = 48;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kUnitRing = kMisc + 16;
    static constexpr int kBytes = kUnitRing + 16;
    // more than half of the SM's shared memory, so that one CTA (and one holder of
    // all 512 TMEM columns) runs per SM
    static constexpr int kAlloc = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
    static_assert(kAlloc <= 227 * 1024, "shared memory");
};

enum : int {
    kBarQFull = 0,
    kBarQEmpty = 1,
    kBarKFull = 2,                         // + stage
    kBarKEmpty = kBarKFull + kMaxStages,   // + stage
    kBarVFull = kBarKEmpty + kMaxStages,   // + stage
    kBarVEmpty = kBarVFull + kMaxStages,   // + stage
    kBarSFull = kBarVEmpty + kMaxStages,   // + buffer (3)
    kBarPFull = kBarSFull + kSBufs,        // + buffer (3)
    kBarPVDone = kBarPFull + kSBufs,       // + parity of the block (2)
    kBarODone = kBarPVDone + 2,
    kBarOFree = kBarODone + 1,
    kBarUnitFull = kBarOFree + 1,          // + slot (2)
    kBarUnitEmpty = kBarUnitFull + kUnitSlots,  // + slot (2)
    kBarDrainIdx = kBarUnitEmpty + kUnitSlots,
    kBarQReady = kBarDrainIdx + 1,         // Q copied into TMEM (d = 256)
    kNumBarsUsed = kBarQReady + 1,
};
static_assert(kNumBarsUsed <= Smem<256>::kNumBars, "barrier slots");
static_assert(k_stages(64) <= kMaxStages && v_stages(64) <= kMaxStages, "ring depth");

// TMEM columns: S buffers at bn(D) b, O after them (256 at d = 256, 384 below); at
// d = 256 the Q tile sits between them (columns 128 .. 255).
constexpr uint32_t kTmemS = 0;
__host__ __device__ constexpr uint32_t tmem_o(int D) { return D == 256 ? 256u : 384u; }
__host__ __device__ constexpr uint32_t tmem_q(int D) { return D == 256 ? 128u : 0u; }

// A row space holds the queries of hps consecutive query heads (b*H + h order), row
// r being query r % Nq of head sp*hps + r / Nq: one head each, or, with few queries,
// all heads of one K/V head, which then shares each K/V tile among them. In memory
// it is rows sp*R .. sp*R + R - 1 of the [B*H*Nq] row order of Q, O and LSE.
//
// A unit: rows r0 .. rl of row space sp, restricted to the K/V tiles of key split
// `split`; qmin .. qmax are the query indices among its rows; j0 .. j1 are the tiles
// holding a key some row sees (empty when j1 < j0, possible only with key splits).
//
// Variable-length batches: the unit also carries its sequence's sizes (nq queries,
// nk keys, query-key offset q_off), its first query and key tokens and its query and
// K/V heads; a block past the sequence's queries is empty.
struct Unit {
    int sp, bkv, r0, rl, qmin, qmax, j0, j1, split;
    int nq, nk, q_off, q_tok0, k_tok0, h, hkv;
};

template <int kBN, bool VARLEN>
__device__ __forceinline__ Unit decode(int u, const Params &p) {
    Unit U;
    const int per_sp = p.n_qb * p.n_splits;
    U.sp = u / per_sp;
    const int rem = u - U.sp * per_sp;
    int qb = rem / p.n_splits;
    U.split = rem - qb * p.n_splits;
    if (p.heavy_first) qb = p.n_qb - 1 - qb;
    U.r0 = qb * kBM;
    if constexpr (VARLEN) {
        const int b = U.sp / p.H;
        U.h = U.sp - b * p.H;
        U.hkv = U.h / p.kv_group;
        const int q0 = min(max(p.cu_q[b], 0), p.total_q);
        const int q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
        const int k0 = min(max(p.cu_k[b], 0), p.total_k);
        const int k1 = min(max(p.cu_k[b + 1], k0), p.total_k);
        U.q_tok0 = q0;
        U.k_tok0 = k0;
        U.nq = q1 - q0;
        U.nk = k1 - k0;
        U.q_off = U.nk - U.nq;
        U.bkv = 0;
        if (U.r0 >= U.nq) {  // past the sequence's queries: no work
            U.rl = U.r0;
            U.qmin = U.qmax = 0;
            U.j0 = 0;
            U.j1 = -1;
            return U;
        }
        U.rl = min(U.r0 + kBM, U.nq) - 1;
        U.qmin = U.r0;
        U.qmax = U.rl;
    } else {
        U.nq = p.Nq;
        U.nk = p.Nk;
        U.q_off = p.q_off;
        U.q_tok0 = U.k_tok0 = U.h = U.hkv = 0;
        U.bkv = U.sp * p.hps / p.kv_group;  // (b*H + h) / group = b*H_kv + h / group
        U.rl = min(U.r0 + kBM, p.R) - 1;
        // rows of one head: queries r0 % Nq .. rl % Nq; rows across a head boundary: all
        const bool one_head = U.r0 / p.Nq == U.rl / p.Nq;
        U.qmin = one_head ? U.r0 % p.Nq : 0;
        U.qmax = one_head ? U.rl % p.Nq : p.Nq - 1;
    }
    const int lo_key = max(0, U.qmin + U.q_off - p.wl);
    const int hi_key = min(U.nk - 1, U.qmax + U.q_off + p.wr);
    const int s_lo = U.split * p.split_tiles, s_hi = s_lo + p.split_tiles - 1;
    U.j0 = max(lo_key / kBN, s_lo);
    U.j1 = hi_key < 0 ? -1 : min(hi_key / kBN, s_hi);
    return U;
}

__device__ __forceinline__ void record_timeout(const Params &p, volatile int *abort_flag, int role,
                                               int unit) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0u, kStatusTimeout) == 0u) {
        p.status[1] = static_cast<unsigned>(role);
        p.status[2] = static_cast<unsigned>(unit);
        p.status[3] = blockIdx.x;
        __threadfence();
    }
}

// TMA coordinates of a unit's Q tile and of its K/V tile j: dense maps are
// (d, rows, row spaces), variable-length maps (d, heads, tokens).
template <bool VARLEN>
__device__ __forceinline__ void q_coords(const Unit &U, int &y, int &z) {
    if constexpr (VARLEN) {
        y = U.h;
        z = U.q_tok0 + U.r0;
    } else {
        y = U.r0;
        z = U.sp;
    }
}
template <bool VARLEN>
__device__ __forceinline__ void kv_coords(const Unit &U, int j, int bn, int &y, int &z) {
    if constexpr (VARLEN) {
        y = U.hkv;
        z = U.k_tok0 + j * bn;
    } else {
        y = j * bn;
        z = U.bkv;
    }
}

template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd1t_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = Smem<D>;
    constexpr int kBN = bn(D);
    constexpr uint32_t kTmemO = tmem_o(D);
    constexpr int kSB = s_bufs(D);
    constexpr bool kQT = q_in_tmem(D);
    constexpr uint32_t kTmemQ = tmem_q(D);
    static_assert(kSB <= kSBufs, "S buffers");
    static_assert(kQT ? (kSB * kBN <= static_cast<int>(kTmemQ) && kTmemQ + D / 2 <= kTmemO)
                      : kSB * kBN <= static_cast<int>(kTmemO),
                  "TMEM columns");
    static_assert(kTmemO + D <= kTmemCols, "TMEM columns");
    constexpr int kKStages = k_stages(D);
    constexpr int kVStages = v_stages(D);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::kQ;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::kUnitRing);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    auto sK = [sbase](int t) { return sbase + L::kK + (t % kKStages) * L::kKVBytes; };
    auto sV = [sbase](int t) { return sbase + L::kV + (t % kVStages) * L::kKVBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.wait_budget_ns;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    int pre_k = -1;  // K tiles of the first unit requested during setup (-1: none, nor Q)
    if (threadIdx.x == kTmaWarp * 32) {
        mbar_init(bar(kBarQFull), 1);
        // Q's shared-memory copy is released by the MMA warp's commit, or at d = 256
        // by the softmax threads once they have copied it into TMEM
        mbar_init(bar(kBarQEmpty), kQT ? 128 : 1);
        mbar_init(bar(kBarQReady), 128);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        for (int b = 0; b < kSB; ++b) {
            mbar_init(bar(kBarSFull + b), 1);
            mbar_init(bar(kBarPFull + b), 128);
        }
        mbar_init(bar(kBarPVDone + 0), 1);
        mbar_init(bar(kBarPVDone + 1), 1);
        mbar_init(bar(kBarODone), 1);
        mbar_init(bar(kBarOFree), 128);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(bar(kBarUnitFull + k), 1);
            mbar_init(bar(kBarUnitEmpty + k), kUnitConsumers);
        }
        mbar_init(bar(kBarDrainIdx), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        // The CTA's first unit is its own index (when it has work): its Q tile and
        // first K tiles are requested now, while the other warps still set up; the
        // producer loop below skips them.
        if (blockIdx.x < static_cast<unsigned>(p.n_units)) {
            const Unit W = decode<kBN, VARLEN>(static_cast<int>(blockIdx.x), p);
            if (W.j0 <= W.j1) {
                mbar_arrive_expect_tx(bar(kBarQFull), L::kQBytes);
                int qy, qz;
                q_coords<VARLEN>(W, qy, qz);
                for (int g = 0; g < L::kRegions; ++g)
                    tma_load_3d(sQ + g * L::kQRegion, &tmQ, bar(kBarQFull), 64 * g, qy, qz);
                pre_k = min(kKStages, W.j1 - W.j0 + 1);
                for (int x = 0; x < pre_k; ++x) {
                    if (x == p.fault_skip_k) continue;
                    int ky, kz;
                    kv_coords<VARLEN>(W, W.j0 + x, kBN, ky, kz);
                    mbar_arrive_expect_tx(bar(kBarKFull + x), L::kKVBytes);
                    for (int g = 0; g < L::kRegions; ++g)
                        tma_load_3d(sK(x) + g * L::kKVRegion, &tmK, bar(kBarKFull + x), 64 * g, ky, kz);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Take the next unit id from this role's ring slot (every role walks the same
    // sequence of units, published by the producer). Returns -1 at the end.
    auto take_unit = [&](int unit_iter, bool &ok) -> int {
        const int slot = unit_iter % kUnitSlots;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarUnitFull + slot),
                                                       (unit_iter / kUnitSlots) & 1, abort_flag, budget));
        if (!ok) return -1;
        const int u = unit_ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarUnitEmpty + slot));
        return u;
    };

    if (warp == kTmaWarp) {
        // ================================================================ scheduler, Q and K
        if (lane == 0) {
            int t = 0, unit_iter = 0, q_loads = 0;
            bool ok = true;
            auto publish = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kBarUnitEmpty + slot), ((k / kUnitSlots) & 1) ^ 1,
                                       abort_flag, budget);
                if (!ok) return -1;
                // units whose key split holds no key of theirs are skipped here; a
                // CTA's first unit is the one numbered like the CTA (no counter round
                // trip at start-up), the counter numbers the rest from gridDim.x on
                // (when the grid covers every unit, nothing is left to count)
                int v = -1;
                auto take_next = [&]() -> unsigned {
                    return static_cast<unsigned>(p.n_units) <= gridDim.x
                               ? static_cast<unsigned>(p.n_units)
                               : gridDim.x + atomicAdd(p.sched, 1u);
                };
                unsigned next = k == 0 ? blockIdx.x : take_next();
                for (;; next = take_next()) {
                    if (next >= static_cast<unsigned>(p.n_units)) break;
                    const Unit W = decode<kBN, VARLEN>(static_cast<int>(next), p);
                    if (W.j0 <= W.j1) {
                        v = static_cast<int>(next);
                        break;
                    }
                }
                unit_ring[slot] = v;
                mbar_arrive(bar(kBarUnitFull + slot));
                return v;
            };
            int u = publish(0);
            for (; ok && u >= 0; ++unit_iter) {
                const Unit U = decode<kBN, VARLEN>(u, p);
                const bool early = unit_iter == 0 && pre_k >= 0;  // Q and K(0 .. pre_k-1) in flight
                if (!early) {
                    ok = mbar_wait_bounded(bar(kBarQEmpty), (unit_iter & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kBarQFull), L::kQBytes);
                    int qy, qz;
                    q_coords<VARLEN>(U, qy, qz);
                    for (int g = 0; g < L::kRegions; ++g)
                        tma_load_3d(sQ + g * L::kQRegion, &tmQ, bar(kBarQFull), 64 * g, qy, qz);
                }
                ++q_loads;
                int u_next = -1;
                bool claimed = false;
                for (int j = U.j0; ok && j <= U.j1; ++j, ++t) {
                    if (!claimed && (j == U.j0 + 2 || j == U.j1)) {
                        claimed = true;
                        u_next = publish(unit_iter + 1);
                        if (!ok) break;
                        if (u_next >= 0) {
                            const Unit W = decode<kBN, VARLEN>(u_next, p);
                            int wy, wz;
                            q_coords<VARLEN>(W, wy, wz);
                            for (int g = 0; g < L::kRegions; ++g) tma_prefetch_l2_3d(&tmQ, 64 * g, wy, wz);
                        }
                    }
                    if (early && t < pre_k) continue;  // requested during setup
                    const int st = t % kKStages;
                    ok = mbar_wait_bounded(bar(kBarKEmpty + st), ((t / kKStages) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    if (t != p.fault_skip_k) {
                        int ky, kz;
                        kv_coords<VARLEN>(U, j, kBN, ky, kz);
                        mbar_arrive_expect_tx(bar(kBarKFull + st), L::kKVBytes);
                        for (int g = 0; g < L::kRegions; ++g)
                            tma_load_3d(sK(t) + g * L::kKVRegion, &tmK, bar(kBarKFull + st),
                                        64 * g, ky, kz);
                    }
                }
                if (!claimed && ok) u_next = publish(unit_iter + 1);
                u = u_next;
            }
            if (!ok) record_timeout(p, abort_flag, kRoleTma, u);
            if (q_loads > 0) mbar_wait_bounded(bar(kBarQFull), (q_loads - 1) & 1, nullptr, budget);
            for (int s = 0; s < kKStages; ++s)
                if (t > s) {
                    const int last = t - 1 - ((t - 1 - s) % kKStages);
                    mbar_wait_bounded(bar(kBarKFull + s), (last / kKStages) & 1, nullptr, budget);
                }
        }
    } else if (warp == kVWarp) {
        // ================================================================ V producer
        int t = 0;
        bool ok = true;
        for (int unit_iter = 0; ok; ++unit_iter) {
            const int u = take_unit(unit_iter, ok);
            if (!ok || u < 0) break;
            const Unit U = decode<kBN, VARLEN>(u, p);
            if (lane == 0) {
                for (int j = U.j0; ok && j <= U.j1; ++j, ++t) {
                    const int st = t % kVStages;
                    ok = mbar_wait_bounded(bar(kBarVEmpty + st), ((t / kVStages) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    int vy, vz;
                    kv_coords<VARLEN>(U, j, kBN, vy, vz);
                    mbar_arrive_expect_tx(bar(kBarVFull + st), L::kKVBytes);
                    for (int g = 0; g < L::kRegions; ++g)
                        tma_load_3d(sV(t) + g * L::kKVRegion, &tmV, bar(kBarVFull + st), 64 * g,
                                    vy, vz);
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            t = __shfl_sync(0xffffffffu, t, 0);
        }
        if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleTma, -1);
        if (lane == 0)
            for (int s = 0; s < kVStages; ++s)
                if (t > s) {
                    const int last = t - 1 - ((t - 1 - s) % kVStages);
                    mbar_wait_bounded(bar(kBarVFull + s), (last / kVStages) & 1, nullptr, budget);
                }
    } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc_s = idesc_f16_ab(BF16, kBM, kBN, false, false);
        constexpr uint32_t idesc_o = idesc_f16_ab(BF16, kBM, D, false, true);
        auto wait = [&](int b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag, budget));
        };
        auto commit = [&](int b) {
            if (elect_one()) umma_commit(bar(b));
            __syncwarp();
        };
        // S(t) = Q K_t^T into S buffer t mod kSB (kBN columns); Q from shared memory,
        // or from TMEM (K-step k of 16 columns = 8 TMEM columns).
        auto issue_s = [&](int t) {
            tc_fence_after();
            const uint64_t dq = sw128_desc(sQ, 16, 1024);
            const uint64_t dk = sw128_desc(sK(t), 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t offq = (k >> 2) * (L::kQRegion >> 4) + (k & 3) * 2;
                    const uint32_t offk = (k >> 2) * (L::kKVRegion >> 4) + (k & 3) * 2;
                    if constexpr (kQT)
                        umma_f16_ts(tmem + kTmemS + (t % kSB) * kBN, tmem + kTmemQ + k * 8, dk + offk,
                                    idesc_s, k > 0 ? 1u : 0u);
                    else
                        umma_f16_ss(tmem + kTmemS + (t % kSB) * kBN, dq + offq, dk + offk, idesc_s,
                                    k > 0 ? 1u : 0u);
                }
                umma_commit(bar(kBarSFull + t % kSB));
            }
            __syncwarp();
        };
        // O (+)= P(t) V_t, P read from the first kBN / 2 columns of S buffer t mod kSB.
        auto issue_pv = [&](int t, bool first) {
            tc_fence_after();
            const uint64_t dv = sw128_desc(sV(t), L::kKVRegion, 1024);
            const uint32_t acc0 = first ? 0u : 1u;
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    umma_f16_ts(tmem + kTmemO, tmem + kTmemS + (t % kSB) * kBN + k * 8,
                                dv + k * ((16 * 128) >> 4), idesc_o, k > 0 ? 1u : acc0);
                umma_commit(bar(kBarPVDone + (t & 1)));
            }
            __syncwarp();
        };
        int t = 0;  // K/V blocks issued so far over all units
        bool ok = true;
        int unit_iter = 0, u = -1;
        for (; ok; ++unit_iter) {
            u = take_unit(unit_iter, ok);
            if (!ok || u < 0) break;
            const Unit U = decode<kBN, VARLEN>(u, p);
            const int n = U.j1 - U.j0 + 1;
            ok = wait(kQT ? kBarQReady : kBarQFull, unit_iter & 1);
            // S for the first min(kSB, n) blocks
            for (int x = 0; ok && x < n && x < kSB; ++x) {
                ok = wait(kBarKFull + (t + x) % kKStages, ((t + x) / kKStages) & 1);
                if (ok) {
                    issue_s(t + x);
                    commit(kBarKEmpty + (t + x) % kKStages);  // K is read by S only
                }
            }
            for (int x = 0; ok && x < n; ++x, ++t) {
                ok = wait(kBarPFull + t % kSB, (t / kSB) & 1) &&
                     wait(kBarVFull + t % kVStages, (t / kVStages) & 1);
                if (ok && x == 0 && unit_iter > 0) ok = wait(kBarOFree, (unit_iter - 1) & 1);
                if (!ok) break;
                issue_pv(t, x == 0);
                commit(kBarVEmpty + t % kVStages);
                if (x + kSB < n) {
                    ok = wait(kBarKFull + (t + kSB) % kKStages, ((t + kSB) / kKStages) & 1);
                    if (!ok) break;
                    issue_s(t + kSB);  // reuses buffer t mod kSB after O += P(t) V_t
                    commit(kBarKEmpty + (t + kSB) % kKStages);
                }
            }
            if (!ok) break;
            if constexpr (!kQT) commit(kBarQEmpty);
            commit(kBarODone);
        }
        if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleMma, u);
        if (elect_one()) umma_commit(bar(kBarDrainIdx));
        __syncwarp();
        if (lane == 0) mbar_wait_bounded(bar(kBarDrainIdx), 0, nullptr, budget);
        __syncwarp();
    } else if (warp < 4) {
        // ================================================================ softmax warpgroup
        const int row = threadIdx.x & 127;
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        // d = 256: copy the k-th unit's Q tile from shared memory into TMEM, this
        // thread's row into its lane (128-byte swizzle: 16-byte chunk c of row r sits
        // at chunk c ^ (r mod 8) of the row), then release both copies' barriers.
        auto copy_q = [&](int k) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarQFull), k & 1, abort_flag, budget)))
                return false;
#pragma unroll
            for (int g = 0; g < L::kRegions; ++g) {
                uint32_t w[32];
                const uint8_t *src = smem + L::kQ + g * L::kQRegion + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src + ((c ^ (row & 7)) << 4));
                    w[4 * c] = v.x;
                    w[4 * c + 1] = v.y;
                    w[4 * c + 2] = v.z;
                    w[4 * c + 3] = v.w;
                }
                tmem_st32(tl + kTmemQ + g * 32, w);
            }
            tmem_st_wait();
            mbar_arrive(bar(kBarQEmpty));
            tc_fence_before();
            mbar_arrive(bar(kBarQReady));
            return true;
        };
        int t = 0;
        bool ok = true;
        int unit_iter = 0, u = -1, u_next = -1;
        for (; ok; ++unit_iter) {
            if (kQT && unit_iter > 0) {
                u = u_next;  // taken, and its Q copied, before the previous unit's epilogue
            } else {
                u = take_unit(unit_iter, ok);
                if (ok && kQT && u >= 0) ok = copy_q(unit_iter);
            }
            if (!ok || u < 0) break;
            const Unit U = decode<kBN, VARLEN>(u, p);
            const int r = U.r0 + row;  // row of the space
            const int i = VARLEN ? r : r % p.Nq;  // its query index; key position i + q_off
            const int lo_i = max(0, i + U.q_off - p.wl);
            const int hi_i = min(U.nk - 1, i + U.q_off + p.wr);
            // a tile with keys in [lo_last, hi_first] only is visible to every row
            const int lo_last = max(0, U.qmax + U.q_off - p.wl);
            const int hi_first = min(U.nk - 1, U.qmin + U.q_off + p.wr);
            float m = -INFINITY, l = 0.f;
            for (int j = U.j0; j <= U.j1; ++j, ++t) {
                const uint32_t tS = tl + kTmemS + (t % kSB) * kBN;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarSFull + t % kSB), (t / kSB) & 1,
                                                               abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                float x[kBN];
                const int kv0 = j * kBN;
                float m_tile;
                if (kv0 >= lo_last && kv0 + kBN - 1 <= hi_first) {
                    // every key visible: the TMEM loads reduce each 32-column run to
                    // its maximum
                    float mr[kBN / 32];
#pragma unroll
                    for (int h = 0; h < kBN; h += 64) {
                        uint32_t a[32], b[32];
                        tmem_ld32_max(tS + h, a, mr[h / 32]);
                        tmem_ld32_max(tS + h + 32, b, mr[h / 32 + 1]);
                        tmem_ld_max_wait(a, mr[h / 32]);
                        tmem_ld_max_wait(b, mr[h / 32 + 1]);
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            x[h + c] = __uint_as_float(a[c]);
                            x[h + c + 32] = __uint_as_float(b[c]);
                        }
                    }
                    float mm = mr[0];
#pragma unroll
                    for (int c = 1; c < kBN / 32; ++c) mm = fmaxf(mm, mr[c]);
                    m_tile = mm * sl2;
                } else {
#pragma unroll
                    for (int h = 0; h < kBN; h += 64) {
                        uint32_t a[32], b[32];
                        tmem_ld32(tS + h, a);
                        tmem_ld32(tS + h + 32, b);
                        tmem_ld_wait(a);
                        tmem_ld_wait(b);
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            x[h + c] = __uint_as_float(a[c]);
                            x[h + c + 32] = __uint_as_float(b[c]);
                        }
                    }
                    mask_outside_run(x, lo_i - kv0, hi_i - kv0, -INFINITY);
                    float ma = fmaxf(x[0], x[1]), mb = fmaxf(x[2], x[3]);
#pragma unroll
                    for (int c = 4; c < kBN; c += 4) {
                        ma = max3f(ma, x[c], x[c + 1]);
                        mb = max3f(mb, x[c + 2], x[c + 3]);
                    }
                    m_tile = fmaxf(ma, mb) * sl2;
                }
                const float m_old = m;
                if (m_tile > m + kRescaleThreshold) m = m_tile;
                const float corr = m != m_old ? ex2_approx(m_old - m) : 1.f;
                const float nm = m == -INFINITY ? 0.f : -m;
                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                for (int c = 0; c < kBN; c += 2) {
                    ffma2(x[c], x[c + 1], sl2, sl2, nm, nm);
                    x[c] = ex2_approx(x[c]);
                    x[c + 1] = ex2_approx(x[c + 1]);
                }
#pragma unroll
                for (int c = 0; c < kBN; c += 4) {
                    fadd2(s0, s1, x[c], x[c + 1]);
                    fadd2(s2, s3, x[c + 2], x[c + 3]);
                }
                // P(j) as 16-bit pairs over the first kBN / 2 columns of the buffer
#pragma unroll
                for (int h = 0; h < kBN; h += 64) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = pack2<BF16>(x[h + 2 * e], x[h + 2 * e + 1]);
                    tmem_st16(tS + h / 2, pk);
                    tmem_st16(tS + h / 2 + 16, pk + 16);
                }
                l = l * corr + ((s0 + s1) + (s2 + s3));
                // The reference max moved: O holds the sum through block j-1 once that
                // product completes; rescale this row's O before P(j) is released.
                if (j > U.j0 && __any_sync(0xffffffffu, corr != 1.f)) {
                    const int tp = t - 1;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarPVDone + (tp & 1)), (tp >> 1) & 1,
                                                                   abort_flag, budget));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tl + kTmemO + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0 = __uint_as_float(o[e]), a1 = __uint_as_float(o[e + 1]);
                            fmul2(a0, a1, corr, corr);
                            o[e] = __float_as_uint(a0);
                            o[e + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(tl + kTmemO + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + t % kSB));
            }
            if (!ok) break;
            if constexpr (kQT) {
                // every S of this unit has completed (its last S buffer was read), so
                // the next unit's Q can replace this one's in TMEM during the epilogue
                u_next = take_unit(unit_iter + 1, ok);
                if (ok && u_next >= 0) ok = copy_q(unit_iter + 1);
                if (!ok) break;
            }
            // ---- epilogue: O / l rounded to 16 bit, LSE = ln 2 (m + log2 l)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarODone), unit_iter & 1, abort_flag, budget));
            if (!ok) break;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            // global row of O and LSE: (row space, row), or (token, head) when VARLEN
            const bool store = r < (VARLEN ? U.nq : p.R);
            const size_t grow = VARLEN ? (static_cast<size_t>(U.q_tok0) + (store ? r : 0)) * p.H + U.h
                                       : static_cast<size_t>(U.sp) * p.R + (store ? r : 0);
            const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            if (p.part_O == nullptr) {
                uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) + grow * (D * 2);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl + kTmemO + c * 32, o);
                    tmem_ld_wait(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
                    if (store) {
                        st_global_v8(orow + c * 64, pk);
                        st_global_v8(orow + c * 64 + 32, pk + 8);
                    }
                }
                if (store) p.LSE[grow] = lse;
            } else {
                // key split: the split's own O / l in fp32 and its LSE, merged later
                const size_t prow = static_cast<size_t>(U.split) * p.BH * p.Nq + grow;
                float *orow = p.part_O + prow * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl + kTmemO + c * 32, o);
                    tmem_ld_wait(o);
                    if (store) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
#pragma unroll
                        for (int q = 0; q < 4; ++q) st_global_v8(orow + c * 32 + q * 8, o + q * 8);
                    }
                }
                if (store) p.part_LSE[prow] = lse;
            }
            tc_fence_before();
            mbar_arrive(bar(kBarOFree));
        }
        if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleSoftmax, u);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The last CTA to finish zeroes this launch's scheduler counters (untouched when
    // the grid covered every unit).
    if (threadIdx.x == 0 && static_cast<unsigned>(p.n_units) > gridDim.x) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

}  // namespace onetile
}  // namespace fa
