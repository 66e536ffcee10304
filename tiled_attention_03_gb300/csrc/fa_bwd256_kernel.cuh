// fa_bwd256_kernel.cuh -- attention backward at head dimension 256 on sm_103a.
//
// Same method as fa_bwd_kernel.cuh: the scores and probabilities are recomputed
// block by block from the forward's saved row statistics instead of storing P
// ("ai6s.net/6af30f4d40858c2d8819b6d5" §2.4). With L_i = LSE_i log2(e) and
// D_i = sum_c dO_ic O_ic (both from the prep kernel of fa_bwd_kernel.cuh):
//     P_ij = 2^(s_ij scale log2(e) - L_i)      dP_ij = dO_i . V_j
//     dS_ij = P_ij (dP_ij - D_i)
//     dQ_i = scale sum_j dS_ij K_j    dK_j = scale sum_i dS_ij Q_i    dV_j = sum_i P_ij dO_i
//
// Why a kernel of its own. At d = 256 a 128 x 256 16-bit tile is 64 KB and a
// 128 x 256 fp32 accumulator takes 256 of the SM's 512 tensor-memory columns, so
// the d <= 128 layout (K_j, V_j, Q_i and dO_i tiles in shared memory, dK_j and dV_j
// both in TMEM) would need 256 KB and 768 columns. Here each gradient has its own
// pass. A pass keeps the 128 rows it accumulates for (its "resident" tiles) on the
// SM and streams the other side in tiles of 64 rows:
//   dQ pass: rows = 128 queries; Q_i, dO_i, L_i, D_i resident; K_j, V_j streamed.
//            X = Q_i K_j^T, Y = dO_i V_j^T, A = P (Y - D), dQ_i += A K_j.
//   dK pass: rows = 128 keys; K_j, V_j resident; Q_i (+ L), dO_i (+ D) streamed.
//            X = K_j Q_i^T, Y = V_j dO_i^T, A = P^T (Y - D), dK_j += A Q_i.
//   dV pass: rows = 128 keys; K_j resident; Q_i (+ L), dO_i streamed.
//            X = K_j Q_i^T, A = P^T, dV_j += A dO_i.
// X and Y are M = 128, N = 64, K = 256 products (K-major operands). X takes its
// resident operand from TMEM, where the compute warps load the first resident tile
// (each thread its row, from global memory) before each unit: from shared memory,
// both operands of an N = 64 product are 6 KB per 32-cycle MMA, more than the SM's
// 128 bytes per cycle of shared-memory bandwidth, and the 64 KB the tile no longer
// takes there deepen the streamed rings. Y reads both operands from shared memory
// (TMEM has no room for the second resident tile). A is written by the compute warps
// as 16-bit pairs into TMEM (over Y's columns, or over X's in the dV pass) and the
// accumulation is an M = 128, N = 256, K = 64 product with A from TMEM and B (the
// streamed tile, 64 rows of 256 columns) MN-major. The scores are
// recomputed once per pass (S three times in all, against twice in the d <= 128
// kernels), the price of fitting one SM.
//
// Warps (192 threads): 0-3 compute (thread = resident row = TMEM lane), 4 TMA
// producer and scheduler, 5 MMA issuer. Units come from a launch-wide counter (a
// CTA's first unit is its own index). Every wait is bounded (global-timer budget);
// on expiry the CTA records the failure in the status word, drains its copies and
// MMAs, frees its tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_mask.cuh"
#include "ptx.cuh"

namespace fa {
namespace bwd256 {

constexpr int kD = 256;
constexpr int kRows = 128;    // resident rows (TMEM lanes)
constexpr int kCols = 64;     // rows of a streamed tile = columns of X and Y
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned kStatusTimeout = 4;  // FA_ERR_TIMEOUT
enum : int { kRoleCompute = 1, kRoleTma = 2, kRoleMma = 3 };
enum : int { kPassDQ = 0, kPassDK = 1, kPassDV = 2 };

// 16-bit tiles are stored as regions of 64 columns (128 bytes per row, the 128-byte
// swizzle TMA writes): 4 regions per 256-column row.
constexpr int kRegions = kD / 64;
constexpr int kResRegion = kRows * 128;  // 16 KB
constexpr int kStrRegion = kCols * 128;  // 8 KB
constexpr int kResBytes = kRegions * kResRegion;  // 64 KB
constexpr int kStrBytes = kRegions * kStrRegion;  // 32 KB

// TMEM columns: X (fp32, 64), then A (16-bit pairs) over its first 32; Y (fp32, 64);
// the first resident tile (16-bit pairs, 128); the accumulator (fp32, 256). The dV
// pass has no Y and alternates X between columns 0 and 64, so that X(t+1) is formed
// while the compute warps turn X(t) into A(t).
constexpr uint32_t kTmemX = 0;
constexpr uint32_t kTmemY = 64;
constexpr uint32_t kTmemR0 = 128;
constexpr uint32_t kTmemAcc = 256;

template <int PASS>
struct Layout {
    // The second resident tile (dO_i in the dQ pass, V_j in the dK pass), the one
    // kept in shared memory (the first lives in TMEM).
    static constexpr bool kRes1 = PASS != kPassDV;
    // Ring depths of the two streamed tiles: s0 (K_j in the dQ pass, Q_i in the
    // others) and s1 (V_j, or dO_i), as deep as shared memory allows.
    static constexpr int kS0 = PASS == kPassDV ? 4 : 3;
    static constexpr int kS1 = PASS == kPassDV ? 3 : 2;
    static constexpr int kRes1Off = 0;
    static constexpr int kStr0 = kRes1Off + (kRes1 ? kResBytes : 0);
    static constexpr int kStr1 = kStr0 + kS0 * kStrBytes;
    static constexpr int kVec = kStr1 + kS1 * kStrBytes;  // dQ: L_i, D_i (2 x 128); else L, D rings
    // ring of the streamed tiles' row-term vectors (L, and D in the dK pass), as
    // deep as the s0 ring (see the producer)
    static constexpr int kVecSlots = kS0;
    static constexpr int kVecBytes =
        PASS == kPassDQ ? 2 * kRows * 4 : (PASS == kPassDK ? 2 : 1) * kVecSlots * kCols * 4;
    static constexpr int kBar = kVec + kVecBytes;
    static constexpr int kNumBars = 32;
    static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, abort flag, unit ring
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;       // slack to align the base to 1024 B
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

enum : int {
    kBarResFull = 0,
    kBarResEmpty = 1,
    kBarS0Full = 2,                  // + slot (<= 4)
    kBarS0Empty = kBarS0Full + 4,    // + slot
    kBarS1Full = kBarS0Empty + 4,    // + slot (<= 3)
    kBarS1Empty = kBarS1Full + 3,    // + slot
    kBarXFull = kBarS1Empty + 3,     // + X buffer (2)
    kBarYFull = kBarXFull + 2,
    kBarAReady = kBarYFull + 1,      // + X buffer (2)
    kBarAccDone = kBarAReady + 2,
    kBarAccFree = kBarAccDone + 1,
    kBarUnitFull = kBarAccFree + 1,  // + slot (2)
    kBarUnitEmpty = kBarUnitFull + 2,
    kBarDrain = kBarUnitEmpty + 2,
    kBarR0Ready = kBarDrain + 1,     // first resident tile copied into TMEM
    kBarXRead = kBarR0Ready + 1,     // dQ / dK passes: the compute warps have loaded X
    kNumBarsUsed = kBarXRead + 1,
};
static_assert(kNumBarsUsed <= Layout<0>::kNumBars, "barrier slots");
constexpr int kUnitSlots = 2;
constexpr int kUnitConsumers = 5;  // the MMA warp and the 4 compute warps

struct Params {
    void *out;                // dQ (B*H x N x 256), dK or dV (B*H_kv x N x 256), 16-bit
    const float *Lw, *Dw;     // B*H x Npad row terms (prep kernel)
    int N, Npad;              // queries = keys per head; N rounded up to 128
    int H, Hkv, group;        // query heads, K/V heads, H / H_kv
    int n_blk;                // 128-row blocks per head
    int n_units;
    int wl, wr;               // key j visible to query i iff i - wl <= j <= i + wr
    float scale_log2, out_scale;
    unsigned long long wait_budget_ns;
    unsigned int *status;     // [code, role, unit, block]
    unsigned int *sched;      // this launch's {next unit, finished CTAs} (zero at launch)
    int fault_unit;           // test hook: every CTA skips its resident load of this unit (-1: none)
    // Variable-length batches (template flag VARLEN): token-major tensors, sequence b
    // owning query tokens cu_q[b] .. cu_q[b+1]-1 and keys cu_k[b] .. cu_k[b+1]-1
    // (clamped to [0, total]), its queries at its last key positions; the row terms
    // of sequence b, head h start at h * vstride + cu_pad[b]; n_blk counts 128-row
    // blocks of the longest sequence's resident side.
    const int *cu_q, *cu_k, *cu_pad;
    const void *res0;         // the first resident tile's tensor: Q (dQ pass) or K
    int total_q, total_k, vstride;
};

// A unit: 128 resident rows r0 .. r0+127 of head `head` (a query head in the dQ
// pass, a K/V head in the others) and the streamed tiles t = 0 .. n_t-1 that hold a
// visible pair: tile t is 64-row block lo + t % per of head `head` (dQ pass), or of
// query head group_head(head, t / per) (dK / dV passes).
// Positions are the sequence's own (queries 0 .. nq-1 at key positions q_off ..
// q_off + nq - 1, keys 0 .. nk-1); the dense case is one sequence of N per head.
// n_t = 0 marks a unit without work (rows past its sequence, or no visible pair).
struct Unit {
    int head, r0, lo, per, n_t;
    int nq, nk, q_off, q_tok0, k_tok0, pad0;
};

template <int PASS, bool VARLEN>
__device__ __forceinline__ Unit decode(int u, const Params &p) {
    Unit U;
    U.head = u / p.n_blk;
    U.r0 = (u - U.head * p.n_blk) * kRows;
    if constexpr (VARLEN) {
        const int b = U.head / (PASS == kPassDQ ? p.H : p.Hkv);
        const int q0 = min(max(p.cu_q[b], 0), p.total_q);
        const int q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
        const int k0 = min(max(p.cu_k[b], 0), p.total_k);
        const int k1 = min(max(p.cu_k[b + 1], k0), p.total_k);
        U.nq = q1 - q0;
        U.nk = k1 - k0;
        U.q_tok0 = q0;
        U.k_tok0 = k0;
        U.pad0 = p.cu_pad[b];
    } else {
        U.nq = U.nk = p.N;
        U.q_tok0 = U.k_tok0 = U.pad0 = 0;
    }
    U.q_off = U.nk - U.nq;
    // dQ: resident rows are queries, streamed rows keys; dK / dV: the other way round.
    const int n_res = PASS == kPassDQ ? U.nq : U.nk;
    const int n_str = PASS == kPassDQ ? U.nk : U.nq;
    const int r1 = min(U.r0 + kRows, n_res) - 1;
    const int lo = PASS == kPassDQ ? max(0, U.r0 + U.q_off - p.wl) : max(0, U.r0 - U.q_off - p.wr);
    const int hi = PASS == kPassDQ ? min(n_str - 1, r1 + U.q_off + p.wr)
                                   : min(n_str - 1, r1 - U.q_off + p.wl);
    U.lo = lo / kCols;
    U.per = hi / kCols - U.lo + 1;
    U.n_t = U.r0 < n_res && lo <= hi ? (PASS == kPassDQ ? 1 : p.group) * U.per : 0;
    return U;
}

// Head of the streamed tile t: the unit's own (dQ pass), or the query head of the
// group reading K/V head `head` (dK / dV passes). Heads are b * H + h (queries) or
// b * H_kv + h (K/V).
template <int PASS>
__device__ __forceinline__ void tile_of(const Unit &U, int t, const Params &p, int &head, int &row0) {
    const int g = t / U.per;
    row0 = (U.lo + (t - g * U.per)) * kCols;
    if constexpr (PASS == kPassDQ) {
        head = U.head / p.H * p.Hkv + (U.head % p.H) / p.group;  // K/V head of query head U.head
    } else {
        const int b = U.head / p.Hkv, hk = U.head - b * p.Hkv;
        head = b * p.H + hk * p.group + g;
    }
}

// TMA coordinates (y, z) of a tile starting at row `row` of head `head` of a tensor
// with `heads` heads per batch entry whose sequence starts at token tok0: dense
// maps are (d, N, heads), variable-length maps (d, heads, tokens).
template <bool VARLEN>
__device__ __forceinline__ void coords(int head, int heads, int tok0, int row, int &y, int &z) {
    if constexpr (VARLEN) {
        y = head % heads;
        z = tok0 + row;
    } else {
        y = row;
        z = head;
    }
}

// Row of the row-term vectors for query row `row` of query head `head`.
template <bool VARLEN>
__device__ __forceinline__ size_t vec_row(const Unit &U, int head, int row, const Params &p) {
    if constexpr (VARLEN)
        return static_cast<size_t>(head % p.H) * p.vstride + U.pad0 + row;
    else
        return static_cast<size_t>(head) * p.Npad + row;
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

// The resident tiles are read through a 128-row TMA map of their tensor, the
// streamed ones through a 64-row map: tmR0 / tmR1 (Q / dO in the dQ pass, K / V
// otherwise) and tmS0 / tmS1 (K / V in the dQ pass, Q / dO otherwise). The first
// resident tile is read by the compute warps from p.res0; tmR0 serves its L2
// prefetch.
template <int PASS, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd256_kernel(const __grid_constant__ CUtensorMap tmR0, const __grid_constant__ CUtensorMap tmR1,
                     const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                     const Params p) {
    using L = Layout<PASS>;
    constexpr int kS0 = L::kS0, kS1 = L::kS1, kVecSlots = L::kVecSlots;
    constexpr bool kHasY = PASS != kPassDV;
    constexpr int kXBufs = kHasY ? 1 : 2;  // X buffers: tile it uses it % kXBufs
    auto xcol = [](int it) { return kTmemX + static_cast<uint32_t>((it % kXBufs) * 64); };
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sR1 = sbase + L::kRes1Off;
    auto sS0 = [sbase](int it) { return sbase + L::kStr0 + (it % kS0) * kStrBytes; };
    auto sS1 = [sbase](int it) { return sbase + L::kStr1 + (it % kS1) * kStrBytes; };
    // row-term vectors: dQ pass L_i, D_i (128 each); dK / dV passes the L (and D) of
    // each streamed tile's 64 rows in a ring of kVecSlots
    float *vec = reinterpret_cast<float *>(smem + L::kVec);
    const uint32_t sVec = sbase + L::kVec;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::kMisc + 8);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.wait_budget_ns;

    // ---- setup
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == kTmaWarp * 32) {
        mbar_init(bar(kBarResFull), 1);
        mbar_init(bar(kBarResEmpty), 1);
        for (int s = 0; s < kS0; ++s) {
            mbar_init(bar(kBarS0Full + s), 1);
            mbar_init(bar(kBarS0Empty + s), 1);
        }
        for (int s = 0; s < kS1; ++s) {
            mbar_init(bar(kBarS1Full + s), 1);
            mbar_init(bar(kBarS1Empty + s), 1);
        }
        for (int b = 0; b < kXBufs; ++b) {
            mbar_init(bar(kBarXFull + b), 1);
            mbar_init(bar(kBarAReady + b), 128);
        }
        mbar_init(bar(kBarYFull), 1);
        mbar_init(bar(kBarAccDone), 1);
        mbar_init(bar(kBarAccFree), 128);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(bar(kBarUnitFull + k), 1);
            mbar_init(bar(kBarUnitEmpty + k), kUnitConsumers);
        }
        mbar_init(bar(kBarDrain), 1);
        mbar_init(bar(kBarR0Ready), 128);
        mbar_init(bar(kBarXRead), 128);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmR0);
        if constexpr (L::kRes1) tma_prefetch_desc(&tmR1);
        tma_prefetch_desc(&tmS0);
        tma_prefetch_desc(&tmS1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Consumers take each unit id from the ring (id -1 ends their loop).
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
        // ================================================================ TMA producer
        if (lane == 0) {
            int it = 0, unit_iter = 0, res_loads = 0;
            bool ok = true;
            auto publish = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kBarUnitEmpty + slot), ((k / kUnitSlots) & 1) ^ 1,
                                       abort_flag, budget);
                if (!ok) return -1;
                // a CTA's first unit is its own index (the grid never exceeds the unit
                // count); the counter numbers the rest from gridDim.x on
                unsigned next = k == 0 ? blockIdx.x : gridDim.x + atomicAdd(p.sched, 1u);
                if constexpr (VARLEN)  // blocks past their sequence, or without a visible pair
                    while (next < static_cast<unsigned>(p.n_units) &&
                           decode<PASS, VARLEN>(static_cast<int>(next), p).n_t == 0)
                        next = gridDim.x + atomicAdd(p.sched, 1u);
                const int v = next < static_cast<unsigned>(p.n_units) ? static_cast<int>(next) : -1;
                unit_ring[slot] = v;
                mbar_arrive(bar(kBarUnitFull + slot));
                return v;
            };
            int u = publish(0);
            for (; ok && u >= 0; ++unit_iter) {
                const Unit U = decode<PASS, VARLEN>(u, p);
                // resident tiles (and, in the dQ pass, their rows' L and D)
                ok = mbar_wait_bounded(bar(kBarResEmpty), (unit_iter & 1) ^ 1, abort_flag, budget);
                if (!ok) break;
                if (unit_iter != p.fault_unit) {
                    constexpr uint32_t kResTx =
                        (L::kRes1 ? kResBytes : 0) + (PASS == kPassDQ ? 2 * kRows * 4 : 0);
                    mbar_arrive_expect_tx(bar(kBarResFull), kResTx);
                    int ry, rz;
                    coords<VARLEN>(U.head, PASS == kPassDQ ? p.H : p.Hkv,
                                   PASS == kPassDQ ? U.q_tok0 : U.k_tok0, U.r0, ry, rz);
                    if constexpr (L::kRes1)
                        for (int g = 0; g < kRegions; ++g)
                            tma_load_3d(sR1 + g * kResRegion, &tmR1, bar(kBarResFull), 64 * g, ry, rz);
                    if constexpr (PASS == kPassDQ) {
                        const size_t vrow = vec_row<VARLEN>(U, U.head, U.r0, p);
                        bulk_load(sVec, p.Lw + vrow, kRows * 4, bar(kBarResFull));
                        bulk_load(sVec + kRows * 4, p.Dw + vrow, kRows * 4, bar(kBarResFull));
                    }
                }
                ++res_loads;
                const int u_next = publish(unit_iter + 1);
                if (!ok) break;
                if (u_next >= 0) {
                    // the next unit's first resident rows into L2 for the compute warps
                    const Unit W = decode<PASS, VARLEN>(u_next, p);
                    int wy, wz;
                    coords<VARLEN>(W.head, PASS == kPassDQ ? p.H : p.Hkv,
                                   PASS == kPassDQ ? W.q_tok0 : W.k_tok0, W.r0, wy, wz);
                    for (int g = 0; g < kRegions; ++g) tma_prefetch_l2_3d(&tmR0, 64 * g, wy, wz);
                }
                for (int t = 0; ok && t < U.n_t; ++t, ++it) {
                    int head, row0;
                    tile_of<PASS>(U, t, p, head, row0);
                    // The L / D vectors of a streamed tile go to slot it % kVecSlots of
                    // their ring, completing on the tile's barrier. Before writing them
                    // this thread has waited for s0's slot of tile it - kS0 to be free,
                    // which the MMA warp signals only after the compute warps finished
                    // tile it - kS0 (dK pass: after its accumulation; dV pass: after its
                    // A was ready), so tile it - kS0 and every older one are done with
                    // their vectors, and the kS0 - 1 tiles after it hold the other slots.
                    const size_t vrow = PASS == kPassDQ ? 0 : vec_row<VARLEN>(U, head, row0, p);
                    const int vs = it % kVecSlots;
                    int sy, sz;
                    coords<VARLEN>(head, PASS == kPassDQ ? p.Hkv : p.H,
                                   PASS == kPassDQ ? U.k_tok0 : U.q_tok0, row0, sy, sz);
                    int s = it % kS0;
                    ok = mbar_wait_bounded(bar(kBarS0Empty + s), ((it / kS0) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kBarS0Full + s),
                                          kStrBytes + (PASS == kPassDQ ? 0 : kCols * 4));
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sS0(it) + g * kStrRegion, &tmS0, bar(kBarS0Full + s), 64 * g, sy, sz);
                    if constexpr (PASS != kPassDQ)
                        bulk_load(sVec + vs * kCols * 4, p.Lw + vrow, kCols * 4, bar(kBarS0Full + s));
                    s = it % kS1;
                    ok = mbar_wait_bounded(bar(kBarS1Empty + s), ((it / kS1) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kBarS1Full + s),
                                          kStrBytes + (PASS == kPassDK ? kCols * 4 : 0));
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sS1(it) + g * kStrRegion, &tmS1, bar(kBarS1Full + s), 64 * g, sy, sz);
                    if constexpr (PASS == kPassDK)
                        bulk_load(sVec + (kVecSlots + vs) * kCols * 4, p.Dw + vrow, kCols * 4,
                                  bar(kBarS1Full + s));
                }
                u = u_next;
            }
            if (!ok) record_timeout(p, abort_flag, kRoleTma, u);
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            if (res_loads > 0)
                mbar_wait_bounded(bar(kBarResFull), (res_loads - 1) & 1, nullptr, budget);
            for (int s = 0; s < kS0; ++s)
                if (it > s) {
                    const int last = it - 1 - ((it - 1 - s) % kS0);
                    mbar_wait_bounded(bar(kBarS0Full + s), (last / kS0) & 1, nullptr, budget);
                }
            for (int s = 0; s < kS1; ++s)
                if (it > s) {
                    const int last = it - 1 - ((it - 1 - s) % kS1);
                    mbar_wait_bounded(bar(kBarS1Full + s), (last / kS1) & 1, nullptr, budget);
                }
        }
    } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        // Per streamed tile t (it counts tiles over the CTA's whole sequence):
        //   dQ / dK: ... X(t+1) ... acc += A(t) B(t) | Y(t+1) | X(t+2) ...
        //   dV:      ... X(t+1) ... acc += A(t) B(t) | X(t+2) ...
        // A(t) lies over Y's columns (dQ, dK) or over X(t)'s buffer (dV), and the
        // product that overwrites it (Y(t+1), X(t+2)) follows the accumulation that
        // reads it; X(t+1) waits until the compute warps have loaded X(t) (dQ, dK) or
        // goes to the other buffer (dV): tcgen05.mma operations of one thread execute
        // in issue order.
        constexpr uint32_t idesc_x = idesc_f16_ab(BF16, kRows, kCols, false, false);
        constexpr uint32_t idesc_acc = idesc_f16_ab(BF16, kRows, kD, false, true);
        auto wait = [&](int b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag, budget));
        };
        auto commit = [&](int b) {
            if (elect_one()) umma_commit(bar(b));
            __syncwarp();
        };
        // C[128 x 64] = A B^T, A the resident tile (128 rows), B a streamed tile (64
        // rows), both K-major; K-step k reads 16 columns of region k / 4.
        auto issue_x = [&](uint32_t a_s, uint32_t b_s, uint32_t dcol) {
            tc_fence_after();
            const uint64_t da = swz_desc<128>(a_s, 16);
            const uint64_t db = swz_desc<128>(b_s, 16);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t oa = (k / 4) * (kResRegion >> 4) + (k % 4) * 2;
                    const uint32_t ob = (k / 4) * (kStrRegion >> 4) + (k % 4) * 2;
                    umma_f16_ss(tmem + dcol, da + oa, db + ob, idesc_x, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
        };
        // The same with A the first resident tile in TMEM (K-step k: 8 columns).
        auto issue_x_t = [&](uint32_t b_s, uint32_t dcol) {
            tc_fence_after();
            const uint64_t db = swz_desc<128>(b_s, 16);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t ob = (k / 4) * (kStrRegion >> 4) + (k % 4) * 2;
                    umma_f16_ts(tmem + dcol, tmem + kTmemR0 + 8 * k, db + ob, idesc_x, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
        };
        // acc[128 x 256] (+)= A[128 x 64] B[64 x 256]: A 16-bit pairs in TMEM over X's
        // columns, B the streamed tile MN-major (its 64-column regions 8 KB apart,
        // 16 rows = 2 KB per K-step).
        auto issue_acc = [&](uint32_t b_s, uint32_t acol, bool accumulate) {
            tc_fence_after();
            const uint64_t db = swz_desc<128>(b_s, kStrRegion);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kCols / 16; ++k)
                    umma_f16_ts(tmem + kTmemAcc, tmem + acol + 8 * k, db + k * ((16 * 128) >> 4),
                                idesc_acc, (k > 0 || accumulate) ? 1u : 0u);
            }
            __syncwarp();
        };
        int it = 0, unit_iter = 0, u = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            u = take_unit(unit_iter, ok);
            if (!ok || u < 0) break;
            const Unit U = decode<PASS, VARLEN>(u, p);
            ok = wait(kBarResFull, unit_iter & 1) && wait(kBarR0Ready, unit_iter & 1);
            // X(t) of the unit's tile t (ring position it0 + t) into its buffer
            auto form_x = [&](int pos) -> bool {
                if (!wait(kBarS0Full + pos % kS0, (pos / kS0) & 1)) return false;
                issue_x_t(sS0(pos), xcol(pos));
                commit(kBarXFull + pos % kXBufs);
                return true;
            };
            if constexpr (PASS == kPassDV) {
                // X one tile ahead: X(t+1) goes into the other buffer before A(t) is
                // awaited, and the accumulation of A(t) precedes X(t+2), which
                // overwrites it (one thread's MMAs execute in issue order).
                if (ok && U.n_t > 0) ok = form_x(it);
                for (int t = 0; ok && t < U.n_t; ++t, ++it) {
                    if (t + 1 < U.n_t && !(ok = form_x(it + 1))) break;
                    ok = wait(kBarAReady + it % kXBufs, (it / kXBufs) & 1);
                    if (ok && t == 0 && unit_iter > 0) ok = wait(kBarAccFree, (unit_iter - 1) & 1);
                    if (!ok) break;
                    commit(kBarS0Empty + it % kS0);  // Q_i: X was its one product reader
                    ok = wait(kBarS1Full + it % kS1, (it / kS1) & 1);
                    if (!ok) break;
                    issue_acc(sS1(it), xcol(it), t > 0);  // dV += P^T dO_i
                    commit(kBarS1Empty + it % kS1);
                }
            } else {
                // A(t) goes over Y's columns, so X(t+1) can run while the compute warps
                // form A(t) (once they have loaded X(t)); Y(t+1) follows the
                // accumulation that reads A(t).
                auto form_y = [&](int pos) -> bool {
                    if (!wait(kBarS1Full + pos % kS1, (pos / kS1) & 1)) return false;
                    issue_x(sR1, sS1(pos), kTmemY);
                    commit(kBarYFull);
                    commit(kBarS1Empty + pos % kS1);  // V_j / dO_i: Y was its one reader
                    return true;
                };
                if (ok && U.n_t > 0) ok = form_x(it) && form_y(it);
                for (int t = 0; ok && t < U.n_t; ++t, ++it) {
                    if (t + 1 < U.n_t && !(ok = wait(kBarXRead, it & 1) && form_x(it + 1))) break;
                    ok = wait(kBarAReady, it & 1);
                    if (ok && t == 0 && unit_iter > 0) ok = wait(kBarAccFree, (unit_iter - 1) & 1);
                    if (!ok) break;
                    issue_acc(sS0(it), kTmemY, t > 0);  // dQ += dS K_j, dK += dS^T Q_i
                    commit(kBarS0Empty + it % kS0);
                    if (t + 1 < U.n_t && !(ok = form_y(it + 1))) break;
                }
            }
            if (!ok) break;
            commit(kBarResEmpty);  // resident tiles free once the unit's products complete
            commit(kBarAccDone);   // and the accumulator is final
        }
        if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleMma, u);
        // Drain: every MMA this warp issued has completed before TMEM is freed.
        if (elect_one()) umma_commit(bar(kBarDrain));
        __syncwarp();
        if (lane == 0) mbar_wait_bounded(bar(kBarDrain), 0, nullptr, budget);
        __syncwarp();
    } else if (warp < 4) {
        // ================================================================ compute warpgroup
        const int r = threadIdx.x;  // resident row = TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        // Unit uu's first resident tile into TMEM: this thread's row (512 contiguous
        // bytes, zeros past the rows) into its lane, 16-bit pairs in column order.
        // Called once every X of the previous unit has completed.
        auto load_r0 = [&](int uu) {
            const Unit W = decode<PASS, VARLEN>(uu, p);
            const int wrow = W.r0 + r;
            const bool wok = wrow < (PASS == kPassDQ ? W.nq : W.nk);
            size_t grow;
            if constexpr (VARLEN) {
                const int heads = PASS == kPassDQ ? p.H : p.Hkv;
                grow = (static_cast<size_t>(PASS == kPassDQ ? W.q_tok0 : W.k_tok0) + (wok ? wrow : 0)) * heads +
                       W.head % heads;
            } else {
                grow = static_cast<size_t>(W.head) * p.N + (wok ? wrow : 0);
            }
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.res0) +
                                                               grow * (kD * 2));
            uint4 v[kD / 8];
#pragma unroll
            for (int c = 0; c < kD / 8; ++c) v[c] = wok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int g = 0; g < kRegions; ++g) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    w[4 * c] = v[8 * g + c].x;
                    w[4 * c + 1] = v[8 * g + c].y;
                    w[4 * c + 2] = v[8 * g + c].z;
                    w[4 * c + 3] = v[8 * g + c].w;
                }
                tmem_st32(tl + kTmemR0 + g * 32, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(kBarR0Ready));
        };
        int it = 0, unit_iter = 0, u = -1, u_next = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            if (unit_iter > 0) {
                u = u_next;  // taken, and its resident tile loaded, before the last epilogue
            } else {
                u = take_unit(unit_iter, ok);
                if (ok && u >= 0) load_r0(u);
            }
            if (!ok || u < 0) break;
            const Unit U = decode<PASS, VARLEN>(u, p);
            const int row = U.r0 + r;  // query (dQ pass) or key of this thread, in its sequence
            const bool row_ok = row < (PASS == kPassDQ ? U.nq : U.nk);
            if constexpr (PASS == kPassDQ) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarResFull), unit_iter & 1,
                                                               abort_flag, budget));
                if (!ok) break;
            }
            // dQ pass: this row's L and D, resident for the unit
            float Lrow = 0.f, Drow = 0.f;
            if constexpr (PASS == kPassDQ) {
                Lrow = vec[r];
                Drow = vec[kRows + r];
            }
            for (int t = 0; t < U.n_t; ++t, ++it) {
                int head, c0;
                tile_of<PASS>(U, t, p, head, c0);  // column c is streamed row c0 + c
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarXFull + it % kXBufs),
                                                               (it / kXBufs) & 1, abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                float x[kCols];
                {
                    uint32_t a[32], b[32];
                    tmem_ld32(tl + xcol(it), a);
                    tmem_ld32(tl + xcol(it) + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        x[c] = __uint_as_float(a[c]);
                        x[c + 32] = __uint_as_float(b[c]);
                    }
                }
                if constexpr (kHasY) mbar_arrive(bar(kBarXRead));  // X may be overwritten
                // P = 2^(x scale log2 e - L) with L of the query: the row's (dQ pass) or
                // the column's (the streamed query rows' L, from the vector ring)
                const int vs = it % kVecSlots;
                if constexpr (PASS == kPassDQ) {
#pragma unroll
                    for (int c = 0; c < kCols; c += 2) ffma2(x[c], x[c + 1], sl2, sl2, -Lrow, -Lrow);
                } else {
                    const float *lv = vec + vs * kCols;
#pragma unroll
                    for (int c = 0; c < kCols; c += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(lv + c);
                        ffma2(x[c], x[c + 1], sl2, sl2, -l4.x, -l4.y);
                        ffma2(x[c + 2], x[c + 3], sl2, sl2, -l4.z, -l4.w);
                    }
                }
#pragma unroll
                for (int c = 0; c < kCols; ++c) x[c] = ex2_approx(x[c]);
                // visible pairs: key j and query i with i - wl <= j <= i + wr, both < N
                if constexpr (PASS == kPassDQ) {
                    // row = query (key position row + q_off), columns = keys c0 + c
                    mask_outside_run(x, max(0, row + U.q_off - p.wl) - c0,
                                     min(U.nk - 1, row + U.q_off + p.wr) - c0, 0.f);
                } else {
                    // row = key, columns = queries c0 + c (at key positions c0 + c + q_off)
                    mask_outside_run(x, max(0, row - U.q_off - p.wr) - c0,
                                     min(U.nq - 1, row - U.q_off + p.wl) - c0, 0.f);
                    if (!row_ok) {
#pragma unroll
                        for (int c = 0; c < kCols; ++c) x[c] = 0.f;
                    }
                }
                if constexpr (kHasY) {
                    // dS = P (dP - D), D of the query: the row's or the column's
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarYFull), it & 1, abort_flag, budget));
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t a[32], b[32];
                    tmem_ld32(tl + kTmemY, a);
                    tmem_ld32(tl + kTmemY + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
                    const float *dv = vec + (kVecSlots + vs) * kCols;
#pragma unroll
                    for (int c = 0; c < kCols; c += 2) {
                        const uint32_t *src = c < 32 ? a + c : b + (c - 32);
                        float y0 = __uint_as_float(src[0]), y1 = __uint_as_float(src[1]);
                        if constexpr (PASS == kPassDQ) {
                            fadd2(y0, y1, -Drow, -Drow);
                        } else {
                            const float2 d2 = *reinterpret_cast<const float2 *>(dv + c);
                            fadd2(y0, y1, -d2.x, -d2.y);
                        }
                        fmul2(y0, y1, x[c], x[c + 1]);
                        x[c] = y0;
                        x[c + 1] = y1;
                    }
                }
                // A as 16-bit pairs over the first 32 columns of Y (dQ, dK: this thread
                // has read its Y row) or of X (dV)
                {
                    const uint32_t acol = kHasY ? kTmemY : xcol(it);
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = pack2<BF16>(x[2 * e], x[2 * e + 1]);
                    tmem_st16(tl + acol, pk);
                    tmem_st16(tl + acol + 16, pk + 16);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kBarAReady + it % kXBufs));
            }
            if (!ok) break;
            // The next unit's first resident tile replaces this one's in TMEM: every X
            // of this unit has completed (its last one was read above), and the MMA
            // warp can form the next unit's first X during this epilogue.
            u_next = take_unit(unit_iter + 1, ok);
            if (!ok) break;
            if (u_next >= 0) load_r0(u_next);
            // ---- epilogue: the row of the accumulator times out_scale, in 16 bit
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarAccDone), unit_iter & 1, abort_flag, budget));
            if (!ok) break;
            tc_fence_after();
            {
                const float f = p.out_scale;
                // global row: (head, row), or (token, head) in a variable-length batch
                size_t orow;
                if constexpr (VARLEN) {
                    const int heads = PASS == kPassDQ ? p.H : p.Hkv;
                    orow = (static_cast<size_t>(PASS == kPassDQ ? U.q_tok0 : U.k_tok0) + (row_ok ? row : 0)) *
                               heads + U.head % heads;
                } else {
                    orow = static_cast<size_t>(U.head) * p.N + (row_ok ? row : 0);
                }
                uint8_t *out = reinterpret_cast<uint8_t *>(p.out) + orow * (kD * 2);
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t a[32];
                    tmem_ld32(tl + kTmemAcc + c * 32, a);
                    tmem_ld_wait(a);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * f, __uint_as_float(a[2 * e + 1]) * f);
                    if (row_ok) {
                        st_global_v8(out + c * 64, pk);
                        st_global_v8(out + c * 64 + 32, pk + 8);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(kBarAccFree));
        }
        if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleCompute, u);
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The last CTA to finish zeroes this launch's scheduler counters for the next
    // launch that uses them (every CTA has stopped taking units by now).
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

}  // namespace bwd256
}  // namespace fa
