// fa_fwd_kernel.cuh -- attention forward for sm_103a: TMA -> shared memory ->
// tcgen05.mma with fp32 accumulators in tensor memory -> online softmax in
// registers -> P back into tensor memory -> tcgen05.mma -> O and LSE.
//
// Method (the pages): Q is cut into Br-row blocks and K/V into Bc-row blocks,
// the outer loop runs over Q blocks and the inner loop over K/V blocks so that
// only O(Br*d + Bc*d) lives on chip ("ai6s.net/6af30f4d40858c2d8819b6d5" §2.2);
// per K/V block the running row max m and row sum l are updated and the output
// accumulator is rescaled by exp(m_old - m_new) (same page, §2.3; the C snippet
// of "aicoding.csdn.net/6a69d3ff10ee7a33f2941f44", "Online softmax算法"); the
// accumulator is divided by l once after the last block and m, l are kept as
// LSE (§2.4 and the teaching kernel's final normalisation, §2.5). exp2 with
// log2(e) folded into the scale and the block-level skip of fully masked K/V
// blocks are refinements listed at the end of §2.5. The mask variants are
// applied right after the score block is formed, as the catlass epilogue does
// ("ai6s.net/6a0ed07b662f9a54cb761aa2", Epilogue Builder). Two Q blocks are
// kept in flight so that the matrix unit works on one while the softmax of the
// other runs: the GPU form of the Cube/Vector overlap of
// "ai6s.net/6af30f4d40858c2d8819b6d5" §3.3 (1). The CTA grid is persistent and
// takes work units (the per-core Q-block split of the same page's host tiling,
// §3.2-§3.3) from a launch-wide counter, heaviest first under causal and window
// masks.
//
// One CTA (384 threads) runs on each SM and loops over work units; a unit is
// 256 query rows (two 128-row Q tiles, t = 0, 1) of one (b, h):
//   warps 0-3 : softmax of Q tile 0 (thread = query row = TMEM lane)
//   warps 4-7 : softmax of Q tile 1
//   warp 8    : scheduler (takes work units from a launch-wide counter) and TMA
//               producer of the Q tiles and of K_j into a multi-stage ring
//   warp 9    : MMA issuer (one elected lane)
//   warp 10   : TMA producer of V_j (its own thread, so K and V prefetch
//               independently: each is issued as soon as its own slot frees)
//   warp 11   : idle (completes warpgroup 2, whose registers move to the
//               softmax warpgroups with setmaxnreg)
// Tensor memory (512 columns): S_t at columns 128 t (fp32, 128 keys), O_t at
// 256 + t d (fp32). After the softmax of S_t(j) the probabilities P_t(j) are
// written as packed 16-bit pairs over the first 64 columns of S_t, and
// O_t += P_t(j) V_j reads them from tensor memory (A operand in TMEM).
// Issue order, iteration j:  S_0(j) | O_1 += P_1(j-1) V_{j-1} | S_1(j) | O_0 += P_0(j) V_j.
// Each softmax overlaps two MMA groups of the other tile. S_t(j+1) follows
// O_t += P_t(j) V_j directly: tcgen05.mma operations of one thread execute in
// issue order, so the P read of the earlier MMA precedes the S write of the
// later one.
//
// On K/V blocks that every row of the Q tile sees whole, the row maximum comes from
// the reducing TMEM load (fa_tmem_max.cuh) instead of 128 comparisons per thread.
//
// Each softmax thread stores its row of O / l with 32-byte stores (one TMEM lane
// per thread, so a warp's stores go to 32 rows; the wider stores halve the store
// instructions, which share the memory-instruction queue with every warp's
// mbarrier operations).
//
// The output accumulator is rescaled lazily: the reference max of a row only
// moves when a block's max exceeds it by more than 2^8 (in log2 units), so
// every probability stays below 256 and O and l share the same reference,
// which keeps the result exact; most blocks then need no rescale at all.
//
// Every wait is bounded (global-timer budget); on expiry the CTA records the
// failure in a status word, drains its own copies and MMAs, frees its tensor
// memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_mask.cuh"
#include "fa_tmem_max.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kBM = 128;       // query rows per Q tile = TMEM lanes
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kQTiles = 2;     // Q tiles per work unit
constexpr int kUnitRows = kBM * kQTiles;
constexpr int kThreads = 384;  // 2 softmax warpgroups + a warpgroup with the TMA and MMA warps
constexpr int kTmaWarp = 8;   // scheduler, Q and K loads
constexpr int kMmaWarp = 9;
constexpr int kVWarp = 10;    // V loads
// Per-thread registers after setmaxnreg. Their sum over the CTA must not exceed
// what the launch allocated (threads x registers of the compiled kernel); the
// host checks this before the first launch.
#ifndef FA_REGS_SOFTMAX
#define FA_REGS_SOFTMAX 200
#endif
#ifndef FA_REGS_CONTROL
#define FA_REGS_CONTROL 104
#endif
constexpr int kRegsSoftmax = FA_REGS_SOFTMAX;
constexpr int kRegsControl = FA_REGS_CONTROL;
constexpr int kRegsNeeded = 2 * 128 * kRegsSoftmax + 128 * kRegsControl;
// Tiles are stored as regions of min(d, 64) columns x 128 rows with the swizzle of
// that row width (128 B, or 64 B for d = 32).
template <int D>
struct Regions {
    static constexpr int kCols = D < 64 ? D : 64;
    static constexpr int kRowBytes = kCols * 2;
    static constexpr int kBytes = 128 * kRowBytes;
    static constexpr int kCount = D / kCols;
    static constexpr int kStepsPerRegion = kCols / 16;  // K-steps of 16 columns per region
};
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: probabilities stay <= 2^8
// How many keys the softmax packs per TMEM store of P.
#ifndef FA_P_CHUNK
#define FA_P_CHUNK 32
#endif
constexpr int kPChunk = FA_P_CHUNK;

constexpr unsigned kStatusTimeout = 4;  // same value as FA_ERR_TIMEOUT
enum : int { kRoleSoftmax = 1, kRoleTma = 2, kRoleMma = 3 };

struct FwdParams {
    void *O;
    float *LSE;
    float *part_O;    // split mode: fp32 partial outputs [split][b*H+h][Nq][d]; null: write O, LSE
    float *part_LSE;  // split mode: partial log-sum-exps [split][b*H+h][Nq]
    int Nq, Nk;       // query rows and keys per head
    int q_off;        // query i sits at key position i + q_off (Nk - Nq: the last Nq positions)
    int H;            // query heads
    int BH;           // B * H
    int kv_group;     // query heads per K/V head (H / H_kv; 1 = one K/V head per query head)
    // Rows are processed in "row spaces" of R rows. Unpacked: one per query head
    // (R = Nq). Packed (kernel template flag; few queries, grouped K/V heads): one
    // per K/V head, holding the Nq queries of each of its kv_group query heads one
    // after the other (R = kv_group * Nq), so that one unit streams a K/V head once
    // for all of them. Row r of row space s is global row s * R + r of the
    // B*H*Nq query rows (in both cases), and query index r mod Nq of its head.
    int R;
    int n_units;      // (row space, 256-row block, key split) work units
    int n_qb;         // 256-row blocks per row space: ceil(R / 256)
    int n_splits;     // key splits per row block (1: no split)
    int split_tiles;  // K/V tiles per key split
    int heavy_first;  // 1: visit row blocks from the last (most keys) to the first
    // Order in which the scheduler hands out units (scheduled_unit): row spaces
    // in groups of `group`, and within a group all spaces' first row blocks in
    // the visiting order (the heaviest, with heavy_first), then their second ones:
    // the lightest units of the launch then come last, where they even out the
    // CTAs' finishing times. 1: one space at a time (space-major).
    int group;
    int n_spaces;     // row spaces of the launch
    int wl, wr;       // key j visible to query i iff i + q_off - wl <= j <= i + q_off + wr
    float scale_log2; // scale * log2(e)
    unsigned long long wait_budget_ns;
    unsigned int *status;  // [code, role, unit, block]
    // Debug builds with FA_DEBUG_BOUNDS: rows of O / LSE (and of each split's part
    // buffers), and a test shift added to every stored row (0 unless armed).
    long long out_rows;
    long long row_shift;
    int fault_skip_k;      // test hook: every CTA skips the K load at this ring position (-1: none)
    // Variable-length batches (kernel template flag): sequence b holds query tokens
    // cu_q[b] .. cu_q[b+1]-1 and keys cu_k[b] .. cu_k[b+1]-1 of token-major tensors
    // (total x heads x d); row spaces are (b, h) and Nq stands for the longest
    // sequence's query count. Lengths are clamped to [0, total] so that no stray
    // value can address memory outside the tensors.
    const int *cu_q;
    const int *cu_k;
    int total_q, total_k;
    unsigned int *sched;   // this launch's {next unit, finished CTAs} counters (zero at launch)
};

// Debug builds (never the default):
//  * FA_DEBUG_SERIALIZE: the least overlap the kernel's protocol allows, to expose
//    ordering mistakes: K/V rings two deep (the minimum: an iteration reads two
//    tiles), the next unit claimed only with the current unit's last K/V tile,
//    and every group of MMAs completed before the next one is issued.
//  * FA_DEBUG_BOUNDS: every store of O, LSE and the split buffers is checked against
//    the output's rows first; an out-of-range row is not stored, and the first one
//    is recorded in the status word (code 5, FA_ERR_BOUNDS) instead of faulting.
#ifdef FA_DEBUG_SERIALIZE
constexpr bool kDebugSerialize = true;
#else
constexpr bool kDebugSerialize = false;
#endif
#ifdef FA_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif
constexpr unsigned kStatusBounds = 5;  // same value as FA_ERR_BOUNDS

#ifndef FA_KSTAGES_128
#define FA_KSTAGES_128 2
#endif
#ifndef FA_VSTAGES_128
#define FA_VSTAGES_128 2
#endif
template <int D>
struct SmemLayout {
    // K and V ring depths. The footprint stays above half of the SM's shared
    // memory, so one CTA (holding all 512 TMEM columns) runs per SM. K_j is
    // needed a whole softmax earlier than V_j, so its ring is the deeper one.
    static constexpr int kStagesK = kDebugSerialize ? 2 : D == 128 ? FA_KSTAGES_128 : 4;
    static constexpr int kStagesV = kDebugSerialize ? 2 : D == 128 ? FA_VSTAGES_128 : 4;
    static constexpr int kTileBytes = kBM * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kQTiles * kTileBytes;
    static constexpr int kV = kK + kStagesK * kTileBytes;
    static constexpr int kBar = kV + kStagesV * kTileBytes;
    static constexpr int kNumBars = 40;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kUnitRing = kMisc + 16;  // kUnitSlots ints: unit ids handed out to the roles
    static constexpr int kBytes = kUnitRing + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t kTmemO = 256;       // O_t at kTmemO + t * D
};

constexpr int kMaxStages = 4;
constexpr int kUnitSlots = 2;  // unit ids in flight between the scheduler and the other roles
// Arrivals that free a unit slot: one per consumer warp (the MMA warp, the V producer
// and the 8 softmax warps).
constexpr int kUnitConsumers = 1 + 1 + 8;
enum : int {
    kBarQFull = 0,                          // + t
    kBarQEmpty = kBarQFull + kQTiles,       // + t
    kBarKFull = kBarQEmpty + kQTiles,       // + stage
    kBarVFull = kBarKFull + kMaxStages,     // + stage
    kBarKEmpty = kBarVFull + kMaxStages,    // + stage
    kBarVEmpty = kBarKEmpty + kMaxStages,   // + stage
    kBarSFull = kBarVEmpty + kMaxStages,    // + t
    kBarPFull = kBarSFull + kQTiles,        // + t
    kBarODone = kBarPFull + kQTiles,        // + t
    kBarOFree = kBarODone + kQTiles,        // + t
    kBarDrain = kBarOFree + kQTiles,
    kBarUnitFull = kBarDrain + 1,           // + slot
    kBarUnitEmpty = kBarUnitFull + 2,       // + slot
    kBarSerial = kBarUnitEmpty + 2,         // FA_DEBUG_SERIALIZE: completion of each MMA group
    kNumBarsUsed = kBarSerial + 1,
};

// A work unit: rows [r0, r0 + 256) of row space rs (global rows rs * R + r)
// whose keys and values are those of K/V head bkv (= b * H_kv + h / kv_group),
// restricted to the K/V tiles of key split `split`; Q tile t covers rows
// [r0 + 128 t, r0 + 128 t + 128) and needs K/V tiles [a[t], b[t]] (empty when
// a > b); [j0, j1] is their union.
struct UnitBase {
    int rs, bkv, r0, split;
    int a[kQTiles], b[kQTiles];
    int j0, j1;
};
// Variable-length batches only: this sequence's query rows and keys, the query
// position offset, its first token rows and its heads.
struct UnitSeq {
    int nq, nk, q_off, q_tok0, k_tok0, h, hkv;
};
template <bool VARLEN>
struct Unit : UnitBase {};
template <>
struct Unit<true> : UnitBase, UnitSeq {};

// Sizes of the unit's problem: the launch's, or (VARLEN) its sequence's.
template <bool VARLEN>
__device__ __forceinline__ int unit_rows(const Unit<VARLEN> &U, const FwdParams &p) {
    if constexpr (VARLEN) return U.nq;
    else return p.R;
}
template <bool VARLEN>
__device__ __forceinline__ int unit_keys(const Unit<VARLEN> &U, const FwdParams &p) {
    if constexpr (VARLEN) return U.nk;
    else return p.Nk;
}
template <bool VARLEN>
__device__ __forceinline__ int unit_qoff(const Unit<VARLEN> &U, const FwdParams &p) {
    if constexpr (VARLEN) return U.q_off;
    else return p.q_off;
}

// Query indices (0..Nq-1) met by the rows [rt0, rl] of a row space (an unpacked
// row space is one head: rows are queries).
template <bool PACKED>
__device__ __forceinline__ void tile_queries(const FwdParams &p, int rt0, int rl, int &i_lo,
                                             int &i_hi) {
    if (!PACKED) {
        i_lo = rt0;
        i_hi = rl;
        return;
    }
    const int a = rt0 % p.Nq, b = rl % p.Nq;
    if (rl - rt0 + 1 >= p.Nq || b < a) {
        i_lo = 0;
        i_hi = p.Nq - 1;
    } else {
        i_lo = a;
        i_hi = b;
    }
}

template <bool PACKED, bool VARLEN>
__device__ __forceinline__ Unit<VARLEN> decode_unit(int u, const FwdParams &p) {
    Unit<VARLEN> U;
    const int per_space = p.n_qb * p.n_splits;
    const int rs = u / per_space;
    const int rem = u - rs * per_space;
    int qb = rem / p.n_splits;
    U.split = rem - qb * p.n_splits;
    U.rs = rs;
    if (PACKED) {
        U.bkv = rs;
    } else {
        const int b = rs / p.H, h = rs - b * p.H;
        U.bkv = b * (p.H / p.kv_group) + h / p.kv_group;
        if constexpr (VARLEN) {
            U.h = h;
            U.hkv = h / p.kv_group;
            const int q0 = min(max(p.cu_q[b], 0), p.total_q);
            const int q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
            const int k0 = min(max(p.cu_k[b], 0), p.total_k);
            const int k1 = min(max(p.cu_k[b + 1], k0), p.total_k);
            U.q_tok0 = q0;
            U.k_tok0 = k0;
            U.nq = q1 - q0;
            U.nk = k1 - k0;
            U.q_off = U.nk - U.nq;
        }
    }
    if (p.heavy_first) qb = p.n_qb - 1 - qb;
    U.r0 = qb * kUnitRows;
    const int s_lo = U.split * p.split_tiles;
    const int s_hi = s_lo + p.split_tiles - 1;
    U.j0 = 0x7fffffff;
    U.j1 = -1;
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {
        const int rt0 = U.r0 + t * kBM;
        U.a[t] = 1;
        U.b[t] = 0;
        const int R = unit_rows<VARLEN>(U, p);
        const int nk = unit_keys<VARLEN>(U, p);
        const int q_off = unit_qoff<VARLEN>(U, p);
        if (rt0 < R) {
            const int rl = min(rt0 + kBM, R) - 1;
            int i_lo, i_hi;
            tile_queries<PACKED>(p, rt0, rl, i_lo, i_hi);
            const int lo_key = i_lo + q_off - p.wl;  // first key any row of the tile sees
            const int hi_key = i_hi + q_off + p.wr;  // last key any row of the tile sees
            if (hi_key >= 0 && lo_key <= nk - 1) {
                const int a = max(max(0, lo_key) / kBN, s_lo);
                const int b = min(min(nk - 1, hi_key) / kBN, s_hi);
                if (a <= b) {
                    U.a[t] = a;
                    U.b[t] = b;
                    U.j0 = min(U.j0, a);
                    U.j1 = max(U.j1, b);
                }
            }
        }
    }
    return U;
}

__device__ __forceinline__ bool unit_empty(const UnitBase &U) { return U.j1 < U.j0; }

// The unit id (numbered space-major, as decode_unit reads it) of the n-th unit the
// launch-wide counter hands out. With p.group > 1 the spaces are taken in groups:
// within a group, every space's first row block in the visiting order, then every
// space's second one, and so on. Only the scheduler calls this, once per unit.
__device__ __forceinline__ int scheduled_unit(int n, const FwdParams &p) {
    if (p.group <= 1) return n;
    const int per_space = p.n_qb * p.n_splits;
    const int g = n / (p.group * per_space);
    const int base = g * p.group;
    const int gs = min(p.group, p.n_spaces - base);  // spaces in this group
    const int rem = n - base * per_space;
    const int qbi = rem / (gs * p.n_splits);
    const int rem2 = rem - qbi * gs * p.n_splits;
    const int hi = rem2 / p.n_splits;
    const int split = rem2 - hi * p.n_splits;
    return (base + hi) * per_space + qbi * p.n_splits + split;
}

__device__ __forceinline__ void record_timeout(const FwdParams &p, volatile int *abort_flag,
                                               int role, int unit) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0u, kStatusTimeout) == 0u) {
        p.status[1] = static_cast<unsigned>(role);
        p.status[2] = static_cast<unsigned>(unit);
        p.status[3] = blockIdx.x;
        __threadfence();
    }
}

// One online-softmax step of this thread's row over a 128-key tile whose fp32
// scores sit at TMEM address tS (this warp's lanes). Masks hidden keys (only
// in the kMasked instance), moves the reference max m lazily, adds the tile's
// probabilities to l, and stores them as packed 16-bit pairs at TMEM address
// tP (64 columns). Returns the factor by which the caller must rescale O
// (1 when the reference max did not move). The stores are left in flight:
// the caller waits with tcgen05.wait::st before signalling.
template <bool BF16, int kPChunk, bool kMasked>
__device__ __forceinline__ float softmax_tile(uint32_t tS, uint32_t tP, int kv0, int lo_i, int hi_i,
                                              float sl2, float &m, float &l) {
    uint32_t sr[4][32];
    float x[kBN];
    float m_tile;
    if constexpr (kMasked) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
#pragma unroll
        for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
        mask_outside_run(x, lo_i - kv0, hi_i - kv0, -INFINITY);
        // Row max: four independent chains of 3-input max.
        float ma = fmaxf(x[0], x[1]), mb = fmaxf(x[2], x[3]);
        float mc = fmaxf(x[4], x[5]), md = fmaxf(x[6], x[7]);
#pragma unroll
        for (int c = 8; c < kBN; c += 8) {
            ma = max3f(ma, x[c + 0], x[c + 1]);
            mb = max3f(mb, x[c + 2], x[c + 3]);
            mc = max3f(mc, x[c + 4], x[c + 5]);
            md = max3f(md, x[c + 6], x[c + 7]);
        }
        m_tile = fmaxf(fmaxf(ma, mb), fmaxf(mc, md)) * sl2;
    } else {
        // every key visible: the TMEM loads reduce each 32-column run to its maximum
        float mr[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + c * 32, sr[c], mr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_max_wait(sr[c], mr[c]);
#pragma unroll
        for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
        m_tile = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])) * sl2;
    }
    // Lazy rescale: move the reference max only when this block's max exceeds
    // it by more than the threshold.
    const float m_old = m;
    if (m_tile > m + kRescaleThreshold) m = m_tile;
    const float corr = m != m_old ? ex2_approx(m_old - m) : 1.f;
    const float nm = m == -INFINITY ? 0.f : -m;
    // p = 2^(x * scale * log2 e - m), 32 keys at a time; each chunk is packed to
    // 16-bit pairs and stored while the next one is computed.
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    static_assert(kPChunk == 16 || kPChunk == 32 || kPChunk == 64, "P chunk");
#pragma unroll
    for (int c = 0; c < kBN; c += kPChunk) {
#pragma unroll
        for (int e = 0; e < kPChunk; e += 2) {
            ffma2(x[c + e], x[c + e + 1], sl2, sl2, nm, nm);
            x[c + e] = ex2_approx(x[c + e]);
            x[c + e + 1] = ex2_approx(x[c + e + 1]);
        }
#pragma unroll
        for (int e = 0; e < kPChunk; e += 4) {
            fadd2(s0, s1, x[c + e], x[c + e + 1]);
            fadd2(s2, s3, x[c + e + 2], x[c + e + 3]);
        }
        uint32_t pk[kPChunk / 2];
#pragma unroll
        for (int e = 0; e < kPChunk / 2; ++e) pk[e] = pack2<BF16>(x[c + 2 * e], x[c + 2 * e + 1]);
        if constexpr (kPChunk == 64) {
            tmem_st16(tP + c / 2, pk);
            tmem_st16(tP + c / 2 + 16, pk + 16);
        } else if constexpr (kPChunk == 32) {
            tmem_st16(tP + c / 2, pk);
        } else {
            tmem_st8(tP + c / 2, pk);
        }
    }
    l = l * corr + ((s0 + s1) + (s2 + s3));
    return corr;
}

// TMA coordinates of a Q tile (row r of the unit's row space) and of K/V tile j.
// Dense maps are (d, rows, row spaces); variable-length maps (d, heads, tokens).
template <bool VARLEN>
__device__ __forceinline__ void q_coords(const Unit<VARLEN> &U, int r, int &y, int &z) {
    if constexpr (VARLEN) {
        y = U.h;
        z = U.q_tok0 + r;
    } else {
        y = r;
        z = U.rs;
    }
}
template <bool VARLEN>
__device__ __forceinline__ void kv_coords(const Unit<VARLEN> &U, int j, int &y, int &z) {
    if constexpr (VARLEN) {
        y = U.hkv;
        z = U.k_tok0 + j * kBN;
    } else {
        y = j * kBN;
        z = U.bkv;
    }
}

template <int D, bool BF16, bool PACKED, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = SmemLayout<D>;
    using G = Regions<D>;
    constexpr int kRegions = G::kCount;
    constexpr int kStagesK = L::kStagesK;
    constexpr int kStagesV = L::kStagesV;
    static_assert(kStagesK <= kMaxStages && kStagesV <= kMaxStages && kNumBarsUsed <= L::kNumBars,
                  "barrier slots");
    static_assert(L::kAlloc <= 232448, "shared memory per CTA");
    static_assert(D == 32 || D == 64 || D == 128, "head dim");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::kQ;
    const uint32_t sK = sbase + L::kK;
    const uint32_t sV = sbase + L::kV;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::kUnitRing);
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
        for (int t = 0; t < kQTiles; ++t) {
            mbar_init(bar(kBarQFull + t), 1);
            mbar_init(bar(kBarQEmpty + t), 1);
            mbar_init(bar(kBarSFull + t), 1);
            mbar_init(bar(kBarPFull + t), 128);
            mbar_init(bar(kBarODone + t), 1);
            mbar_init(bar(kBarOFree + t), 128);
        }
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        mbar_init(bar(kBarDrain), 1);
        mbar_init(bar(kBarSerial), 1);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(bar(kBarUnitFull + k), 1);
            mbar_init(bar(kBarUnitEmpty + k), kUnitConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Each role's code sits inside the branch of its setmaxnreg, so the
    // compiler allocates it under that register limit.
    if (warp >= 8) {
      setmaxnreg_dec<kRegsControl>();
      if (warp == kTmaWarp) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int kv_iter = 0, unit_iter = 0, q_loads = 0;
            bool ok = true;
            // Scheduler: take units from the launch-wide counter and hand their ids
            // to the other roles through the shared-memory unit ring (id -1 ends
            // every role's loop). The producer works one unit ahead: once the
            // first K tiles of unit u are on their way it already claims and
            // publishes the next unit and prefetches that unit's Q tiles (read
            // once, from DRAM) into L2, so that loading them into shared memory
            // at the unit boundary is an L2 hit.
            auto publish = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kBarUnitEmpty + slot), ((k / kUnitSlots) & 1) ^ 1,
                                       abort_flag, budget);
                if (!ok) return -1;
                // Units with no visible key in their split (possible only with key
                // splits) are skipped here, so every published unit has work. A CTA's
                // first unit is the one numbered like the CTA (the grid never exceeds
                // the unit count), which spares the launch-wide counter's round trip
                // at start-up; the counter then numbers the rest from gridDim.x on.
                int v = -1;
                unsigned next = k == 0 ? blockIdx.x : gridDim.x + atomicAdd(p.sched, 1u);
                for (;; next = gridDim.x + atomicAdd(p.sched, 1u)) {
                    if (next >= static_cast<unsigned>(p.n_units)) break;
                    const int un = scheduled_unit(static_cast<int>(next), p);
                    if (!unit_empty(decode_unit<PACKED, VARLEN>(un, p))) {
                        v = un;
                        break;
                    }
                }
                unit_ring[slot] = v;
                mbar_arrive(bar(kBarUnitFull + slot));
                return v;
            };
            auto prefetch_q_l2 = [&](int v) {
                const auto W = decode_unit<PACKED, VARLEN>(v, p);
                for (int t = 0; t < kQTiles; ++t) {
                    int y, z;
                    q_coords<VARLEN>(W, W.r0 + t * kBM, y, z);
                    for (int g = 0; g < kRegions; ++g) tma_prefetch_l2_3d(&tmQ, G::kCols * g, y, z);
                }
            };
            int u = publish(0);
            for (; ok && u >= 0; ++unit_iter) {
                const auto U = decode_unit<PACKED, VARLEN>(u, p);
                for (int t = 0; t < kQTiles && ok; ++t) {
                    ok = mbar_wait_bounded(bar(kBarQEmpty + t), (unit_iter & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kBarQFull + t), L::kTileBytes);
                    int y, z;
                    q_coords<VARLEN>(U, U.r0 + t * kBM, y, z);
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sQ + t * L::kTileBytes + g * G::kBytes, &tmQ,
                                    bar(kBarQFull + t), G::kCols * g, y, z);
                }
                if (!ok) break;
                ++q_loads;
                int u_next = -1;
                bool claimed = false;
                const int j1 = U.j1;
                for (int j = U.j0; ok && j <= j1; ++j, ++kv_iter) {
                    // claim the next unit after the first two K loads (or at the last one)
                    if (!claimed && ((!kDebugSerialize && j == U.j0 + 2) || j == j1)) {
                        claimed = true;
                        u_next = publish(unit_iter + 1);
                        if (!ok) break;
                        if (u_next >= 0) prefetch_q_l2(u_next);
                    }
                    const int st = kv_iter % kStagesK;
                    const uint32_t ph = (kv_iter / kStagesK) & 1;
                    ok = mbar_wait_bounded(bar(kBarKEmpty + st), ph ^ 1, abort_flag, budget);
                    if (!ok) break;
                    if (kv_iter != p.fault_skip_k) {
                        mbar_arrive_expect_tx(bar(kBarKFull + st), L::kTileBytes);
                        int y, z;
                        kv_coords<VARLEN>(U, j, y, z);
                        for (int g = 0; g < kRegions; ++g)
                            tma_load_3d(sK + st * L::kTileBytes + g * G::kBytes, &tmK,
                                        bar(kBarKFull + st), G::kCols * g, y, z);
                    }
                }
                u = u_next;
            }
            if (!ok) record_timeout(p, abort_flag, kRoleTma, u);
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            if (q_loads > 0)
                for (int t = 0; t < kQTiles; ++t)
                    mbar_wait_bounded(bar(kBarQFull + t), (q_loads - 1) & 1, nullptr, budget);
            for (int s = 0; s < kStagesK; ++s) {
                if (kv_iter > s) {
                    const int last = kv_iter - 1 - ((kv_iter - 1 - s) % kStagesK);
                    mbar_wait_bounded(bar(kBarKFull + s), (last / kStagesK) & 1, nullptr, budget);
                }
            }
        }
      } else if (warp == kVWarp) {
        // ================================================================ V producer
        if (lane == 0) {
            int kv_iter = 0;
            bool ok = true;
            for (int unit_iter = 0; ok; ++unit_iter) {
                const int slot = unit_iter % kUnitSlots;
                ok = mbar_wait_bounded(bar(kBarUnitFull + slot), (unit_iter / kUnitSlots) & 1,
                                       abort_flag, budget);
                if (!ok) break;
                const int u = unit_ring[slot];
                mbar_arrive(bar(kBarUnitEmpty + slot));
                if (u < 0) break;
                const auto U = decode_unit<PACKED, VARLEN>(u, p);
                for (int j = U.j0; ok && j <= U.j1; ++j, ++kv_iter) {
                    const int st = kv_iter % kStagesV;
                    ok = mbar_wait_bounded(bar(kBarVEmpty + st), ((kv_iter / kStagesV) & 1) ^ 1,
                                           abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kBarVFull + st), L::kTileBytes);
                    int y, z;
                    kv_coords<VARLEN>(U, j, y, z);
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sV + st * L::kTileBytes + g * G::kBytes, &tmV,
                                    bar(kBarVFull + st), G::kCols * g, y, z);
                }
                if (!ok) record_timeout(p, abort_flag, kRoleTma, u);
            }
            if (!ok) record_timeout(p, abort_flag, kRoleTma, -1);
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            for (int s = 0; s < kStagesV; ++s) {
                if (kv_iter > s) {
                    const int last = kv_iter - 1 - ((kv_iter - 1 - s) % kStagesV);
                    mbar_wait_bounded(bar(kBarVFull + s), (last / kStagesV) & 1, nullptr, budget);
                }
            }
        }
      } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        // The whole warp walks the schedule (uniform control flow); one elected
        // lane issues each group of tcgen05 instructions. A group of K-steps is
        // fully unrolled with compile-time descriptor offsets: the tensor core
        // accepts only about one MMA ahead, so any instruction latency between
        // two issues becomes idle tensor-core time.
        //
        // Issue order, iteration j of a unit:
        //     S_0(j) | O_1 += P_1(j-1) V_{j-1} | S_1(j) | O_0 += P_0(j) V_j
        // so that each softmax overlaps two MMA groups of the other tile. S_t(j+1)
        // is issued right after O_t += P_t(j) V_j, which reads P_t(j) from the
        // same columns: tcgen05.mma operations from one thread execute in issue
        // order, so the earlier MMA reads its TMEM operand before the later one
        // writes there (an in-order pipeline has no write-after-read hazard).
        constexpr uint32_t idesc_s = idesc_f16(BF16, kBM, kBN, false);
        constexpr uint32_t idesc_o = idesc_f16(BF16, kBM, D, true);
        auto wait = [&](int b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag, budget));
        };
        int kv_base = 0, unit_iter = 0;
        int pv_count[kQTiles] = {0, 0};   // O_t += P_t V issued so far
        int epi_count[kQTiles] = {0, 0};  // units in which Q tile t had an epilogue
        bool ok = true;
        int serial_count = 0;  // FA_DEBUG_SERIALIZE: MMA groups waited for
        // FA_DEBUG_SERIALIZE: the group just issued completes before anything else
        auto serialize = [&]() {
            if constexpr (kDebugSerialize) {
                if (elect_one()) umma_commit(bar(kBarSerial));
                __syncwarp();
                ok = ok && wait(kBarSerial, serial_count++ & 1);
            }
        };
        // S_t(j) = Q_t K_j^T into TMEM columns t * 128.
        auto issue_s = [&](int t, int st) {
            tc_fence_after();
            const uint64_t dq = swz_desc<G::kRowBytes>(sQ + t * L::kTileBytes, 16);
            const uint64_t dk = swz_desc<G::kRowBytes>(sK + st * L::kTileBytes, 16);
            if (elect_one()) {
                // K-step k reads 16 columns: 32 bytes into 64-column region k / 4.
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    constexpr uint32_t kRegion16 = G::kBytes >> 4;
                    const uint32_t off = (k / G::kStepsPerRegion) * kRegion16 +
                                         (k % G::kStepsPerRegion) * 2;
                    umma_f16_ss(tmem + t * kBN, dq + off, dk + off, idesc_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(kBarSFull + t));
            }
            __syncwarp();
            serialize();
        };
        // O_t (+)= P_t V_j, P_t read from TMEM.
        auto issue_pv = [&](int t, int st, bool first) {
            tc_fence_after();
            const uint64_t dv = swz_desc<G::kRowBytes>(sV + st * L::kTileBytes, G::kBytes);
            const uint32_t acc0 = first ? 0u : 1u;
            if (elect_one()) {
                // K-step k reads keys 16k..16k+15: 16 rows of 128 B of V.
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    umma_f16_ts(tmem + L::kTmemO + t * D, tmem + t * kBN + k * 8,
                                dv + k * ((16 * G::kRowBytes) >> 4), idesc_o, k > 0 ? 1u : acc0);
                umma_commit(bar(kBarODone + t));
            }
            __syncwarp();
            ++pv_count[t];
            serialize();
        };
        auto commit = [&](int b) {
            if (elect_one()) umma_commit(bar(b));
            __syncwarp();
        };

        for (; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = wait(kBarUnitFull + slot, (unit_iter / kUnitSlots) & 1);
            if (!ok) break;
            const int u = unit_ring[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(kBarUnitEmpty + slot));
            __syncwarp();
            if (u < 0) break;
            const auto U = decode_unit<PACKED, VARLEN>(u, p);
            for (int t = 0; t < kQTiles && ok; ++t) ok = wait(kBarQFull + t, unit_iter & 1);
            const int j0 = U.j0;
            const int j1 = U.j1;
            auto in = [&U](int t, int j) { return j >= U.a[t] && j <= U.b[t]; };
            // Tile 1's visible keys start exactly one K/V tile after tile 0's (a
            // sliding window whose left edge moves one tile per Q tile): pair the
            // tiles by their own block index instead of by key position. Iteration
            // i then computes S_0 on K/V tile j0 + i and S_1 on j0 + 1 + i, both Q
            // tiles are busy in every iteration (in key order, tile 0 alone would
            // run the first one and tile 1 alone the last), and both P V products
            // of iteration i read the same V tile.
            const bool shifted = U.a[0] <= U.b[0] && U.a[1] <= U.b[1] && U.a[1] == U.a[0] + 1;
            if (shifted) {
                const int last_s = max(U.b[0] - j0, U.b[1] - j0 - 1);  // iteration of the last S
                for (int i = 0; ok && i <= j1 - j0; ++i) {
                    const int ja = j0 + i;
                    const int pa = kv_base + i, pb = pa + 1;  // ring positions of K/V tiles ja, ja + 1
                    const int ka = pa % kStagesK, kb = pb % kStagesK, va = pa % kStagesV;
                    const uint32_t kpa = (pa / kStagesK) & 1, kpb = (pb / kStagesK) & 1;
                    const uint32_t vpa = (pa / kStagesV) & 1;
                    const bool s0 = in(0, ja);      // S_0 on tile ja, then O_0 += P_0 V_ja
                    const bool s1 = in(1, ja + 1);  // S_1 on tile ja + 1
                    const bool v1 = in(1, ja);      // O_1 += P_1 V_ja (S_1 of the last iteration)
                    // K_ja was already waited for by S_1 of the last iteration
                    if (s0 && !v1) ok = wait(kBarKFull + ka, kpa);
                    if (ok && s0) issue_s(0, ka);
                    if (ok && v1) {
                        ok = wait(kBarVFull + va, vpa) && wait(kBarPFull + 1, pv_count[1] & 1);
                        if (ok && ja == U.a[1]) ok = wait(kBarOFree + 1, (epi_count[1] & 1) ^ 1);
                        if (ok) issue_pv(1, va, ja == U.a[1]);
                    }
                    if (ok && s1) {
                        ok = wait(kBarKFull + kb, kpb);
                        if (ok) issue_s(1, kb);
                    }
                    if (ok) {
                        commit(kBarKEmpty + ka);  // S_1(i - 1) and S_0(i) were K_ja's readers
                        if (i == last_s)
                            for (int t = 0; t < kQTiles; ++t) commit(kBarQEmpty + t);
                    }
                    if (ok && s0) {
                        if (!v1) ok = wait(kBarVFull + va, vpa);
                        ok = ok && wait(kBarPFull + 0, pv_count[0] & 1);
                        if (ok && ja == U.a[0]) ok = wait(kBarOFree + 0, (epi_count[0] & 1) ^ 1);
                        if (ok) issue_pv(0, va, ja == U.a[0]);
                    }
                    if (ok) commit(kBarVEmpty + va);  // both products of this iteration read V_ja
                }
            }
            for (int j = j0; !shifted && ok && j <= j1 + 1; ++j) {
                const int pos = kv_base + (j - j0);  // ring position of K_j / V_j
                const int kst = pos % kStagesK;
                const uint32_t kph = (pos / kStagesK) & 1;
                const int vst = pos % kStagesV;
                const uint32_t vph = (pos / kStagesV) & 1;
                const int pvst = (pos - 1 + kStagesV) % kStagesV;
                const uint32_t pvph = ((pos - 1) / kStagesV) & 1;
                if (j <= j1) ok = wait(kBarKFull + kst, kph);
                if (ok && in(0, j)) issue_s(0, kst);
                if (ok && in(1, j - 1)) {
                    // V_{j-1} was already waited for by O_0 += P_0(j-1) V_{j-1}
                    if (!in(0, j - 1)) ok = wait(kBarVFull + pvst, pvph);
                    ok = ok && wait(kBarPFull + 1, pv_count[1] & 1);
                    if (ok && j - 1 == U.a[1]) ok = wait(kBarOFree + 1, (epi_count[1] & 1) ^ 1);
                    if (ok) issue_pv(1, pvst, j - 1 == U.a[1]);
                }
                if (ok && in(1, j)) issue_s(1, kst);
                if (ok && j <= j1) {
                    commit(kBarKEmpty + kst);  // K_j is free once its S MMAs complete
                    if (j == j1)               // both Q buffers too
                        for (int t = 0; t < kQTiles; ++t) commit(kBarQEmpty + t);
                }
                if (ok && in(0, j)) {
                    ok = wait(kBarVFull + vst, vph) && wait(kBarPFull + 0, pv_count[0] & 1);
                    if (ok && j == U.a[0]) ok = wait(kBarOFree + 0, (epi_count[0] & 1) ^ 1);
                    if (ok) issue_pv(0, vst, j == U.a[0]);
                }
                // V_{j-1} is free once O_1 += P_1(j-1) V_{j-1} (issued above) completes.
                if (ok && j > j0) commit(kBarVEmpty + pvst);
            }
            kv_base += j1 - j0 + 1;
            for (int t = 0; t < kQTiles; ++t)
                if (U.a[t] <= U.b[t]) ++epi_count[t];
            if (!ok && lane == 0) record_timeout(p, abort_flag, kRoleMma, u);
        }
        // Drain: every MMA this warp issued has completed before TMEM is freed.
        if (elect_one()) umma_commit(bar(kBarDrain));
        __syncwarp();
        if (lane == 0) mbar_wait_bounded(bar(kBarDrain), 0, nullptr, budget);
        __syncwarp();
      }
    } else {
      setmaxnreg_inc<kRegsSoftmax>();
      {
        // ================================================================ softmax warpgroups
        const int t = warp >> 2;                 // Q tile of this warpgroup
        const int row = threadIdx.x & 127;       // TMEM lane and row of the Q tile
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t tS = tl + t * kBN;
        const uint32_t tO = tl + L::kTmemO + t * D;
        const float sl2 = p.scale_log2;
        int s_count = 0;  // S_t tiles consumed so far (= O_t += P_t V issued)
        bool ok = true;
        for (int unit_iter = 0; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarUnitFull + slot),
                                                           (unit_iter / kUnitSlots) & 1, abort_flag, budget));
            if (!ok) {
                if (lane == 0) record_timeout(p, abort_flag, kRoleSoftmax, -1);
                break;
            }
            const int u = unit_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarUnitEmpty + slot));
            if (u < 0) break;
            const auto U = decode_unit<PACKED, VARLEN>(u, p);
            if (U.a[t] > U.b[t]) continue;
            const int R = unit_rows<VARLEN>(U, p);
            const int nk = unit_keys<VARLEN>(U, p);
            const int q_off = unit_qoff<VARLEN>(U, p);
            const int rt0 = U.r0 + t * kBM;
            const int rl = min(rt0 + kBM, R) - 1;
            const int r = rt0 + row;     // row of the row space
            const int i = PACKED ? r % p.Nq : r;  // query index in its head
            int i_lo, i_hi;
            tile_queries<PACKED>(p, rt0, rl, i_lo, i_hi);
            // visible keys of query i: [i + q_off - wl, i + q_off + wr] within [0, Nk)
            const int lo_i = max(0, i + q_off - p.wl);
            const int hi_i = min(nk - 1, i + q_off + p.wr);
            const int lo_last = max(0, i_hi + q_off - p.wl);
            const int hi_first = min(nk - 1, i_lo + q_off + p.wr);
            float m = -INFINITY;  // reference max of the row, in log2 units of the scaled logits
            float l = 0.f;        // running sum of 2^(logit - m)
            for (int j = U.a[t]; j <= U.b[t]; ++j, ++s_count) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarSFull + t), s_count & 1,
                                                               abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                const int kv0 = j * kBN;
                // Tiles visible to every row of the Q tile take the unmasked instance.
                const float corr =
                    kv0 >= lo_last && kv0 + kBN - 1 <= hi_first
                        ? softmax_tile<BF16, kPChunk, false>(tS, tS, kv0, lo_i, hi_i, sl2, m, l)
                        : softmax_tile<BF16, kPChunk, true>(tS, tS, kv0, lo_i, hi_i, sl2, m, l);
                // O_t holds the sum up to block j-1: that MMA was issued before S_t(j),
                // whose completion (s_full) implies its completion.
                if (j > U.a[t] && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0 = __uint_as_float(o[e]), a1 = __uint_as_float(o[e + 1]);
                            fmul2(a0, a1, corr, corr);
                            o[e] = __float_as_uint(a0);
                            o[e + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(tO + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + t));
            }
            if (!ok) {
                if (lane == 0) record_timeout(p, abort_flag, kRoleSoftmax, u);
                break;
            }
            // ---- epilogue: O = O_t / l, LSE = ln 2 * (m + log2 l)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarODone + t), (s_count - 1) & 1,
                                                           abort_flag, budget));
            if (!ok) {
                if (lane == 0) record_timeout(p, abort_flag, kRoleSoftmax, u);
                break;
            }
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const bool store = r < R;
            // global row of O and LSE: (row space, row), or (token, head) when VARLEN
            size_t grow;
            if constexpr (VARLEN)
                grow = (static_cast<size_t>(U.q_tok0) + (store ? r : 0)) * p.H + U.h;
            else
                grow = static_cast<size_t>(U.rs) * p.R + (store ? r : 0);
            const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            bool store_ok = store;
            if constexpr (kDebugBounds) {
                grow += static_cast<size_t>(p.row_shift);
                if (store && grow >= static_cast<size_t>(p.out_rows)) {
                    store_ok = false;  // refused: recorded instead of written
                    if (atomicCAS(p.status, 0u, kStatusBounds) == 0u) {
                        p.status[1] = static_cast<unsigned>(kRoleSoftmax);
                        p.status[2] = static_cast<unsigned>(grow);
                        p.status[3] = blockIdx.x;
                        __threadfence();
                    }
                }
            }
            if (p.part_O == nullptr) {
                // O / l rounded to 16 bit, and LSE
                uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) + grow * (D * 2);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_ld_wait(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                                            __uint_as_float(o[2 * e + 1]) * inv_l);
                    if (store_ok) {
                        st_global_v8(orow + c * 64, pk);
                        st_global_v8(orow + c * 64 + 32, pk + 8);
                    }
                }
                if (store_ok) p.LSE[grow] = lse;
            } else {
                // key split: the split's own O / l in fp32 and its LSE, merged later
                const size_t prow = static_cast<size_t>(U.split) * p.BH * p.Nq + grow;
                float *orow = p.part_O + prow * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_ld_wait(o);
                    if (store_ok) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
#pragma unroll
                        for (int q = 0; q < 4; ++q) st_global_v8(orow + c * 32 + q * 8, o + q * 8);
                    }
                }
                if (store_ok) p.part_LSE[prow] = lse;
            }
            tc_fence_before();
            mbar_arrive(bar(kBarOFree + t));
        }
      }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The last CTA to finish zeroes this launch's scheduler counters for the next
    // launch that uses them (every CTA has stopped fetching units by now).
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

}  // namespace fa
