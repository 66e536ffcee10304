// fa_bwd_kernel.cuh -- attention backward for sm_103a: dQ, dK, dV from Q, K, V,
// the forward's O and LSE, and dO.
//
// Method. The forward keeps only O and the row statistics m, l (as LSE); the
// backward recomputes the scores and probabilities block by block from them
// instead of storing the N x N matrix P ("ai6s.net/6af30f4d40858c2d8819b6d5"
// §2.4, and the recomputation row of its §4.1 table). With D_i = sum_c dO_ic O_ic
// (equal to sum_j P_ij dP_ij, the row term of the softmax Jacobian):
//     P_ij = exp(s_ij - LSE_i)            dV_j += P_ij dO_i
//     dP_ij = dO_i . V_j                  dS_ij = P_ij (dP_ij - D_i)
//     dK_j += scale dS_ij Q_i             dQ_i += scale dS_ij K_j
// over the same 128 x 128 tiles and with the same causal / window block skip
// as the forward (§3.3 (4) of the same page).
//
// GPU form: three kernels.
//  * prep: per query row D_i and L_i = LSE_i log2(e) into a small workspace.
//  * dK/dV: one work unit is a 128-key block of one K/V head; its CTA keeps K_j
//    and V_j in shared memory and dK_j, dV_j in tensor memory, and walks every
//    128-row query block (of every query head reading that K/V head) that sees
//    one of its keys. Scores are formed transposed, S^T = K Q^T, so that the
//    TMEM lane is the key: P^T and dS^T are written by the threads owning the
//    key rows straight into TMEM as the A operand of dV += P^T dO and
//    dK += dS^T Q.
//  * dQ: one work unit is a 128-row query block of one head; it walks the key
//    blocks that the rows see, recomputes S = Q K^T and dP = dO V^T, forms dS in
//    TMEM and accumulates dQ += dS K there.
// Computing dQ in its own pass costs two more matrix products (S and dP are
// formed twice) but needs no atomics: on this GPU, adding the dQ tiles of every
// key block into an fp32 buffer is bounded by the L2's reduction rate (about
// 2.9 TB/s measured), which was slower than the extra products. dQ, dK and dV
// are therefore deterministic.
//
// Both main kernels: 384 threads; warps 0-7 compute (two warpgroups splitting a
// tile's 128 columns 64 / 64; thread = TMEM lane), warp 8 TMA producer, warp 9
// MMA issuer, warp 10 second TMA producer (dQ kernel) or idle, warp 11 idle
// (warpgroup 2's registers move to the compute warpgroups with setmaxnreg).
// Every wait is bounded (global-timer budget); on expiry the CTA records the
// failure in the status word, drains its copies and MMAs, frees its tensor memory
// and returns.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_mask.cuh"
#include "ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kTile = 128;     // rows of every tile (TMEM lanes)
constexpr int kThreads = 384;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTma2Warp = 10;
constexpr int kRegsCompute = 208;
constexpr int kRegsControl = 88;
constexpr int kRegsNeeded = 256 * kRegsCompute + 128 * kRegsControl;
// Tiles are stored as regions of min(d, 64) columns x 128 rows with the swizzle of
// that row width (128 B; 64 B at d = 32), as TMA writes them.
template <int D>
struct Rg {
    static constexpr int kCols = D < 64 ? D : 64;
    static constexpr int kRowBytes = kCols * 2;
    static constexpr int kBytes = 128 * kRowBytes;   // one region
    static constexpr int kCount = D / kCols;
    static constexpr int kStepsPerRegion = kCols / 16;  // K-steps of 16 columns per region
};
constexpr uint32_t kTmemCols = 512;
constexpr unsigned kStatusTimeout = 4;   // FA_ERR_TIMEOUT
constexpr int kMaxDynSmem = 232448;      // per-CTA opt-in limit of sm_100-class GPUs
enum : int { kRoleCompute = 1, kRoleTma = 2, kRoleMma = 3 };

struct BwdParams {
    void *dQ, *dK, *dV;       // dQ: B*H x N x d; dK, dV: B*H_kv x N x d (16-bit)
    const float *Lw;          // B*H x Npad: LSE * log2(e); +inf on rows past N
    const float *Dw;          // B*H x Npad: sum_c dO * O; 0 on rows past N
    int N, Npad;              // keys = queries per head, N rounded up to 128
    int H, Hkv, group;        // query heads, K/V heads, H / H_kv
    int BH, BHkv;
    int n_blk;                // 128-row blocks per head
    int n_units;              // units of the kernel this struct is passed to
    int wl, wr;               // key j visible to query i iff i - wl <= j <= i + wr
    int heavy_first;          // dQ kernel: visit a head's query blocks from the last one
    float scale_log2;         // scale * log2(e)
    float scale;
    unsigned long long wait_budget_ns;
    unsigned int *status;     // [code, role, unit, block]
    unsigned int *sched;      // this launch's {next unit, finished CTAs} counters (zero at launch)
    // Variable-length batches (kernel template flag VARLEN): token-major tensors,
    // sequence b owns query tokens cu_q[b] .. cu_q[b+1]-1 and keys cu_k[b] ..
    // cu_k[b+1]-1 (clamped to [0, total]); its queries stand at its last positions.
    // The row terms of sequence b, head h start at h * vstride + cu_pad[b] (each
    // sequence padded to 128 rows); n_blk counts blocks of the longest sequence.
    const int *cu_q, *cu_k, *cu_pad;
    int total_q, total_k, vstride;
    // Test hook (dK/dV kernel): when >= 0, every CTA skips the K/V load of its
    // unit number fault_unit, so that unit's waits run out; -1: none.
    int fault_unit;
};

// This sequence's sizes and first rows (variable-length batches only).
struct SeqInfo {
    int nq, nk, q_off, q_tok0, k_tok0, pad0;
};

__device__ __forceinline__ SeqInfo seq_info(int b, const BwdParams &p) {
    SeqInfo S;
    const int q0 = min(max(p.cu_q[b], 0), p.total_q);
    const int q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
    const int k0 = min(max(p.cu_k[b], 0), p.total_k);
    const int k1 = min(max(p.cu_k[b + 1], k0), p.total_k);
    S.nq = q1 - q0;
    S.nk = k1 - k0;
    S.q_off = S.nk - S.nq;
    S.q_tok0 = q0;
    S.k_tok0 = k0;
    S.pad0 = p.cu_pad[b];
    return S;
}

// 32 lanes x 16 consecutive 32-bit TMEM columns into registers, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Units are taken from a launch-wide counter by the TMA producer and handed to
// the other roles through a two-slot ring in shared memory (id -1 ends every
// role's loop), so that CTAs that finish early take more of the units.
constexpr int kUnitSlots = 2;

__device__ __forceinline__ void bwd_record_timeout(const BwdParams &p, volatile int *abort_flag,
                                                   int role, int unit) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0u, kStatusTimeout) == 0u) {
        p.status[1] = static_cast<unsigned>(role);
        p.status[2] = static_cast<unsigned>(unit);
        p.status[3] = blockIdx.x;
        __threadfence();
    }
}

// The last CTA to finish zeroes this launch's scheduler counters for the next
// launch that uses them (every CTA has stopped taking units by now).
__device__ __forceinline__ void release_sched(const BwdParams &p) {
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

// Query head (b * H + h) of the g-th query head reading K/V head bkv.
__device__ __forceinline__ int group_head(int bkv, int g, const BwdParams &p) {
    const int b = bkv / p.Hkv, hk = bkv - b * p.Hkv;
    return b * p.H + hk * p.group + g;
}

// =============================================================================== dK / dV
// Two rings: Q_i (with L of its rows), read by S^T(i) and last by dK += dS^T Q_i,
// and dO_i (with D of its rows), read by dP^T(i) and last by dV += P^T dO_i,
// which comes earlier. The Q ring is the deeper one: its slots are held longer.
template <int D>
struct KvSmem {
    static constexpr int kQStages = D <= 64 ? 4 : 3;
    static constexpr int kOStages = D <= 64 ? 4 : 2;
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kVecBytes = kTile * 4;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kTileBytes;
    static constexpr int kQ = kV + kTileBytes;                 // + s * kTileBytes
    static constexpr int kO = kQ + kQStages * kTileBytes;
    static constexpr int kL = kO + kOStages * kTileBytes;      // + s * kVecBytes
    static constexpr int kDv = kL + kQStages * kVecBytes;
    static constexpr int kBar = kDv + kOStages * kVecBytes;
    static constexpr int kNumBars = 32;
    static constexpr int kMisc = kBar + kNumBars * 8;          // tmem slot, abort flag, unit ring
    static constexpr int kBytes = kMisc + 16;
    // Slack to align the base to 1024 B when it fits; without it (d = 128) the
    // kernel checks the base's alignment itself.
    static constexpr int kAlloc = kBytes + 1024 <= kMaxDynSmem ? kBytes + 1024 : kBytes;
    static_assert(kBytes <= kMaxDynSmem, "shared memory");
};

constexpr unsigned kStatusLayout = 2;  // FA_ERR_UNSUPPORTED: shared memory base not 1024-aligned

enum : int {
    kKvKVFull = 0,
    kKvKVEmpty = 1,
    kKvSFull = 2,    // + S^T buffer (a second one at 29 when double-buffered)
    kKvDPFull = 3,
    kKvDone = 4,
    kKvPReady = 5,
    kKvDSReady = 6,
    kKvFree = 7,
    kKvDrain = 8,
    kKvQFull = 9,    // + Q stage (<= 4)
    kKvQEmpty = 13,
    kKvOFull = 17,   // + dO stage (<= 4)
    kKvOEmpty = 21,  // .. 24
    kKvUnitFull = 25,   // + slot (2)
    kKvUnitEmpty = 27,  // + slot (2)
    kKvSFull1 = 29,
};
constexpr int kKvUnitConsumers = 9;  // the MMA warp and the 8 compute warps

template <int D>
struct KvTmem {
    static constexpr uint32_t kS = 0;        // S^T, then P^T (16-bit) over columns 0-31, 64-95
    static constexpr uint32_t kDP = 128;     // dP^T, then dS^T (16-bit) over 128-159, 192-223
    static constexpr uint32_t kDV = 256;
    static constexpr uint32_t kDK = 256 + D;
    // d <= 64 leaves 128 columns for a second S^T buffer (query block n uses buffer
    // n mod 2), so S^T(n+2) needs only dV(n) before it, not the whole chain.
    static constexpr bool kDoubleS = D <= 64;
    static constexpr uint32_t kS1 = kDoubleS ? 256 + 2 * D : kS;
    static_assert(D == 32 || D == 64 || D == 128, "head dim");
    __device__ static constexpr uint32_t s_buf(int it) { return (kDoubleS && (it & 1)) ? kS1 : kS; }
};

// A dK/dV unit: key block kb (keys k0 .. k0+127) of K/V head bkv; the query
// blocks ib_lo .. ib_lo+nib-1 of each of the `group` query heads reading that
// head see one of its keys: n_it = group * nib iterations. Units are numbered
// head-major, so that the CTAs running at the same time share the Q and dO of
// a few heads in L2.
struct KvUnitBase {
    int bkv, k0, ib_lo, nib, n_it;
};
template <bool VARLEN>
struct KvUnit : KvUnitBase {};
template <>
struct KvUnit<true> : KvUnitBase, SeqInfo {};

// Problem sizes of a unit: the launch's (queries and keys at the same N
// positions), or its sequence's.
template <typename U_>
__device__ __forceinline__ int u_nq(const U_ &U, const BwdParams &p) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value) return U.nq;
    else return p.N;
}
template <typename U_>
__device__ __forceinline__ int u_nk(const U_ &U, const BwdParams &p) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value) return U.nk;
    else return p.N;
}
template <typename U_>
__device__ __forceinline__ int u_qoff(const U_ &U) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value) return U.q_off;
    else return 0;
}

// n_it = 0 marks a unit without work (a key block past its sequence's end).
template <bool VARLEN>
__device__ __forceinline__ KvUnit<VARLEN> decode_kv_unit(int u, const BwdParams &p) {
    KvUnit<VARLEN> U;
    U.bkv = u / p.n_blk;
    U.k0 = (u - U.bkv * p.n_blk) * kTile;
    if constexpr (VARLEN) static_cast<SeqInfo &>(U) = seq_info(U.bkv / p.Hkv, p);
    const int nq = u_nq(U, p), nk = u_nk(U, p), q_off = u_qoff(U);
    const int k1 = min(U.k0 + kTile, nk) - 1;
    const int q_lo = max(0, U.k0 - q_off - p.wr);
    const int q_hi = min(nq - 1, k1 - q_off + p.wl);
    U.ib_lo = q_lo / kTile;
    U.nib = q_hi / kTile - U.ib_lo + 1;
    U.n_it = (U.k0 < nk && q_lo <= q_hi) ? p.group * U.nib : 0;
    return U;
}

template <typename U_>
__device__ __forceinline__ void kv_unit_iter(const U_ &U, int n, const BwdParams &p, int &bh,
                                             int &i0) {
    const int g = n / U.nib;
    bh = group_head(U.bkv, g, p);
    i0 = (U.ib_lo + (n - g * U.nib)) * kTile;
}

// Row of the row-term vectors (L, D) for query row i0 of query head bh.
template <typename U_>
__device__ __forceinline__ size_t vec_row(const U_ &U, int bh, int i0, const BwdParams &p) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value)
        return static_cast<size_t>(bh % p.H) * p.vstride + U.pad0 + i0;
    else
        return static_cast<size_t>(bh) * p.Npad + i0;
}

// TMA coordinates (y, z) of a 128-row Q / dO tile and of a K / V tile: dense maps
// are (d, N, heads), variable-length maps (d, heads, tokens).
template <typename U_>
__device__ __forceinline__ void q_coords(const U_ &U, int bh, int i0, const BwdParams &p, int &y,
                                         int &z) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value) {
        y = bh % p.H;
        z = U.q_tok0 + i0;
    } else {
        y = i0;
        z = bh;
    }
}
template <typename U_>
__device__ __forceinline__ void kv_coords(const U_ &U, int bkv, int k0, const BwdParams &p, int &y,
                                          int &z) {
    if constexpr (std::is_base_of<SeqInfo, U_>::value) {
        y = bkv % p.Hkv;
        z = U.k_tok0 + k0;
    } else {
        y = k0;
        z = bkv;
    }
}

// Per query block n of a unit the MMA warp issues
//     S^T(n), dP^T(n) ... dV += P^T(n) dO(n) | S^T(n+1) | dK += dS^T(n) Q(n) | dP^T(n+1)
// S^T(n+1) overwrites the P^T(n) that the dV product before it reads, and
// dP^T(n+1) the dS^T(n) of the dK product before it: tcgen05.mma operations of
// one thread execute in issue order, so each read precedes the later write.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
    using L = KvSmem<D>;
    using T = KvTmem<D>;
    using G = Rg<D>;
    constexpr int kRegions = G::kCount;
    constexpr int kQS = L::kQStages;
    constexpr int kOS = L::kOStages;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(smem_raw);
    if constexpr (L::kAlloc > L::kBytes)
        smem = reinterpret_cast<uint8_t *>(
            (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    // The 128-byte swizzle needs 1024-byte aligned tiles. Uniform exit before any
    // barrier or tensor-memory allocation if the base is not.
    if ((sbase & 1023u) != 0u) {
        if (threadIdx.x == 0 && atomicCAS(p.status, 0u, kStatusLayout) == 0u) {
            p.status[3] = blockIdx.x;
            __threadfence();
        }
        return;
    }
    const uint32_t sK = sbase + L::kK;
    const uint32_t sV = sbase + L::kV;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::kMisc + 8);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    // Ring slot of query block `it` (counted over this CTA's whole sequence).
    auto sQ = [sbase](int it) { return sbase + L::kQ + (it % kQS) * L::kTileBytes; };
    auto sdO = [sbase](int it) { return sbase + L::kO + (it % kOS) * L::kTileBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.wait_budget_ns;

    // ---- setup
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == kTmaWarp * 32) {
        mbar_init(bar(kKvKVFull), 1);
        mbar_init(bar(kKvKVEmpty), 1);
        for (int s = 0; s < kQS; ++s) {
            mbar_init(bar(kKvQFull + s), 1);
            mbar_init(bar(kKvQEmpty + s), 1);
        }
        for (int s = 0; s < kOS; ++s) {
            mbar_init(bar(kKvOFull + s), 1);
            mbar_init(bar(kKvOEmpty + s), 1);
        }
        mbar_init(bar(kKvSFull), 1);
        mbar_init(bar(kKvSFull1), 1);
        mbar_init(bar(kKvDPFull), 1);
        mbar_init(bar(kKvDone), 1);
        mbar_init(bar(kKvPReady), 256);
        mbar_init(bar(kKvDSReady), 256);
        mbar_init(bar(kKvFree), 256);
        mbar_init(bar(kKvDrain), 1);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(bar(kKvUnitFull + k), 1);
            mbar_init(bar(kKvUnitEmpty + k), kKvUnitConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
      setmaxnreg_dec<kRegsControl>();
      if (warp == kTmaWarp) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int it = 0, unit_iter = 0, kv_loads = 0, q_loads = 0;
            bool ok = true;
            auto publish = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kKvUnitEmpty + slot), ((k / kUnitSlots) & 1) ^ 1,
                                       abort_flag, budget);
                if (!ok) return -1;
                unsigned next = atomicAdd(p.sched, 1u);
                if constexpr (VARLEN)  // key blocks past their sequence's end have no work
                    while (next < static_cast<unsigned>(p.n_units) &&
                           decode_kv_unit<VARLEN>(static_cast<int>(next), p).n_it == 0)
                        next = atomicAdd(p.sched, 1u);
                const int v = next < static_cast<unsigned>(p.n_units) ? static_cast<int>(next) : -1;
                unit_ring[slot] = v;
                mbar_arrive(bar(kKvUnitFull + slot));
                return v;
            };
            int u = publish(0);
            for (; ok && u >= 0; ++unit_iter) {
                const auto U = decode_kv_unit<VARLEN>(u, p);
                ok = mbar_wait_bounded(bar(kKvKVEmpty), (unit_iter & 1) ^ 1, abort_flag, budget);
                if (!ok) break;
                if (unit_iter != p.fault_unit) {
                    mbar_arrive_expect_tx(bar(kKvKVFull), 2 * L::kTileBytes);
                    int ky, kz;
                    kv_coords(U, U.bkv, U.k0, p, ky, kz);
                    for (int g = 0; g < kRegions; ++g) {
                        tma_load_3d(sK + g * G::kBytes, &tmK, bar(kKvKVFull), G::kCols * g, ky, kz);
                        tma_load_3d(sV + g * G::kBytes, &tmV, bar(kKvKVFull), G::kCols * g, ky, kz);
                    }
                }
                ++kv_loads;
                // Claim the next unit now; its K and V go to L2 while this unit runs
                // (their shared-memory load waits for this unit's last products).
                const int u_next = publish(unit_iter + 1);
                if (!ok) break;
                if (u_next >= 0) {
                    const auto W = decode_kv_unit<VARLEN>(u_next, p);
                    int wy, wz;
                    kv_coords(W, W.bkv, W.k0, p, wy, wz);
                    for (int g = 0; g < kRegions; ++g) {
                        tma_prefetch_l2_3d(&tmK, G::kCols * g, wy, wz);
                        tma_prefetch_l2_3d(&tmV, G::kCols * g, wy, wz);
                    }
                }
                for (int n = 0; ok && n < U.n_it; ++n, ++it) {
                    int bh, i0;
                    kv_unit_iter(U, n, p, bh, i0);
                    const size_t vrow = vec_row(U, bh, i0, p);
                    int qy, qz;
                    q_coords(U, bh, i0, p, qy, qz);
                    // Q_i and L of its rows
                    const int qs = it % kQS;
                    ok = mbar_wait_bounded(bar(kKvQEmpty + qs), ((it / kQS) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    uint32_t fb = bar(kKvQFull + qs);
                    mbar_arrive_expect_tx(fb, L::kTileBytes + L::kVecBytes);
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sQ(it) + g * G::kBytes, &tmQ, fb, G::kCols * g, qy, qz);
                    bulk_load(sbase + L::kL + qs * L::kVecBytes, p.Lw + vrow, L::kVecBytes, fb);
                    ++q_loads;
                    // dO_i and D of its rows
                    const int os = it % kOS;
                    ok = mbar_wait_bounded(bar(kKvOEmpty + os), ((it / kOS) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    fb = bar(kKvOFull + os);
                    mbar_arrive_expect_tx(fb, L::kTileBytes + L::kVecBytes);
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(sdO(it) + g * G::kBytes, &tmdO, fb, G::kCols * g, qy, qz);
                    bulk_load(sbase + L::kDv + os * L::kVecBytes, p.Dw + vrow, L::kVecBytes, fb);
                }
                u = u_next;
            }
            if (!ok) bwd_record_timeout(p, abort_flag, kRoleTma, u);
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            // q_loads Q copies and `it` dO copies were issued (q_loads = it + 1 if the
            // loop broke between the two).
            if (kv_loads > 0)
                mbar_wait_bounded(bar(kKvKVFull), (kv_loads - 1) & 1, nullptr, budget);
            for (int s = 0; s < kQS; ++s) {
                if (q_loads > s) {
                    const int last = q_loads - 1 - ((q_loads - 1 - s) % kQS);
                    mbar_wait_bounded(bar(kKvQFull + s), (last / kQS) & 1, nullptr, budget);
                }
            }
            for (int s = 0; s < kOS; ++s) {
                if (it > s) {
                    const int last = it - 1 - ((it - 1 - s) % kOS);
                    mbar_wait_bounded(bar(kKvOFull + s), (last / kOS) & 1, nullptr, budget);
                }
            }
        }
      } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc_kk = idesc_f16_ab(BF16, kTile, kTile, false, false);
        constexpr uint32_t idesc_tn = idesc_f16_ab(BF16, kTile, D, false, true);
        constexpr uint32_t kRegion16 = G::kBytes >> 4;
        constexpr uint32_t kKStep16 = (16 * G::kRowBytes) >> 4;  // 16 rows of the tile
        auto wait = [&](int b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag, budget));
        };
        auto commit = [&](int b) {
            if (elect_one()) umma_commit(bar(b));
            __syncwarp();
        };
        // C[128 x 128] = A B^T with A, B both K-major (rows of d): S^T = K Q^T, dP^T = V dO^T.
        auto issue_kk = [&](uint32_t a_s, uint32_t b_s, uint32_t dcol) {
            tc_fence_after();
            const uint64_t da = swz_desc<G::kRowBytes>(a_s, 16);
            const uint64_t db = swz_desc<G::kRowBytes>(b_s, 16);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / G::kStepsPerRegion) * kRegion16 +
                                         (k % G::kStepsPerRegion) * 2;
                    umma_f16_ss(tmem + dcol, da + off, db + off, idesc_kk, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
        };
        // C[128 x d] (+)= A^T B with A^T in TMEM (the query pairs of warpgroup w at
        // columns acol + 64 w ...) and B MN-major in shared memory (rows = queries).
        auto issue_tn = [&](uint32_t acol, uint32_t b_s, uint32_t dcol, bool accumulate) {
            tc_fence_after();
            const uint64_t db = swz_desc<G::kRowBytes>(b_s, G::kBytes);
            const uint32_t acc0 = accumulate ? 1u : 0u;
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kTile / 16; ++k) {
                    const uint32_t ac = acol + (k < 4 ? 8 * k : 64 + 8 * (k - 4));
                    umma_f16_ts(tmem + dcol, tmem + ac, db + k * kKStep16, idesc_tn,
                                k > 0 ? 1u : acc0);
                }
            }
            __syncwarp();
        };
        int it = 0, unit_iter = 0, u = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = wait(kKvUnitFull + slot, (unit_iter / kUnitSlots) & 1);
            if (!ok) break;
            u = unit_ring[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(kKvUnitEmpty + slot));
            __syncwarp();
            if (u < 0) break;
            const auto U = decode_kv_unit<VARLEN>(u, p);
            auto qfull = [&](int i) { return wait(kKvQFull + i % kQS, (i / kQS) & 1); };
            auto ofull = [&](int i) { return wait(kKvOFull + i % kOS, (i / kOS) & 1); };
            // S^T(i) into its buffer, completion on that buffer's barrier
            auto issue_sT = [&](int i) {
                issue_kk(sK, sQ(i), T::s_buf(i));
                commit(T::kDoubleS && (i & 1) ? kKvSFull1 : kKvSFull);
            };
            ok = wait(kKvKVFull, unit_iter & 1);
            // prologue: S^T and dP^T of the unit's first query block (and S^T of the
            // second one when S^T is double-buffered)
            if (ok) ok = qfull(it);
            if (!ok) break;
            issue_sT(it);
            ok = ofull(it);
            if (!ok) break;
            issue_kk(sV, sdO(it), T::kDP);
            commit(kKvDPFull);
            if (T::kDoubleS && U.n_it > 1) {
                ok = qfull(it + 1);
                if (!ok) break;
                issue_sT(it + 1);
            }
            for (int n = 0; ok && n < U.n_it; ++n, ++it) {
                ok = wait(kKvPReady, it & 1);
                if (ok && n == 0 && unit_iter > 0) ok = wait(kKvFree, (unit_iter - 1) & 1);
                if (!ok) break;
                issue_tn(T::s_buf(it), sdO(it), T::kDV, n > 0);  // dV += P^T dO
                commit(kKvOEmpty + it % kOS);                    // dO(n), D no longer read
                if (!T::kDoubleS && n + 1 < U.n_it) {
                    ok = qfull(it + 1);
                    if (!ok) break;
                    issue_sT(it + 1);  // S^T(n+1) over P^T(n), after dV read it
                }
                ok = wait(kKvDSReady, it & 1);
                if (!ok) break;
                issue_tn(T::kDP, sQ(it), T::kDK, n > 0);  // dK += dS^T Q
                commit(kKvQEmpty + it % kQS);             // Q(n), L no longer read
                if (n + 1 < U.n_it) {
                    ok = ofull(it + 1);
                    if (!ok) break;
                    issue_kk(sV, sdO(it + 1), T::kDP);  // dP^T(n+1)
                    commit(kKvDPFull);
                }
                if (T::kDoubleS && n + 2 < U.n_it) {
                    ok = qfull(it + 2);
                    if (!ok) break;
                    issue_sT(it + 2);  // into the buffer of S^T(n), after dV(n)
                }
            }
            if (!ok) break;
            commit(kKvKVEmpty);  // K, V free once the unit's products complete
            commit(kKvDone);     // and dK, dV are final
        }
        if (!ok && lane == 0) bwd_record_timeout(p, abort_flag, kRoleMma, u);
        // Drain: every MMA this warp issued has completed before TMEM is freed.
        if (elect_one()) umma_commit(bar(kKvDrain));
        __syncwarp();
        if (lane == 0) mbar_wait_bounded(bar(kKvDrain), 0, nullptr, budget);
        __syncwarp();
      }
    } else {
      setmaxnreg_inc<kRegsCompute>();
      {
        // ================================================================ compute warpgroups
        const int wg = warp >> 2;                // query columns 64 wg .. 64 wg + 63
        const int r = threadIdx.x & 127;         // key row
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        int it = 0, unit_iter = 0, u = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kKvUnitFull + slot),
                                                           (unit_iter / kUnitSlots) & 1, abort_flag, budget));
            if (!ok) break;
            u = unit_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kKvUnitEmpty + slot));
            if (u < 0) break;
            const auto U = decode_kv_unit<VARLEN>(u, p);
            const int key = U.k0 + r;
            const bool key_ok = key < u_nk(U, p);
            const int q_off = u_qoff(U);
            for (int n = 0; n < U.n_it; ++n, ++it) {
                int bh, i0;
                kv_unit_iter(U, n, p, bh, i0);
                const float *sLw =
                    reinterpret_cast<const float *>(smem + L::kL + (it % kQS) * L::kVecBytes) + 64 * wg;
                const float *sDw =
                    reinterpret_cast<const float *>(smem + L::kDv + (it % kOS) * L::kVecBytes) + 64 * wg;
                // Element masks unless every (query, key) pair of the tile is visible.
                const bool boundary =
                    !(i0 + kTile - 1 + q_off - p.wl <= U.k0 && U.k0 + kTile - 1 <= i0 + q_off + p.wr);
                const int q0 = i0 + 64 * wg + q_off;  // key position of the first column's query
                // ---- P^T = 2^(S^T * scale * log2 e - LSE * log2 e)
                const uint32_t sb = T::s_buf(it);
                const int sfb = T::kDoubleS && (it & 1) ? kKvSFull1 : kKvSFull;
                const uint32_t sph = T::kDoubleS ? (it >> 1) & 1 : it & 1;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(sfb), sph, abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                float pr[64];
                {
                    uint32_t a[32], b[32];
                    tmem_ld32(tl + sb + 64 * wg, a);
                    tmem_ld32(tl + sb + 64 * wg + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        pr[c] = __uint_as_float(a[c]);
                        pr[c + 32] = __uint_as_float(b[c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 lw = *reinterpret_cast<const float4 *>(sLw + c);
                    ffma2(pr[c], pr[c + 1], sl2, sl2, -lw.x, -lw.y);
                    ffma2(pr[c + 2], pr[c + 3], sl2, sl2, -lw.z, -lw.w);
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) pr[c] = ex2_approx(pr[c]);
                // column c is query position q0 + c: visible iff key - wr <= q0 + c <= key + wl
                if (boundary) mask_outside_run(pr, key - p.wr - q0, key + p.wl - q0, 0.f);
                if (!key_ok) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) pr[c] = 0.f;
                }
                {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = pack2<BF16>(pr[2 * e], pr[2 * e + 1]);
                    tmem_st16(tl + sb + 64 * wg, pk);
                    tmem_st16(tl + sb + 64 * wg + 16, pk + 16);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kKvPReady));
                // ---- dS^T = P^T (dP^T - D)
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kKvDPFull), it & 1, abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t a[32], b[32];
                    tmem_ld32(tl + T::kDP + 64 * wg, a);
                    tmem_ld32(tl + T::kDP + 64 * wg + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float4 dw = *reinterpret_cast<const float4 *>(sDw + c);
                        const uint32_t *src = c < 32 ? a + c : b + (c - 32);
                        float d0 = __uint_as_float(src[0]), d1 = __uint_as_float(src[1]);
                        float d2 = __uint_as_float(src[2]), d3 = __uint_as_float(src[3]);
                        fadd2(d0, d1, -dw.x, -dw.y);
                        fadd2(d2, d3, -dw.z, -dw.w);
                        fmul2(d0, d1, pr[c], pr[c + 1]);
                        fmul2(d2, d3, pr[c + 2], pr[c + 3]);
                        pr[c] = d0;
                        pr[c + 1] = d1;
                        pr[c + 2] = d2;
                        pr[c + 3] = d3;
                    }
                }
                {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = pack2<BF16>(pr[2 * e], pr[2 * e + 1]);
                    tmem_st16(tl + T::kDP + 64 * wg, pk);
                    tmem_st16(tl + T::kDP + 64 * wg + 16, pk + 16);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kKvDSReady));
            }
            if (!ok) break;
            // ---- epilogue of the unit: warpgroup 0 stores dV, warpgroup 1 dK * scale
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kKvDone), unit_iter & 1, abort_flag, budget));
            if (!ok) break;
            tc_fence_after();
            {
                const float f = wg == 0 ? 1.f : p.scale;
                size_t orow;
                if constexpr (VARLEN)
                    orow = static_cast<size_t>(U.k_tok0 + (key_ok ? key : 0)) * p.Hkv + U.bkv % p.Hkv;
                else
                    orow = static_cast<size_t>(U.bkv) * p.N + (key_ok ? key : 0);
                uint8_t *out = reinterpret_cast<uint8_t *>(wg == 0 ? p.dV : p.dK) + orow * (D * 2);
                const uint32_t col = wg == 0 ? T::kDV : T::kDK;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t a[32];
                    tmem_ld32(tl + col + c * 32, a);
                    tmem_ld_wait(a);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * f, __uint_as_float(a[2 * e + 1]) * f);
                    if (key_ok) {
                        st_global_v8(out + c * 64, pk);
                        st_global_v8(out + c * 64 + 32, pk + 8);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(kKvFree));
        }
        if (!ok && lane == 0) bwd_record_timeout(p, abort_flag, kRoleCompute, u);
      }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    release_sched(p);
}

// =============================================================================== dQ
template <int D>
struct QSmem {
    // K and V rings: K_j is read by S(j) and, later, by dQ += dS K_j, so its ring
    // is one deeper than V's (V_j is read by dP(j) only).
    static constexpr int kKStages = D <= 64 ? 4 : 3;
    static constexpr int kVStages = D <= 64 ? 4 : 2;
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kdO = kQ + kTileBytes;
    static constexpr int kK = kdO + kTileBytes;
    static constexpr int kV = kK + kKStages * kTileBytes;
    static constexpr int kBar = kV + kVStages * kTileBytes;
    static constexpr int kNumBars = 32;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= kMaxDynSmem, "shared memory");
};

enum : int {
    kQQFull = 0,
    kQQEmpty = 1,
    kQSFull = 2,     // + S buffer (2)
    kQDPFull = 4,
    kQDSReady = 5,
    kQDone = 6,
    kQFree = 7,
    kQDrain = 8,
    kQKFull = 9,     // + stage (<= 4)
    kQKEmpty = 13,   // + stage
    kQVFull = 17,    // + stage
    kQVEmpty = 21,   // .. 24
    kQUnitFull = 25,   // + slot (2)
    kQUnitEmpty = 27,  // + slot (2)
};
constexpr int kQUnitConsumers = 10;  // the MMA warp, the V producer warp, the 8 compute warps

template <int D>
struct QTmem {
    static constexpr uint32_t kS = 0;        // S buffers b = 0, 1 at 128 b; dS (16-bit) over their columns 0-31, 64-95
    static constexpr uint32_t kDP = 256;
    static constexpr uint32_t kDQ = 384;
    static_assert(D == 32 || D == 64 || D == 128, "head dim");
};

// A dQ unit: query block (rows i0 .. i0+127) of query head bh and the key blocks
// j0 .. j1 that hold a key one of its rows sees. Units are numbered head-major;
// with heavy_first the blocks of a head run from the last one (most keys under
// a causal mask) to the first.
struct QUnitBase {
    int bh, bkv, i0, j0, j1;
};
template <bool VARLEN>
struct QUnit : QUnitBase {};
template <>
struct QUnit<true> : QUnitBase, SeqInfo {};

// j1 < j0 marks a unit without work (a query block past its sequence's end).
template <bool VARLEN>
__device__ __forceinline__ QUnit<VARLEN> decode_q_unit(int u, const BwdParams &p) {
    QUnit<VARLEN> U;
    U.bh = u / p.n_blk;
    int ib = u - U.bh * p.n_blk;
    if (p.heavy_first) ib = p.n_blk - 1 - ib;
    const int b = U.bh / p.H, h = U.bh - b * p.H;
    U.bkv = b * p.Hkv + h / p.group;
    if constexpr (VARLEN) static_cast<SeqInfo &>(U) = seq_info(b, p);
    const int nq = u_nq(U, p), nk = u_nk(U, p), q_off = u_qoff(U);
    U.i0 = ib * kTile;
    const int i1 = min(U.i0 + kTile, nq) - 1;
    const int lo = max(0, U.i0 + q_off - p.wl), hi = min(nk - 1, i1 + q_off + p.wr);
    U.j0 = lo / kTile;
    U.j1 = (U.i0 < nq && lo <= hi) ? hi / kTile : U.j0 - 1;
    return U;
}

// Per key block j (global iteration t) the MMA warp issues
//     ... dQ += dS(t) K(t) | dP(t+1) | S(t+2)
// with two S buffers, so that S(t+1) is ready when the compute warps finish
// iteration t. S(t+2) reuses the buffer of S(t), whose dS the dQ product before
// it reads (in-order execution), and dP(t+1) overwrites dP(t) only after the
// compute warps reported dS(t) (and so have read dP(t)).
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const BwdParams p) {
    using L = QSmem<D>;
    using T = QTmem<D>;
    using G = Rg<D>;
    constexpr int kRegions = G::kCount;
    constexpr int kKS = L::kKStages;
    constexpr int kVS = L::kVStages;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::kQ;
    const uint32_t sdO = sbase + L::kdO;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::kMisc + 8);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    auto sK = [sbase](int st) { return sbase + L::kK + st * L::kTileBytes; };
    auto sV = [sbase](int st) { return sbase + L::kV + st * L::kTileBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.wait_budget_ns;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == kTmaWarp * 32) {
        mbar_init(bar(kQQFull), 1);
        mbar_init(bar(kQQEmpty), 1);
        mbar_init(bar(kQSFull + 0), 1);
        mbar_init(bar(kQSFull + 1), 1);
        mbar_init(bar(kQDPFull), 1);
        mbar_init(bar(kQDSReady), 256);
        mbar_init(bar(kQDone), 1);
        mbar_init(bar(kQFree), 256);
        mbar_init(bar(kQDrain), 1);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(bar(kQUnitFull + k), 1);
            mbar_init(bar(kQUnitEmpty + k), kQUnitConsumers);
        }
        for (int s = 0; s < kKS; ++s) {
            mbar_init(bar(kQKFull + s), 1);
            mbar_init(bar(kQKEmpty + s), 1);
        }
        for (int s = 0; s < kVS; ++s) {
            mbar_init(bar(kQVFull + s), 1);
            mbar_init(bar(kQVEmpty + s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
      setmaxnreg_dec<kRegsControl>();
      if (warp == kTmaWarp || warp == kTma2Warp) {
        // ================================================================ TMA producers
        // warp 8: Q, dO and the K ring; warp 10: the V ring.
        if (lane == 0) {
            const bool kq = warp == kTmaWarp;
            const int nst = kq ? kKS : kVS;
            const int full0 = kq ? kQKFull : kQVFull, empty0 = kq ? kQKEmpty : kQVEmpty;
            const CUtensorMap *map = kq ? &tmK : &tmV;
            int t = 0, unit_iter = 0, q_loads = 0;
            bool ok = true;
            // warp 8 claims units and publishes them; warp 10 takes them like the other roles
            auto publish = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kQUnitEmpty + slot), ((k / kUnitSlots) & 1) ^ 1,
                                       abort_flag, budget);
                if (!ok) return -1;
                unsigned next = atomicAdd(p.sched, 1u);
                if constexpr (VARLEN) {  // query blocks past their sequence's end have no work
                    while (next < static_cast<unsigned>(p.n_units)) {
                        const auto W = decode_q_unit<VARLEN>(static_cast<int>(next), p);
                        if (W.j1 >= W.j0) break;
                        next = atomicAdd(p.sched, 1u);
                    }
                }
                const int v = next < static_cast<unsigned>(p.n_units) ? static_cast<int>(next) : -1;
                unit_ring[slot] = v;
                mbar_arrive(bar(kQUnitFull + slot));
                return v;
            };
            auto take = [&](int k) -> int {
                const int slot = k % kUnitSlots;
                ok = mbar_wait_bounded(bar(kQUnitFull + slot), (k / kUnitSlots) & 1, abort_flag, budget);
                if (!ok) return -1;
                const int v = unit_ring[slot];
                mbar_arrive(bar(kQUnitEmpty + slot));
                return v;
            };
            int u = kq ? publish(0) : take(0);
            for (; ok && u >= 0; ++unit_iter) {
                const auto U = decode_q_unit<VARLEN>(u, p);
                int u_next = -1;
                if (kq) {
                    ok = mbar_wait_bounded(bar(kQQEmpty), (unit_iter & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(kQQFull), 2 * L::kTileBytes);
                    int qy, qz;
                    q_coords(U, U.bh, U.i0, p, qy, qz);
                    for (int g = 0; g < kRegions; ++g) {
                        tma_load_3d(sQ + g * G::kBytes, &tmQ, bar(kQQFull), G::kCols * g, qy, qz);
                        tma_load_3d(sdO + g * G::kBytes, &tmdO, bar(kQQFull), G::kCols * g, qy, qz);
                    }
                    ++q_loads;
                    // Claim the next unit now; its Q and dO go to L2 while this unit
                    // runs (their shared-memory load waits for this unit's products).
                    u_next = publish(unit_iter + 1);
                    if (!ok) break;
                    if (u_next >= 0) {
                        const auto W = decode_q_unit<VARLEN>(u_next, p);
                        int wy, wz;
                        q_coords(W, W.bh, W.i0, p, wy, wz);
                        for (int g = 0; g < kRegions; ++g) {
                            tma_prefetch_l2_3d(&tmQ, G::kCols * g, wy, wz);
                            tma_prefetch_l2_3d(&tmdO, G::kCols * g, wy, wz);
                        }
                    }
                }
                for (int j = U.j0; ok && j <= U.j1; ++j, ++t) {
                    const int st = t % nst;
                    ok = mbar_wait_bounded(bar(empty0 + st), ((t / nst) & 1) ^ 1, abort_flag, budget);
                    if (!ok) break;
                    const uint32_t dst = kq ? sK(st) : sV(st);
                    mbar_arrive_expect_tx(bar(full0 + st), L::kTileBytes);
                    int ky, kz;
                    kv_coords(U, U.bkv, j * kTile, p, ky, kz);
                    for (int g = 0; g < kRegions; ++g)
                        tma_load_3d(dst + g * G::kBytes, map, bar(full0 + st), G::kCols * g, ky, kz);
                }
                if (!ok) break;
                if (!kq) u_next = take(unit_iter + 1);
                u = u_next;
            }
            if (!ok) bwd_record_timeout(p, abort_flag, kRoleTma, u);
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            if (q_loads > 0) mbar_wait_bounded(bar(kQQFull), (q_loads - 1) & 1, nullptr, budget);
            for (int s = 0; s < nst; ++s) {
                if (t > s) {
                    const int last = t - 1 - ((t - 1 - s) % nst);
                    mbar_wait_bounded(bar(full0 + s), (last / nst) & 1, nullptr, budget);
                }
            }
        }
      } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc_s = idesc_f16_ab(BF16, kTile, kTile, false, false);
        constexpr uint32_t idesc_q = idesc_f16_ab(BF16, kTile, D, false, true);
        constexpr uint32_t kRegion16 = G::kBytes >> 4;
        constexpr uint32_t kKStep16 = (16 * G::kRowBytes) >> 4;  // 16 rows of the tile
        auto wait = [&](int b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag, budget));
        };
        auto commit = [&](int b) {
            if (elect_one()) umma_commit(bar(b));
            __syncwarp();
        };
        // C[128 x 128] = A B^T, A (Q or dO) and B (K or V) K-major.
        auto issue_kk = [&](uint32_t a_s, uint32_t b_s, uint32_t dcol) {
            tc_fence_after();
            const uint64_t da = swz_desc<G::kRowBytes>(a_s, 16);
            const uint64_t db = swz_desc<G::kRowBytes>(b_s, 16);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / G::kStepsPerRegion) * kRegion16 +
                                         (k % G::kStepsPerRegion) * 2;
                    umma_f16_ss(tmem + dcol, da + off, db + off, idesc_s, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
        };
        // dQ (+)= dS K: dS in TMEM (keys of warpgroup w at columns acol + 64 w ...),
        // K MN-major in shared memory (rows = keys).
        auto issue_dq = [&](uint32_t acol, uint32_t k_s, bool accumulate) {
            tc_fence_after();
            const uint64_t db = swz_desc<G::kRowBytes>(k_s, G::kBytes);
            const uint32_t acc0 = accumulate ? 1u : 0u;
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < kTile / 16; ++k) {
                    const uint32_t ac = acol + (k < 4 ? 8 * k : 64 + 8 * (k - 4));
                    umma_f16_ts(tmem + T::kDQ, tmem + ac, db + k * kKStep16, idesc_q,
                                k > 0 ? 1u : acc0);
                }
            }
            __syncwarp();
        };
        auto kfull = [&](int t) { return wait(kQKFull + t % kKS, (t / kKS) & 1); };
        auto vfull = [&](int t) { return wait(kQVFull + t % kVS, (t / kVS) & 1); };
        int t = 0, unit_iter = 0, u = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = wait(kQUnitFull + slot, (unit_iter / kUnitSlots) & 1);
            if (!ok) break;
            u = unit_ring[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(kQUnitEmpty + slot));
            __syncwarp();
            if (u < 0) break;
            const auto U = decode_q_unit<VARLEN>(u, p);
            const int n = U.j1 - U.j0 + 1;
            ok = wait(kQQFull, unit_iter & 1);
            // prologue: S(t), dP(t), S(t+1)
            if (ok) ok = kfull(t);
            if (!ok) break;
            issue_kk(sQ, sK(t % kKS), T::kS + (t & 1) * 128);
            commit(kQSFull + (t & 1));
            ok = vfull(t);
            if (!ok) break;
            issue_kk(sdO, sV(t % kVS), T::kDP);
            commit(kQDPFull);
            commit(kQVEmpty + t % kVS);
            if (n > 1) {
                ok = kfull(t + 1);
                if (!ok) break;
                issue_kk(sQ, sK((t + 1) % kKS), T::kS + ((t + 1) & 1) * 128);
                commit(kQSFull + ((t + 1) & 1));
            }
            for (int x = 0; ok && x < n; ++x, ++t) {
                ok = wait(kQDSReady, t & 1);
                if (ok && x == 0 && unit_iter > 0) ok = wait(kQFree, (unit_iter - 1) & 1);
                if (!ok) break;
                issue_dq(T::kS + (t & 1) * 128, sK(t % kKS), x > 0);  // dQ += dS K
                commit(kQKEmpty + t % kKS);
                if (x + 1 < n) {
                    ok = vfull(t + 1);
                    if (!ok) break;
                    issue_kk(sdO, sV((t + 1) % kVS), T::kDP);  // dP(t+1)
                    commit(kQDPFull);
                    commit(kQVEmpty + (t + 1) % kVS);
                }
                if (x + 2 < n) {
                    ok = kfull(t + 2);
                    if (!ok) break;
                    issue_kk(sQ, sK((t + 2) % kKS), T::kS + (t & 1) * 128);  // S(t+2)
                    commit(kQSFull + (t & 1));
                }
            }
            if (!ok) break;
            commit(kQQEmpty);  // Q, dO free once the unit's products complete
            commit(kQDone);    // and dQ is final
        }
        if (!ok && lane == 0) bwd_record_timeout(p, abort_flag, kRoleMma, u);
        if (elect_one()) umma_commit(bar(kQDrain));
        __syncwarp();
        if (lane == 0) mbar_wait_bounded(bar(kQDrain), 0, nullptr, budget);
        __syncwarp();
      }
    } else {
      setmaxnreg_inc<kRegsCompute>();
      {
        // ================================================================ compute warpgroups
        const int wg = warp >> 2;                // key columns 64 wg .. 64 wg + 63
        const int r = threadIdx.x & 127;         // query row
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        int t = 0, unit_iter = 0, u = -1;
        bool ok = true;
        for (; ok; ++unit_iter) {
            const int slot = unit_iter % kUnitSlots;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kQUnitFull + slot),
                                                           (unit_iter / kUnitSlots) & 1, abort_flag, budget));
            if (!ok) break;
            u = unit_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kQUnitEmpty + slot));
            if (u < 0) break;
            const auto U = decode_q_unit<VARLEN>(u, p);
            const int i = U.i0 + r;
            const size_t vrow = vec_row(U, U.bh, U.i0, p) + r;
            const float lw = p.Lw[vrow], dw = p.Dw[vrow];
            const int nk = u_nk(U, p), q_off = u_qoff(U);
            // visible keys of query i
            const int lo_i = max(0, i + q_off - p.wl);
            const int hi_i = min(nk - 1, i + q_off + p.wr);
            const int i1 = U.i0 + kTile - 1;
            for (int j = U.j0; j <= U.j1; ++j, ++t) {
                const int k0 = j * kTile;
                // Element masks unless every pair of the tile is visible and every key exists.
                const bool boundary = !(i1 + q_off - p.wl <= k0 && k0 + kTile - 1 <= U.i0 + q_off + p.wr &&
                                        k0 + kTile <= nk);
                const int kc0 = k0 + 64 * wg;
                const uint32_t tS = tl + T::kS + (t & 1) * 128 + 64 * wg;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kQSFull + (t & 1)), (t >> 1) & 1,
                                                               abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                float pr[64];
                {
                    uint32_t a[32], b[32];
                    tmem_ld32(tS, a);
                    tmem_ld32(tS + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        pr[c] = __uint_as_float(a[c]);
                        pr[c + 32] = __uint_as_float(b[c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; c += 2) ffma2(pr[c], pr[c + 1], sl2, sl2, -lw, -lw);
#pragma unroll
                for (int c = 0; c < 64; ++c) pr[c] = ex2_approx(pr[c]);
                if (boundary) mask_outside_run(pr, lo_i - kc0, hi_i - kc0, 0.f);
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kQDPFull), t & 1, abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t a[32], b[32];
                    tmem_ld32(tl + T::kDP + 64 * wg, a);
                    tmem_ld32(tl + T::kDP + 64 * wg + 32, b);
                    tmem_ld_wait(a);
                    tmem_ld_wait(b);
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const uint32_t *src = c < 32 ? a + c : b + (c - 32);
                        float d0 = __uint_as_float(src[0]), d1 = __uint_as_float(src[1]);
                        fadd2(d0, d1, -dw, -dw);
                        fmul2(d0, d1, pr[c], pr[c + 1]);
                        pr[c] = d0;
                        pr[c + 1] = d1;
                    }
                }
                {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = pack2<BF16>(pr[2 * e], pr[2 * e + 1]);
                    tmem_st16(tS, pk);
                    tmem_st16(tS + 16, pk + 16);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kQDSReady));
            }
            if (!ok) break;
            // ---- epilogue: dQ * scale, rounded to 16 bit; warpgroup w stores columns w d/2 ..
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kQDone), unit_iter & 1, abort_flag, budget));
            if (!ok) break;
            tc_fence_after();
            {
                const bool store = i < u_nq(U, p);
                size_t orow;
                if constexpr (VARLEN)
                    orow = static_cast<size_t>(U.q_tok0 + (store ? i : 0)) * p.H + U.bh % p.H;
                else
                    orow = static_cast<size_t>(U.bh) * p.N + (store ? i : 0);
                uint8_t *out = reinterpret_cast<uint8_t *>(p.dQ) + (orow * D + wg * (D / 2)) * 2;
                if constexpr (D / 2 >= 32) {
#pragma unroll
                    for (int c = 0; c < D / 2; c += 32) {
                        uint32_t a[32];
                        tmem_ld32(tl + T::kDQ + wg * (D / 2) + c, a);
                        tmem_ld_wait(a);
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * p.scale,
                                                __uint_as_float(a[2 * e + 1]) * p.scale);
                        if (store) {
                            st_global_v8(out + c * 2, pk);
                            st_global_v8(out + c * 2 + 32, pk + 8);
                        }
                    }
                } else {
                    // d = 32: 16 columns per warpgroup
                    uint32_t a[16];
                    tmem_ld16(tl + T::kDQ + wg * (D / 2), a);
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * p.scale,
                                            __uint_as_float(a[2 * e + 1]) * p.scale);
                    if (store) st_global_v8(out, pk);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(kQFree));
        }
        if (!ok && lane == 0) bwd_record_timeout(p, abort_flag, kRoleCompute, u);
      }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    release_sched(p);
}

// =============================================================================== prep
struct PrepParams {
    const void *O, *dO;
    const float *LSE;
    float *Lw, *Dw;
    int BH, N, Npad;
};

constexpr int kPrepWarps = 8;

__device__ __forceinline__ float to_f32(uint16_t h, bool bf16) {
    return bf16 ? __bfloat162float(__ushort_as_bfloat16(h)) : __half2float(__ushort_as_half(h));
}

// One warp per (head, padded row): D = sum_c dO * O in fp32 and L = LSE * log2(e)
// (+inf for rows past N and for rows without a visible key, so that their
// recomputed probabilities are 0).
template <int D, bool BF16>
__global__ void __launch_bounds__(kPrepWarps * 32) fa_bwd_prep_kernel(const PrepParams p) {
    const int row = blockIdx.x * kPrepWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.BH * p.Npad) return;
    const int bh = row / p.Npad, i = row - bh * p.Npad;
    float dsum = 0.f;
    if (i < p.N) {
        const size_t base = (static_cast<size_t>(bh) * p.N + i) * D;
        constexpr int kPer = D / 32;  // elements per lane
        const uint16_t *o = reinterpret_cast<const uint16_t *>(p.O) + base + lane * kPer;
        const uint16_t *g = reinterpret_cast<const uint16_t *>(p.dO) + base + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e) dsum = fmaf(to_f32(g[e], BF16), to_f32(o[e], BF16), dsum);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, s);
    }
    if (lane == 0) {
        p.Dw[row] = i < p.N ? dsum : 0.f;
        const float lse = i < p.N ? p.LSE[static_cast<size_t>(bh) * p.N + i] : -INFINITY;
        p.Lw[row] = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
    }
}

// ---- variable-length batches
// Start of each sequence's row-term block: sum of the earlier sequences' query
// counts, each rounded up to 128 (one thread; cu_pad has B + 1 entries).
__global__ void fa_bwd_cu_pad_kernel(const int *cu_q, int B, int total_q, int *cu_pad) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    int acc = 0;
    for (int b = 0; b < B; ++b) {
        cu_pad[b] = acc;
        const int q0 = min(max(cu_q[b], 0), total_q);
        const int q1 = min(max(cu_q[b + 1], q0), total_q);
        acc += (q1 - q0 + kTile - 1) / kTile * kTile;
    }
    cu_pad[B] = acc;
}

struct PrepVarlenParams {
    const void *O, *dO;
    const float *LSE;        // total_q x H
    const int *cu_q, *cu_pad;
    float *Lw, *Dw;          // H x vstride
    int B, H, total_q, vstride;
};

// One warp per (head, padded row) of the row-term blocks: the row's sequence by
// binary search in cu_pad, then D and L of its token as in fa_bwd_prep_kernel;
// rows past a sequence's queries get D = 0, L = +inf.
template <int D, bool BF16>
__global__ void __launch_bounds__(kPrepWarps * 32) fa_bwd_prep_varlen_kernel(const PrepVarlenParams p) {
    const int row = blockIdx.x * kPrepWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.H * p.vstride) return;
    const int h = row / p.vstride, r = row - h * p.vstride;
    int lo = 0, hi = p.B;  // largest b with cu_pad[b] <= r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cu_pad[mid] <= r) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const int i = r - p.cu_pad[b];
    const int q0 = min(max(p.cu_q[b], 0), p.total_q);
    const int q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
    const bool valid = r < p.cu_pad[p.B] && i < q1 - q0;
    float dsum = 0.f;
    size_t t = 0;
    if (valid) {
        t = static_cast<size_t>(q0 + i) * p.H + h;  // token-major row of O, dO, LSE
        constexpr int kPer = D / 32;
        const uint16_t *o = reinterpret_cast<const uint16_t *>(p.O) + t * D + lane * kPer;
        const uint16_t *g = reinterpret_cast<const uint16_t *>(p.dO) + t * D + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e) dsum = fmaf(to_f32(g[e], BF16), to_f32(o[e], BF16), dsum);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, s);
    }
    if (lane == 0) {
        p.Dw[row] = valid ? dsum : 0.f;
        const float lse = valid ? p.LSE[t] : -INFINITY;
        p.Lw[row] = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
    }
}

}  // namespace bwd
}  // namespace fa
