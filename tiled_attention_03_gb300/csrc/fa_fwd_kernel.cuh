// fa_fwd_kernel.cuh -- attention forward for sm_103a: TMA -> shared memory ->
// tcgen05.mma with fp32 accumulators in tensor memory -> online softmax in
// registers -> O and LSE.
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
// blocks are the refinements listed at the end of §2.5. The mask variants are
// applied right after the score block is formed, as the catlass epilogue does
// ("ai6s.net/6a0ed07b662f9a54cb761aa2", Epilogue Builder).
//
// GB300 mapping of one CTA (192 threads) = one 128-row Q tile of one (b, h):
//   warp 4  : TMA producer. Q once; K_j and V_j into a 2-stage (d = 128) or
//             4-stage (d = 64) ring.
//   warp 5  : MMA issuer (one thread). S_j = Q K_j^T into one of two TMEM
//             S buffers, then O += P_{j-1} V_{j-1} into the TMEM O accumulator.
//   warps 0-3: softmax; thread t owns query row t (= TMEM lane t). Reads S_j
//             with tcgen05.ld, masks, updates m and l, writes P_j (16-bit)
//             to shared memory in the MMA's swizzled K-major layout, rescales
//             its O row in TMEM, and finally writes O / l and LSE.
// The two S buffers let the tensor core compute S_{j+1} and P_{j-1} V_{j-1}
// while the softmax warps work on S_j.
//
// Every wait is bounded (global-timer budget); on expiry the CTA records the
// failure in a status word, drains its own copies and MMAs, frees its tensor
// memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile = TMEM lanes
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kThreads = 192;     // 4 softmax warps + TMA warp + MMA warp
constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 B: one 64-column swizzle region
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;  // first TMEM column of the O accumulator

constexpr unsigned kStatusTimeout = 4;  // same value as FA_ERR_TIMEOUT
enum : int { kRoleSoftmax = 1, kRoleTma = 2, kRoleMma = 3 };

struct FwdParams {
    void *O;
    float *LSE;
    int N;            // sequence length
    int num_q_tiles;  // ceil(N / kBM)
    int heavy_first;  // 1: within a head, visit Q tiles from the last (most keys) to the first
    int wl, wr;       // key j visible to query i iff i - wl <= j <= i + wr (clamped to [0, N])
    float scale_log2; // scale * log2(e)
    unsigned long long wait_budget_ns;
    unsigned int *status;  // [code, role, iteration, block]
};

template <int D>
struct SmemLayout {
    // K/V ring depth. d = 64 takes 4 stages: it pipelines deeper and keeps the
    // footprint above half of the SM's shared memory, so that one CTA (which
    // holds all 512 TMEM columns) runs per SM.
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr int kTileBytes = kBM * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kP = kV + kStages * kTileBytes;
    static constexpr int kBar = kP + kBM * kBN * 2;
    static constexpr int kNumBars = 24;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
};

// Barrier slots (kMaxStages per ring).
constexpr int kMaxStages = 4;
enum : int {
    kBarQFull = 0,
    kBarKFull = 1,                             // + stage
    kBarVFull = kBarKFull + kMaxStages,        // + stage
    kBarKVEmpty = kBarVFull + kMaxStages,      // + stage
    kBarSFull = kBarKVEmpty + kMaxStages,      // + S buffer
    kBarSEmpty = kBarSFull + 2,                // + S buffer
    kBarPFull = kBarSEmpty + 2,
    kBarODone = kBarPFull + 1,
    kBarDrain = kBarODone + 1,
    kNumBarsUsed = kBarDrain + 1,
};

__device__ __forceinline__ void record_timeout(const FwdParams &p, volatile int *abort_flag,
                                               int role, int iteration) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0u, kStatusTimeout) == 0u) {
        p.status[1] = static_cast<unsigned>(role);
        p.status[2] = static_cast<unsigned>(iteration);
        p.status[3] = blockIdx.x;
        __threadfence();
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = SmemLayout<D>;
    constexpr int kRegions = D / 64;
    constexpr int kStages = L::kStages;
    static_assert(kStages <= kMaxStages && kNumBarsUsed <= L::kNumBars, "barrier slots");
    static_assert(D == 64 || D == 128, "head dim");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::kQ;
    const uint32_t sK = sbase + L::kK;
    const uint32_t sV = sbase + L::kV;
    const uint32_t sP = sbase + L::kP;
    const uint32_t bar0 = sbase + L::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.wait_budget_ns;

    // ---- work unit: (b*H + h, Q tile), heads outermost so that the CTAs running
    // at the same time share K/V in L2.
    const int bh = static_cast<int>(blockIdx.x) / p.num_q_tiles;
    int qt = static_cast<int>(blockIdx.x) % p.num_q_tiles;
    if (p.heavy_first) qt = p.num_q_tiles - 1 - qt;
    const int r0 = qt * kBM;
    const int r_last = min(r0 + kBM, p.N) - 1;
    // Visible key range of a row i: [max(0, i - wl), min(N - 1, i + wr)].
    const int lo_first = max(0, r0 - p.wl);
    const int hi_first = min(p.N - 1, r0 + p.wr);
    const int lo_last = max(0, r_last - p.wl);
    const int hi_last = min(p.N - 1, r_last + p.wr);
    const int j_lo = lo_first / kBN;  // K/V tiles that hold any visible key
    const int n_kv = hi_last / kBN - j_lo + 1;

    // ---- setup
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 128) {
        mbar_init(bar(kBarQFull), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarKVEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarSFull + b), 1);
            mbar_init(bar(kBarSEmpty + b), 128);
        }
        mbar_init(bar(kBarPFull), 128);
        mbar_init(bar(kBarODone), 1);
        mbar_init(bar(kBarDrain), 1);
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

    if (warp == 4) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int issued[kStages];
            for (int s = 0; s < kStages; ++s) issued[s] = 0;
            mbar_arrive_expect_tx(bar(kBarQFull), L::kTileBytes);
            for (int g = 0; g < kRegions; ++g)
                tma_load_3d(sQ + g * kRegionBytes, &tmQ, bar(kBarQFull), 64 * g, r0, bh);
            for (int it = 0; it < n_kv; ++it) {
                const int st = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait_bounded(bar(kBarKVEmpty + st), ph ^ 1, abort_flag, budget)) {
                    record_timeout(p, abort_flag, kRoleTma, it);
                    break;
                }
                const int kv0 = (j_lo + it) * kBN;
                const uint32_t kdst = sK + st * L::kTileBytes;
                const uint32_t vdst = sV + st * L::kTileBytes;
                mbar_arrive_expect_tx(bar(kBarKFull + st), L::kTileBytes);
                for (int g = 0; g < kRegions; ++g)
                    tma_load_3d(kdst + g * kRegionBytes, &tmK, bar(kBarKFull + st), 64 * g, kv0, bh);
                mbar_arrive_expect_tx(bar(kBarVFull + st), L::kTileBytes);
                for (int g = 0; g < kRegions; ++g)
                    tma_load_3d(vdst + g * kRegionBytes, &tmV, bar(kBarVFull + st), 64 * g, kv0, bh);
                issued[st] = it / kStages + 1;
            }
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            mbar_wait_bounded(bar(kBarQFull), 0, nullptr, budget);
            for (int s = 0; s < kStages; ++s) {
                if (issued[s] > 0) {
                    const uint32_t ph = (issued[s] - 1) & 1;
                    mbar_wait_bounded(bar(kBarKFull + s), ph, nullptr, budget);
                    mbar_wait_bounded(bar(kBarVFull + s), ph, nullptr, budget);
                }
            }
        }
    } else if (warp == 5) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(BF16, kBM, kBN, false);
            constexpr uint32_t idesc_o = idesc_f16(BF16, kBM, D, true);
            bool ok = mbar_wait_bounded(bar(kBarQFull), 0, abort_flag, budget);
            int it = 0;
            for (; ok && it <= n_kv; ++it) {
                if (it < n_kv) {
                    const int st = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    const int sb = it & 1;
                    ok = mbar_wait_bounded(bar(kBarKFull + st), ph, abort_flag, budget) &&
                         mbar_wait_bounded(bar(kBarSEmpty + sb), ((it >> 1) & 1) ^ 1, abort_flag,
                                           budget);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kbase = sK + st * L::kTileBytes;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * kRegionBytes + (k & 3) * 32;
                        umma_f16_ss(tmem + sb * kBN, sw128_desc(sQ + off, 16, 1024),
                                    sw128_desc(kbase + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(kBarSFull + sb));
                }
                if (it > 0) {
                    const int pj = it - 1;
                    const int pst = pj % kStages;
                    const uint32_t pph = (pj / kStages) & 1;
                    ok = mbar_wait_bounded(bar(kBarVFull + pst), pph, abort_flag, budget) &&
                         mbar_wait_bounded(bar(kBarPFull), pj & 1, abort_flag, budget);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vbase = sV + pst * L::kTileBytes;
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k) {
                        const uint32_t aoff = (k >> 2) * kRegionBytes + (k & 3) * 32;
                        const uint32_t boff = k * 16 * 128;
                        umma_f16_ss(tmem + kTmemO, sw128_desc(sP + aoff, 16, 1024),
                                    sw128_desc(vbase + boff, kRegionBytes, 1024), idesc_o,
                                    (pj > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(kBarODone));
                    umma_commit(bar(kBarKVEmpty + pst));
                }
            }
            if (!ok) record_timeout(p, abort_flag, kRoleMma, it);
            // Drain: every MMA this thread issued has completed before TMEM is freed.
            umma_commit(bar(kBarDrain));
            mbar_wait_bounded(bar(kBarDrain), 0, nullptr, budget);
        }
    } else {
        // ================================================================ softmax warps
        const int row = threadIdx.x;  // TMEM lane and row of the Q tile
        const int i = r0 + row;       // query index
        const int lo_i = max(0, i - p.wl);
        const int hi_i = min(p.N - 1, i + p.wr);
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        float m = -INFINITY;  // running max of the logits, scaled to log2 units
        float l = 0.f;        // running sum of 2^(logit - m)
        bool ok = true;
        int it = 0;
        for (; it < n_kv; ++it) {
            const int sb = it & 1;
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(bar(kBarSFull + sb), (it >> 1) & 1, abort_flag, budget));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tl + sb * kBN + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
            tc_fence_before();
            mbar_arrive(bar(kBarSEmpty + sb));  // the S buffer may be overwritten now

            float x[kBN];
#pragma unroll
            for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
            const int kv0 = (j_lo + it) * kBN;
            const bool full = kv0 >= lo_last && kv0 + kBN - 1 <= hi_first;
            if (!full) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const int key = kv0 + c;
                    if (key < lo_i || key > hi_i) x[c] = -INFINITY;
                }
            }
            float mx = x[0];
#pragma unroll
            for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, x[c]);
            const float m_new = fmaxf(m, mx * sl2);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float corr = ex2_approx(m - m_use);
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                x[c] = ex2_approx(fmaf(x[c], sl2, -m_use));
                sum += x[c];
            }
            l = l * corr + sum;
            m = m_new;

            if (it > 0) {
                // P_{j-1} V_{j-1} must be done: it reads the P buffer and writes O.
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarODone), (it - 1) & 1,
                                                               abort_flag, budget));
                if (!ok) break;
                tc_fence_after();
            }
            // P row -> shared memory, K-major with the 128-byte swizzle.
            uint8_t *prow = smem + L::kP + row * 128;
#pragma unroll
            for (int g = 0; g < kBN / 64; ++g) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int b = g * 64 + c * 8;
                    uint4 v;
                    v.x = pack2<BF16>(x[b + 0], x[b + 1]);
                    v.y = pack2<BF16>(x[b + 2], x[b + 3]);
                    v.z = pack2<BF16>(x[b + 4], x[b + 5]);
                    v.w = pack2<BF16>(x[b + 6], x[b + 7]);
                    *reinterpret_cast<uint4 *>(prow + g * kRegionBytes + ((c ^ (row & 7)) << 4)) = v;
                }
            }
            if (it > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl + kTmemO + c * 32, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    tmem_st32(tl + kTmemO + c * 32, o);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(kBarPFull));
        }
        if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarODone), (n_kv - 1) & 1,
                                                           abort_flag, budget));
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const bool store = i < p.N;
            uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) +
                            (static_cast<size_t>(bh) * p.N + (store ? i : 0)) * (D * 2);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tl + kTmemO + c * 32, o);
                tmem_ld_wait(o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                                        __uint_as_float(o[2 * e + 1]) * inv_l);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 64);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (store)
                p.LSE[static_cast<size_t>(bh) * p.N + i] =
                    l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        } else if (lane == 0) {
            record_timeout(p, abort_flag, kRoleSoftmax, it);
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace fa
