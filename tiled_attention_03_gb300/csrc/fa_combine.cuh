// fa_combine.cuh -- merge of key-split partial results (split-KV attention).
//
// With the keys of a head cut into splits s, each split yields for query row i
// its own softmax-normalised output O_s and log-sum-exp LSE_s over the keys of
// that split. The full result follows from the same rescaling the online
// softmax applies between K/V blocks ("ai6s.net/6af30f4d40858c2d8819b6d5"
// §2.3), applied once across splits:
//     LSE = ln sum_s exp(LSE_s)          O = sum_s exp(LSE_s - LSE) O_s
// computed around the largest LSE_s for range safety. This is the split
// (Flash-Decoding) variant that §5 of the same page lists after FlashAttention.
//
// One warp per query row; lane c handles columns c, c + 32, ... . Only splits
// that intersect the row's own visible key range are read (every one of them
// was written by the attention kernel, possibly as an all-masked row with
// LSE_s = -inf); the rest are never touched.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fa {

struct CombineParams {
    const float *part_O;    // [split][b*H+h][Nq][d]
    const float *part_LSE;  // [split][b*H+h][Nq]
    void *O;                // [b*H+h][Nq][d], 16-bit
    float *LSE;             // [b*H+h][Nq]
    int BH, Nq, Nk, q_off, wl, wr;
    int n_splits;
    int split_keys;  // keys per split (a multiple of the kernel's K/V tile)
};

constexpr int kCombineWarps = 8;

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineWarps * 32)
    fa_combine_kernel(const CombineParams p) {
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.BH * p.Nq) return;
    const int i = row % p.Nq;
    const int lo = max(0, i + p.q_off - p.wl);
    const int hi = min(p.Nk - 1, i + p.q_off + p.wr);
    constexpr int kCols = D / 32;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    float lse = -INFINITY;
    if (lo <= hi) {
        const int s0 = lo / p.split_keys;
        const int s1 = min(p.n_splits - 1, hi / p.split_keys);
        const size_t stride = static_cast<size_t>(p.BH) * p.Nq;  // rows per split
        float m = -INFINITY;
        for (int s = s0; s <= s1; ++s) m = fmaxf(m, p.part_LSE[s * stride + row]);
        if (m != -INFINITY) {
            float wsum = 0.f;
            for (int s = s0; s <= s1; ++s) {
                const float ls = p.part_LSE[s * stride + row];
                if (ls == -INFINITY) continue;
                const float w = expf(ls - m);
                wsum += w;
                const float *o = p.part_O + (s * stride + row) * static_cast<size_t>(D);
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, o[lane + 32 * c], acc[c]);
            }
            const float inv = 1.f / wsum;
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[c] *= inv;
            lse = m + logf(wsum);
        }
    }
    uint16_t *orow = reinterpret_cast<uint16_t *>(p.O) + static_cast<size_t>(row) * D;
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
        const uint32_t pk = pack2<BF16>(acc[c], 0.f);
        orow[lane + 32 * c] = static_cast<uint16_t>(pk & 0xffffu);
    }
    if (lane == 0) p.LSE[row] = lse;
}

}  // namespace fa
