// fa_mask.cuh -- element masks of a score block whose visible columns form one
// run [clo, chi] per row (every mask of the method does: the causal and window
// masks of "ai6s.net/6a0ed07b662f9a54cb761aa2" (使用) hide keys before i - wl and
// after i + wr, and keys past the sequence end are hidden too, so a row of a
// block sees a contiguous range of its columns).
#pragma once

#include <cstdint>

namespace fa {

// Bit b set <=> column 32 w + b of the block lies in [clo, chi].
__device__ __forceinline__ uint32_t visible_bits(int clo, int chi, int w) {
    const int lo = clo - 32 * w, hi = chi - 32 * w;
    uint32_t v = lo <= 0 ? 0xffffffffu : (lo >= 32 ? 0u : 0xffffffffu << lo);
    v &= hi >= 31 ? 0xffffffffu : (hi < 0 ? 0u : 0xffffffffu >> (31 - hi));
    return v;
}

// x[c] = fill for every column c of the block outside [clo, chi]. The run is
// turned into one visibility word per 32 columns; each column then costs a test
// of a constant bit and a select (comparing every column with both bounds costs
// several more instructions per column).
template <int N>
__device__ __forceinline__ void mask_outside_run(float (&x)[N], int clo, int chi, float fill) {
    static_assert(N % 32 == 0, "whole words of columns");
#pragma unroll
    for (int w = 0; w < N / 32; ++w) {
        const uint32_t vis = visible_bits(clo, chi, w);
#pragma unroll
        for (int b = 0; b < 32; ++b)
            if (!(vis & (1u << b))) x[32 * w + b] = fill;
    }
}

}  // namespace fa
