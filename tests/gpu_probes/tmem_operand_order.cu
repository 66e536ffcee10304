// Hardware-assumption probe for the attention kernel's MMA schedule.
//
// The kernel issues S_t(j+1) = Q K^T right after O_t += P_t(j) V_j, where P_t(j) is the A
// operand of the second MMA and lives in the TMEM columns the first MMA overwrites. That is
// correct when one thread's tcgen05.mma operations execute in issue order (no write-after-
// read hazard in an in-order pipeline). This probe checks it: P = all ones (bf16) in TMEM
// columns [0, 64), V in shared memory with V[k][c] = (k mod 8) / 8, then O = P V followed at
// once by an MMA that writes fp32 values over columns [0, 128). O must equal 56 everywhere.
// Every wait is bounded; the program prints the count of wrong elements.
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime.h>
#include "ptx.cuh"
using namespace fa;

__global__ void __launch_bounds__(128, 1) war(int iters, unsigned int *bad, float *osample) {
    extern __shared__ uint8_t raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t slot;
    // V: 128 keys x 128 d, MN-major SW128 layout (two 16 KB regions of 64 d); value V[k][c] = (k % 8) * 0.125
    // -> sum over 128 keys = 16 * (0+1+...+7) * 0.125 = 56 for every column (exact in fp32)
    // A/B for the SS MMA: random bf16 in [1, 2)
    uint32_t seed = 99u + threadIdx.x * 7919u + blockIdx.x * 104729u;
    for (int i = threadIdx.x; i < 32768 / 2; i += blockDim.x) {   // V region: 32 KB = 16384 u16
        const int byte = i * 2;
        const int region = byte / 16384, within = byte % 16384;
        const int k = within / 128;                 // key row
        (void)region;
        const float val = (k % 8) * 0.125f;
        const uint32_t bits = __float_as_uint(val) >> 16;  // exact in bf16
        ((uint16_t *)smem)[i] = (uint16_t)bits;
    }
    for (int i = threadIdx.x; i < 32768 / 4; i += blockDim.x) {    // A, B for SS: 32 KB after V
        seed = seed * 1664525u + 1013904223u;
        ((uint32_t *)(smem + 32768))[i] = 0x3f803f80u | (seed & 0x007f007fu);
    }
    if (threadIdx.x < 32) { tmem_alloc(smem_u32(&slot), 512); tmem_relinquish(); }
    if (threadIdx.x == 0) { mbar_init(smem_u32(&bar), 1); fence_mbar_init(); }
    fence_proxy_async_smem();
    tc_fence_before(); __syncthreads(); tc_fence_after();
    const uint32_t tmem = slot;
    const uint32_t tl = tmem + ((uint32_t)((threadIdx.x >> 5) * 32) << 16);
    const uint32_t sV = smem_u32(smem), sA = sV + 32768, sB = sA + 16384;
    const uint64_t dv = sw128_desc(sV, 16384, 1024);
    const uint64_t da = sw128_desc(sA, 16, 1024), db = sw128_desc(sB, 16, 1024);
    constexpr uint32_t idesc_o = idesc_f16(true, 128, 128, true);
    constexpr uint32_t idesc_s = idesc_f16(true, 128, 128, false);
    uint32_t ones[32];
    for (int e = 0; e < 32; ++e) ones[e] = 0x3f803f80u;  // two bf16 1.0
    unsigned int nbad = 0;
    for (int it = 0; it < iters; ++it) {
        // P = ones over cols [0, 64)
        tmem_st32(tl + 0, ones); tmem_st32(tl + 32, ones);
        tmem_st_wait();
        tc_fence_before(); __syncthreads(); tc_fence_after();
        if (threadIdx.x == 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                umma_f16_ts(tmem + 256, tmem + k * 8, dv + k * ((16 * 128) >> 4), idesc_o, k > 0 ? 1u : 0u);
            // immediately overwrite S/P columns [0,128)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_f16_ss(tmem + 0, da + k * 2, db + k * 2, idesc_s, k > 0 ? 1u : 0u);
            umma_commit(smem_u32(&bar));
            if (!mbar_wait_bounded(smem_u32(&bar), it & 1, nullptr, 2000000000ull)) atomicAdd(bad, 1000000);
        }
        __syncthreads();
        tc_fence_after();
        uint32_t o[32];
        for (int c = 0; c < 4; ++c) {
            tmem_ld32(tl + 256 + 32 * c, o); tmem_ld_wait(o);
            for (int e = 0; e < 32; ++e) if (__uint_as_float(o[e]) != 56.0f) ++nbad;
            if (it == 0 && blockIdx.x == 0 && threadIdx.x == 0 && c == 0) osample[0] = __uint_as_float(o[0]);
        }
        tc_fence_before(); __syncthreads(); tc_fence_after();
    }
    if (nbad) atomicAdd(bad, nbad);
    tc_fence_before(); __syncthreads();
    if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

int main(int argc, char **argv) {
    int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    unsigned int *d_bad; float *d_s;
    cudaMalloc(&d_bad, 4); cudaMemset(d_bad, 0, 4); cudaMalloc(&d_s, 4);
    cudaFuncSetAttribute(war, cudaFuncAttributeMaxDynamicSharedMemorySize, 140 * 1024);
    const int iters = argc > 1 ? atoi(argv[1]) : 2000;
    war<<<sms, 128, 140 * 1024>>>(iters, d_bad, d_s);
    cudaError_t e = cudaDeviceSynchronize();
    unsigned int bad = 0; float s = 0;
    cudaMemcpy(&bad, d_bad, 4, cudaMemcpyDeviceToHost); cudaMemcpy(&s, d_s, 4, cudaMemcpyDeviceToHost);
    printf("WAR test: %d CTAs x %d iterations, bad elements %u, sample O %.3f [%s]\n", sms, iters, bad, s, cudaGetErrorString(e));
    return 0;
}
