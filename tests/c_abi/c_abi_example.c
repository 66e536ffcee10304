/*
 * c_abi_example.c -- the C ABI of include/fa.h used from plain C (no Python):
 * a causal forward and its backward on a small bf16 problem, both compared with
 * the fp64 oracle (liboracle.so, test infrastructure). Exit status 0 on success.
 *
 * Inputs come from a counter-based hash (splitmix64) mapped to [-1, 1) and
 * rounded to bf16; nothing here computes attention except the two libraries.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "fa.h"

/* the oracle's entry points (oracle/attention_oracle.c, oracle/attention_bwd_oracle.c) */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype, int64_t B,
                     int64_t H, int64_t N, int64_t d, double scale, int mask, int64_t wl,
                     int64_t wr, const int64_t *units, int64_t n_units, double *O, double *LSE,
                     double *P, int64_t bc, int nthreads);
int oracle_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         const uint16_t *dO, int dtype, int64_t B, int64_t H, int64_t Hk,
                         int64_t Nq, int64_t N, int64_t d, double scale, int mask, int64_t wl,
                         int64_t wr, const int64_t *kv, int64_t n_kv, double *dQ, double *dK,
                         double *dV, int nthreads);

enum { B = 1, H = 2, N = 300, D = 128 };

static uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

/* float32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    return (uint16_t)((v.u + 0x7FFFu + ((v.u >> 16) & 1u)) >> 16);
}

static double from_bf16(uint16_t h) {
    union { float f; uint32_t u; } v;
    v.u = (uint32_t)h << 16;
    return (double)v.f;
}

static void fill(uint16_t *x, size_t n, uint64_t stream) {
    for (size_t i = 0; i < n; ++i) {
        const uint64_t r = splitmix64((stream << 40) ^ (uint64_t)i);
        x[i] = to_bf16((float)((double)(r >> 11) * (2.0 / 9007199254740992.0) - 1.0));
    }
}

#define CHECK_CUDA(call)                                                                  \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                 \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

static double max_abs_diff_bf16(const uint16_t *got, const double *ref, size_t n, double *ref_max) {
    double err = 0.0, m = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double g = from_bf16(got[i]);
        if (!isfinite(g)) return INFINITY;
        if (fabs(g - ref[i]) > err) err = fabs(g - ref[i]);
        if (fabs(ref[i]) > m) m = fabs(ref[i]);
    }
    if (ref_max) *ref_max = m;
    return err;
}

int main(void) {
    const size_t n = (size_t)B * H * N * D, rows = (size_t)B * H * N;
    const float scale = 0.088f;
    uint16_t *q = malloc(n * 2), *k = malloc(n * 2), *v = malloc(n * 2), *dout = malloc(n * 2);
    uint16_t *o = malloc(n * 2), *dq = malloc(n * 2), *dk = malloc(n * 2), *dv = malloc(n * 2);
    float *lse = malloc(rows * 4);
    double *o_ref = malloc(n * 8), *lse_ref = malloc(rows * 8);
    double *dq_ref = malloc(n * 8), *dk_ref = malloc(n * 8), *dv_ref = malloc(n * 8);
    if (!q || !k || !v || !dout || !o || !dq || !dk || !dv || !lse || !o_ref || !lse_ref ||
        !dq_ref || !dk_ref || !dv_ref)
        return 1;
    fill(q, n, 1);
    fill(k, n, 2);
    fill(v, n, 3);
    fill(dout, n, 4);

    void *d_q, *d_k, *d_v, *d_o, *d_do, *d_dq, *d_dk, *d_dv, *ws;
    float *d_lse;
    const size_t ws_bytes = fa_backward_workspace_bytes(B, H, N, D);
    CHECK_CUDA(cudaMalloc(&d_q, n * 2));
    CHECK_CUDA(cudaMalloc(&d_k, n * 2));
    CHECK_CUDA(cudaMalloc(&d_v, n * 2));
    CHECK_CUDA(cudaMalloc(&d_o, n * 2));
    CHECK_CUDA(cudaMalloc(&d_do, n * 2));
    CHECK_CUDA(cudaMalloc(&d_dq, n * 2));
    CHECK_CUDA(cudaMalloc(&d_dk, n * 2));
    CHECK_CUDA(cudaMalloc(&d_dv, n * 2));
    CHECK_CUDA(cudaMalloc((void **)&d_lse, rows * 4));
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(d_q, q, n * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_k, k, n * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_v, v, n * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_do, dout, n * 2, cudaMemcpyHostToDevice));

    /* an invalid call enqueues nothing and says why */
    if (fa_forward(NULL, d_k, d_v, d_o, d_lse, B, H, N, D, scale, FA_MASK_CAUSAL, 0, 0, FA_DTYPE_BF16,
                   NULL) != FA_ERR_INVALID_ARG) {
        fprintf(stderr, "null Q was not rejected\n");
        return 1;
    }

    fa_status st = fa_forward(d_q, d_k, d_v, d_o, d_lse, B, H, N, D, scale, FA_MASK_CAUSAL, 0, 0,
                              FA_DTYPE_BF16, NULL);
    if (st == FA_OK)
        st = fa_backward(d_q, d_k, d_v, d_o, d_do, d_lse, d_dq, d_dk, d_dv, B, H, H, N, D, scale,
                         FA_MASK_CAUSAL, 0, 0, FA_DTYPE_BF16, ws, ws_bytes, NULL);
    if (st == FA_OK) st = fa_sync_status(NULL);
    if (st != FA_OK) {
        fprintf(stderr, "fa calls: %s\n", fa_status_string(st));
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(o, d_o, n * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(lse, d_lse, rows * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dq, d_dq, n * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dk, d_dk, n * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dv, d_dv, n * 2, cudaMemcpyDeviceToHost));

    int64_t units[3 * B * H], kv[B * H];
    for (int bh = 0; bh < B * H; ++bh) {
        units[3 * bh] = bh;
        units[3 * bh + 1] = 0;
        units[3 * bh + 2] = N;
        kv[bh] = bh;
    }
    if (oracle_attention(q, k, v, 1, B, H, N, D, scale, 1, 0, 0, units, B * H, o_ref, lse_ref,
                         NULL, 0, 0) != 0 ||
        oracle_attention_bwd(q, k, v, dout, 1, B, H, H, N, N, D, scale, 1, 0, 0, kv, B * H, dq_ref,
                             dk_ref, dv_ref, 0) != 0) {
        fprintf(stderr, "oracle call failed\n");
        return 1;
    }
    double lse_err = 0.0;
    for (size_t i = 0; i < rows; ++i)
        if (!(fabs(lse[i] - lse_ref[i]) <= lse_err)) lse_err = fabs(lse[i] - lse_ref[i]);
    double m_q, m_k, m_v;
    const double o_err = max_abs_diff_bf16(o, o_ref, n, NULL);
    const double q_err = max_abs_diff_bf16(dq, dq_ref, n, &m_q);
    const double k_err = max_abs_diff_bf16(dk, dk_ref, n, &m_k);
    const double v_err = max_abs_diff_bf16(dv, dv_ref, n, &m_v);
    printf("O %.3g  LSE %.3g  dQ %.3g/%.3g  dK %.3g/%.3g  dV %.3g/%.3g\n", o_err, lse_err, q_err,
           m_q, k_err, m_k, v_err, m_v);
    /* the bf16 bounds of the parity tests: O 2e-2 absolute, LSE 1e-3, gradients 3e-2 of the
       largest exact entry (floor 0.1) */
    if (!(o_err <= 2e-2) || !(lse_err <= 1e-3) || !(q_err <= 3e-2 * fmax(m_q, 0.1)) ||
        !(k_err <= 3e-2 * fmax(m_k, 0.1)) || !(v_err <= 3e-2 * fmax(m_v, 0.1))) {
        fprintf(stderr, "mismatch against the oracle\n");
        return 1;
    }
    printf("c_abi_example: ok\n");
    return 0;
}
