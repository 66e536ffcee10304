/*
 * attention_bwd_oracle.c -- plain, slow fp64 CPU oracle for the gradients of
 * the attention forward pass. TEST INFRASTRUCTURE ONLY (like
 * attention_oracle.c, which it is linked with): the product path never calls
 * it and shares no code with it.
 *
 * The pages state that the backward pass needs P, which the forward pass does
 * not keep, and that FlashAttention recomputes S and P from the saved O, m and
 * l ("ai6s.net/6af30f4d40858c2d8819b6d5" §2.4; also the table of §4.1). They
 * print no gradient formula, so this file takes the plainest reading: the
 * exact gradient of the forward definition (see attention_oracle.c)
 *
 *   O_i = sum_j P_ij V_j,   P_ij = exp(s_ij) / sum_k exp(s_ik),   s_ij = scale q_i . k_j
 *
 * for a loss whose gradient with respect to O is dO, written out by the chain
 * rule in fp64 from the exact 16-bit inputs:
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (Jacobian of the row softmax)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_i dS_ij Q_i
 *
 * P is built by the direct definition (row max subtracted), hidden keys have
 * P_ij = 0 and so no gradient. With grouped K/V heads, dK and dV of a K/V head
 * sum the contributions of every query head that reads it. The kernel side
 * recomputes P from the saved LSE and uses sum_c dO_ic O_ic for the row sum;
 * both equal the quantities above in exact arithmetic.
 *
 * Pins (tests/test_oracle_bwd.py): torch.autograd in float64 on the naive
 * three-matmul form; central finite differences of an independent numpy
 * forward; a two-key closed form worked by hand; invariants (keys' gradients
 * sum to zero, values' gradients sum to the summed dO, linearity in dO); the
 * uniform-score case (Q = 0).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

double oracle_fp16_to_double(uint16_t h);
double oracle_bf16_to_double(uint16_t h);

static double bwd_decode(uint16_t h, int dtype) {
    return dtype == 1 ? oracle_bf16_to_double(h) : oracle_fp16_to_double(h);
}

static int bwd_visible(int64_t pos, int64_t j, int mask, int64_t wl, int64_t wr) {
    if (mask == 1) return j <= pos;
    if (mask == 2) return j >= pos - wl && j <= pos + wr;
    return 1;
}

typedef struct {
    const uint16_t *Q, *K, *V, *dO;
    int dtype;
    int64_t H, Hk, Nq, N, d;
    double scale;
    int mask;
    int64_t wl, wr;
    const int64_t *kv; /* listed K/V heads b * Hk + hk */
    int64_t n_kv;
    double *dQ;        /* n_kv x group x Nq x d */
    double *dK, *dV;   /* this thread's partial sums: n_kv x N x d each */
    int nthreads, tid;
} bwd_job_t;

/* One task: query head g of listed K/V head t, all of its rows. */
static void bwd_task(bwd_job_t *jb, int64_t t, int64_t g, double *q, double *k, double *v,
                     double *dO, double *p, double *dp) {
    const int64_t N = jb->N, Nq = jb->Nq, d = jb->d, group = jb->H / jb->Hk;
    const int64_t bkv = jb->kv[t];
    const int64_t b = bkv / jb->Hk, hk = bkv % jb->Hk;
    const int64_t bh = b * jb->H + hk * group + g;
    for (int64_t x = 0; x < Nq * d; ++x) q[x] = bwd_decode(jb->Q[bh * Nq * d + x], jb->dtype);
    for (int64_t x = 0; x < Nq * d; ++x) dO[x] = bwd_decode(jb->dO[bh * Nq * d + x], jb->dtype);
    for (int64_t x = 0; x < N * d; ++x) k[x] = bwd_decode(jb->K[bkv * N * d + x], jb->dtype);
    for (int64_t x = 0; x < N * d; ++x) v[x] = bwd_decode(jb->V[bkv * N * d + x], jb->dtype);
    double *dq_out = jb->dQ + ((t * group + g) * Nq) * d;
    double *dk = jb->dK + t * N * d, *dv = jb->dV + t * N * d;
    for (int64_t i = 0; i < Nq; ++i) {
        const int64_t pos = i + N - Nq;
        /* row i of P by the direct definition */
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            double s = -INFINITY;
            if (bwd_visible(pos, j, jb->mask, jb->wl, jb->wr)) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];
                s = jb->scale * dot;
            }
            p[j] = s;
            if (s > m) m = s;
        }
        double *dqi = dq_out + i * d;
        for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
        if (m == -INFINITY) continue; /* no visible key: no gradient */
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (int64_t j = 0; j < N; ++j) p[j] /= l;
        /* dP_ij = dO_i . V_j and the row sum sum_j P_ij dP_ij */
        double rs = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) {
                dp[j] = 0.0;
                continue;
            }
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += dO[i * d + c] * v[j * d + c];
            dp[j] = dot;
            rs += p[j] * dot;
        }
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            const double ds = p[j] * (dp[j] - rs);
            for (int64_t c = 0; c < d; ++c) {
                dqi[c] += jb->scale * ds * k[j * d + c];
                dk[j * d + c] += jb->scale * ds * q[i * d + c];
                dv[j * d + c] += p[j] * dO[i * d + c];
            }
        }
    }
}

static void *bwd_worker(void *arg) {
    bwd_job_t *jb = (bwd_job_t *)arg;
    const int64_t N = jb->N, Nq = jb->Nq, d = jb->d, group = jb->H / jb->Hk;
    double *q = (double *)malloc((size_t)(Nq * d) * sizeof(double));
    double *dO = (double *)malloc((size_t)(Nq * d) * sizeof(double));
    double *k = (double *)malloc((size_t)(N * d) * sizeof(double));
    double *v = (double *)malloc((size_t)(N * d) * sizeof(double));
    double *p = (double *)malloc((size_t)N * sizeof(double));
    double *dp = (double *)malloc((size_t)N * sizeof(double));
    for (int64_t task = jb->tid; task < jb->n_kv * group; task += jb->nthreads)
        bwd_task(jb, task / group, task % group, q, k, v, dO, p, dp);
    free(q); free(dO); free(k); free(v); free(p); free(dp);
    return NULL;
}

/*
 * Gradients for the listed K/V heads kv[0..n_kv) (each b * Hk + hk). Q and dO
 * are B x H x Nq x d, K and V are B x Hk x N x d (16-bit, dtype 0 = fp16,
 * 1 = bf16); query head h reads K/V head h / (H / Hk) and query i stands at key
 * position i + N - Nq. Outputs (fp64): dQ n_kv x (H/Hk) x Nq x d for the query
 * heads of each listed K/V head in order, dK and dV n_kv x N x d. nthreads <= 0
 * uses all online cores. Returns 0, or -1 on a bad argument.
 */
int oracle_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         const uint16_t *dO, int dtype, int64_t B, int64_t H, int64_t Hk,
                         int64_t Nq, int64_t N, int64_t d, double scale, int mask, int64_t wl,
                         int64_t wr, const int64_t *kv, int64_t n_kv, double *dQ, double *dK,
                         double *dV, int nthreads) {
    if (!Q || !K || !V || !dO || !kv || !dQ || !dK || !dV) return -1;
    if (B < 1 || H < 1 || Nq < 1 || N < 1 || d < 1 || n_kv < 0) return -1;
    if (Hk < 1 || H % Hk != 0) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    if (mask < 0 || mask > 2) return -1;
    if (mask == 2 && (wl < 0 || wr < 0)) return -1;
    for (int64_t t = 0; t < n_kv; ++t)
        if (kv[t] < 0 || kv[t] >= B * Hk) return -1;
    const int64_t group = H / Hk, tasks = n_kv * group;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > tasks) nthreads = tasks > 0 ? (int)tasks : 1;
    const size_t per = (size_t)(n_kv * N * d);
    double *part = (double *)calloc(2 * per * (size_t)nthreads + 1, sizeof(double));
    bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)nthreads, sizeof(bwd_job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        bwd_job_t j = {Q, K, V, dO, dtype, H, Hk, Nq, N, d, scale, mask, wl, wr, kv, n_kv,
                       dQ, part + 2 * per * t, part + 2 * per * t + per, nthreads, t};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, bwd_worker, &jobs[t]);
    bwd_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    /* sum the threads' partials in thread order (deterministic) */
    for (size_t x = 0; x < per; ++x) {
        double sk = 0.0, sv = 0.0;
        for (int t = 0; t < nthreads; ++t) {
            sk += part[2 * per * t + x];
            sv += part[2 * per * t + per + x];
        }
        dK[x] = sk;
        dV[x] = sv;
    }
    free(part); free(jobs); free(th);
    return 0;
}
