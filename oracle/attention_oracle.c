/*
 * attention_oracle.c -- plain, slow fp64 CPU oracle for the attention forward
 * pass. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product path never does, and it
 * shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, which the tiled method reaches up to
 * rounding, as the pages state in "ai6s.net/6af30f4d40858c2d8819b6d5" §2.3 and
 * §1, and "aicoding.csdn.net/6a69d3ff10ee7a33f2941f44" "attention计算到底卡在哪"):
 *
 *   s_ij  = scale * sum_k Q[i,k] K[j,k]          (fp64, from the exact 16-bit inputs)
 *   s_ij  = -inf  when key j is not visible to query i
 *   m_i   = max_j s_ij
 *   P_ij  = exp(s_ij - m_i) / sum_j exp(s_ij - m_i)
 *   O_i   = sum_j P_ij V[j,:]
 *   LSE_i = m_i + log sum_j exp(s_ij - m_i)
 *
 * Visibility: none -> every key 0..Nk-1; causal -> j <= i + off; window ->
 * i + off - wl <= j <= i + off + wr (both ends inclusive; the reading taken for
 * the (window_left, window_right) tuple of "ai6s.net/6a0ed07b662f9a54cb761aa2",
 * section "使用：ops-transformer 怎么调 FlashAttention"). off = Nk - Nq places
 * the Nq queries at the last Nq key positions (off = 0 when Nq = Nk).
 *
 * A second entry point restates the online-softmax recurrence of
 * "ai6s.net/6af30f4d40858c2d8819b6d5" §2.3 (running max m, running sum l,
 * correction factor exp(m_old - m_new)) and the C snippet of
 * "aicoding.csdn.net/6a69d3ff10ee7a33f2941f44" section "Online softmax算法",
 * in fp64 with a caller-chosen key-block size Bc. It exists only so that tests
 * can check that recurrence against the direct definition.
 *
 * Pins (tests/test_oracle.py): 16-bit decoding against numpy/torch for all
 * 65536 patterns; brute force against an independent numpy three-matmul form;
 * uniform scores (closed form: mean of visible V, LSE = ln #visible); a
 * dominant key; rows of P summing to 1; affine V; mask invariance; key
 * permutation; logit shift; the online recurrence equal to the direct form.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_FP16 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_MASK_NONE = 0, ORACLE_MASK_CAUSAL = 1, ORACLE_MASK_WINDOW = 2 };

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x400), e - 25); /* (1024+f) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double: bfloat16 is the upper half of an IEEE 754 binary32
 * (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits). */
double oracle_bf16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x80), e - 134); /* (128+f) * 2^(e-127-7) */
    }
    return sign ? -v : v;
}

static double decode(uint16_t h, int dtype) {
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(h) : oracle_fp16_to_double(h);
}

/* pos = i + off: the key position of query i */
static int is_visible(int64_t pos, int64_t j, int mask, int64_t wl, int64_t wr) {
    if (mask == ORACLE_MASK_CAUSAL) return j <= pos;
    if (mask == ORACLE_MASK_WINDOW) return j >= pos - wl && j <= pos + wr;
    return 1;
}

typedef struct {
    const uint16_t *Q, *K, *V;
    int dtype;
    int64_t H, Hk, Nq, N, d; /* query heads, K/V heads, query rows, keys (N), head dim */
    double scale;
    int mask;
    int64_t wl, wr;
    const int64_t *units; /* n_units x 3: (b*H + h, row0, row1) */
    const int64_t *out_row; /* first output row of each unit */
    int64_t n_units;
    double *O, *LSE, *P; /* P may be NULL */
    int64_t bc;          /* 0: direct form; >0: online recurrence with blocks of bc keys */
    int nthreads;
    int tid;
} job_t;

/* Decode one (b,h) slab of N x d 16-bit values into doubles. */
static void decode_slab(const uint16_t *src, int dtype, int64_t n, double *dst) {
    for (int64_t t = 0; t < n; ++t) dst[t] = decode(src[t], dtype);
}

/* The direct definition for rows [r0, r1) of one (b,h): S and P are built
 * explicitly as a (r1-r0) x N fp64 matrix. */
static void unit_direct(const job_t *jb, const double *q, const double *k, const double *v,
                        int64_t r0, int64_t r1, double *O, double *LSE, double *P,
                        double *S) {
    const int64_t N = jb->N, d = jb->d;
    for (int64_t i = r0; i < r1; ++i) {
        double *srow = S + (i - r0) * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            double s = -INFINITY;
            if (is_visible(i + jb->N - jb->Nq, j, jb->mask, jb->wl, jb->wr)) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];
                s = jb->scale * dot;
            }
            srow[j] = s;
            if (s > m) m = s;
        }
        double *orow = O + (i - r0) * d;
        for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
        if (m == -INFINITY) { /* no visible key: empty softmax */
            LSE[i - r0] = -INFINITY;
            if (P) for (int64_t j = 0; j < N; ++j) P[(i - r0) * N + j] = 0.0;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            srow[j] = exp(srow[j] - m); /* exp(-inf) = 0 for hidden keys */
            l += srow[j];
        }
        for (int64_t j = 0; j < N; ++j) srow[j] /= l; /* srow now holds P_i */
        for (int64_t j = 0; j < N; ++j) {
            double p = srow[j];
            if (p == 0.0) continue;
            for (int64_t c = 0; c < d; ++c) orow[c] += p * v[j * d + c];
        }
        LSE[i - r0] = m + log(l);
        if (P) memcpy(P + (i - r0) * N, srow, (size_t)N * sizeof(double));
    }
}

/* The online recurrence, key blocks of bc, for rows [r0, r1). */
static void unit_online(const job_t *jb, const double *q, const double *k, const double *v,
                        int64_t r0, int64_t r1, double *O, double *LSE, double *sblk) {
    const int64_t N = jb->N, d = jb->d, bc = jb->bc;
    for (int64_t i = r0; i < r1; ++i) {
        double m = -INFINITY, l = 0.0;
        double *acc = O + (i - r0) * d;
        for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
        for (int64_t j0 = 0; j0 < N; j0 += bc) {
            int64_t j1 = j0 + bc < N ? j0 + bc : N;
            double bmax = -INFINITY;
            for (int64_t j = j0; j < j1; ++j) {
                double s = -INFINITY;
                if (is_visible(i + jb->N - jb->Nq, j, jb->mask, jb->wl, jb->wr)) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];
                    s = jb->scale * dot;
                }
                sblk[j - j0] = s;
                if (s > bmax) bmax = s;
            }
            double m_new = m > bmax ? m : bmax;
            if (m_new == -INFINITY) continue; /* nothing visible yet */
            double corr = exp(m - m_new);     /* exp(-inf) = 0 on the first visible block */
            double bsum = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] *= corr;
            for (int64_t j = j0; j < j1; ++j) {
                double p = exp(sblk[j - j0] - m_new);
                bsum += p;
                if (p != 0.0)
                    for (int64_t c = 0; c < d; ++c) acc[c] += p * v[j * d + c];
            }
            l = l * corr + bsum;
            m = m_new;
        }
        if (m == -INFINITY) {
            LSE[i - r0] = -INFINITY;
            continue;
        }
        for (int64_t c = 0; c < d; ++c) acc[c] /= l;
        LSE[i - r0] = m + log(l);
    }
}

static void *worker(void *arg) {
    job_t *jb = (job_t *)arg;
    const int64_t N = jb->N, Nq = jb->Nq, d = jb->d;
    double *q = (double *)malloc((size_t)(Nq * d) * sizeof(double));
    double *k = (double *)malloc((size_t)(N * d) * sizeof(double));
    double *v = (double *)malloc((size_t)(N * d) * sizeof(double));
    int64_t maxrows = 0;
    for (int64_t u = 0; u < jb->n_units; ++u) {
        int64_t r = jb->units[3 * u + 2] - jb->units[3 * u + 1];
        if (r > maxrows) maxrows = r;
    }
    double *S = (double *)malloc((size_t)((jb->bc ? jb->bc : maxrows * N) + 1) * sizeof(double));
    int64_t cur_bh = -1;
    for (int64_t u = jb->tid; u < jb->n_units; u += jb->nthreads) {
        int64_t bh = jb->units[3 * u], r0 = jb->units[3 * u + 1], r1 = jb->units[3 * u + 2];
        if (bh != cur_bh) {
            /* query head h of batch b reads K/V head h / (H / Hk) of batch b */
            const int64_t b = bh / jb->H, h = bh % jb->H;
            const int64_t bkv = b * jb->Hk + h / (jb->H / jb->Hk);
            decode_slab(jb->Q + bh * Nq * d, jb->dtype, Nq * d, q);
            decode_slab(jb->K + bkv * N * d, jb->dtype, N * d, k);
            decode_slab(jb->V + bkv * N * d, jb->dtype, N * d, v);
            cur_bh = bh;
        }
        int64_t orow = jb->out_row[u];
        if (jb->bc)
            unit_online(jb, q, k, v, r0, r1, jb->O + orow * d, jb->LSE + orow, S);
        else
            unit_direct(jb, q, k, v, r0, r1, jb->O + orow * d, jb->LSE + orow,
                        jb->P ? jb->P + orow * N : NULL, S);
    }
    free(q); free(k); free(v); free(S);
    return NULL;
}

/*
 * Attention over a list of units (b*H+h, row0, row1). Q is B x H x Nq x d; K
 * and V are B x Hk x N x d, query head h reading K/V head h / (H / Hk) (Hk = H
 * is ordinary multi-head attention, Hk < H grouped-query attention); query i
 * stands at key position i + N - Nq. Output rows
 * are packed in unit order: O is sum(row1-row0) x d, LSE is sum(row1-row0), P
 * (optional, tiny cases only) is sum(row1-row0) x N. bc = 0 selects the direct
 * form, bc > 0 the online recurrence with key blocks of bc. nthreads <= 0 uses
 * all online cores. Returns 0, or -1 on a bad argument.
 */
int oracle_attention_ex(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                        int64_t B, int64_t H, int64_t Hk, int64_t Nq, int64_t N, int64_t d,
                        double scale, int mask, int64_t wl, int64_t wr, const int64_t *units,
                        int64_t n_units, double *O, double *LSE, double *P, int64_t bc,
                        int nthreads) {
    if (!Q || !K || !V || !units || !O || !LSE) return -1;
    if (B < 1 || H < 1 || Nq < 1 || N < 1 || d < 1 || n_units < 0 || bc < 0) return -1;
    if (Hk < 1 || H % Hk != 0) return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16) return -1;
    if (mask < ORACLE_MASK_NONE || mask > ORACLE_MASK_WINDOW) return -1;
    if (mask == ORACLE_MASK_WINDOW && (wl < 0 || wr < 0)) return -1;
    if (P && bc) return -1;
    int64_t *out_row = (int64_t *)malloc((size_t)(n_units + 1) * sizeof(int64_t));
    int64_t acc = 0;
    for (int64_t u = 0; u < n_units; ++u) {
        int64_t bh = units[3 * u], r0 = units[3 * u + 1], r1 = units[3 * u + 2];
        if (bh < 0 || bh >= B * H || r0 < 0 || r1 > Nq || r0 > r1) { free(out_row); return -1; }
        out_row[u] = acc;
        acc += r1 - r0;
    }
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? (int)n_units : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        job_t j = {Q, K, V, dtype, H, Hk, Nq, N, d, scale, mask, wl, wr, units, out_row, n_units,
                   O, LSE, P, bc, nthreads, t};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &jobs[t]);
    worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(jobs); free(th); free(out_row);
    return 0;
}

/* Grouped-query attention with Nq = N (queries at every key position). */
int oracle_attention_gqa(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                         int64_t B, int64_t H, int64_t Hk, int64_t N, int64_t d, double scale,
                         int mask, int64_t wl, int64_t wr, const int64_t *units, int64_t n_units,
                         double *O, double *LSE, double *P, int64_t bc, int nthreads) {
    return oracle_attention_ex(Q, K, V, dtype, B, H, Hk, N, N, d, scale, mask, wl, wr, units,
                               n_units, O, LSE, P, bc, nthreads);
}

/* Multi-head attention: oracle_attention_gqa with one K/V head per query head. */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                     int64_t B, int64_t H, int64_t N, int64_t d, double scale, int mask,
                     int64_t wl, int64_t wr, const int64_t *units, int64_t n_units,
                     double *O, double *LSE, double *P, int64_t bc, int nthreads) {
    return oracle_attention_gqa(Q, K, V, dtype, B, H, H, N, d, scale, mask, wl, wr, units,
                                n_units, O, LSE, P, bc, nthreads);
}
