/*
 * Plain fp64 CPU attention: the oracle the GPU path is checked against.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes ("vectorized-flash-attention-kernel", Evidence & signatures:
 * the tiled kernel is checked against "standard attention"; and
 * "js-flash-attention-tiled-online-softmax-exactness", problem statement:
 * a "naive full-softmax reference").  For batch b, head h and query row i:
 *
 *   L      = clamp(kv_len[b], 0, N)            (N when kv_len is NULL)
 *   A_i    = { j : j < L  and  (not causal  or  j <= i) }
 *            (causal mask "kvRow > qRow -> -inf", Core algorithm step 2)
 *   s_j    = scale * sum_d Q[i,d] K[j,d]       (scale: Constructor options,
 *                                                default 1/sqrt(d))
 *   m      = max_{j in A_i} s_j
 *   l      = sum_{j in A_i} exp(s_j - m)
 *   O[i,:] = sum_{j in A_i} exp(s_j - m) V[j,:] / l
 *   LSE[i] = m + ln l       (the saved row statistics of "Gradient
 *                            checkpointing", folded into one number)
 *
 * A row with A_i empty gives O[i,:] = +0.0 and LSE[i] = -inf: the pages ask
 * for finite zeros on fully masked rows, also from the reference
 * ("js-flash-attention-tiled-online-softmax-exactness", Root causes 2 and
 * Verification).
 *
 * Two passes over the keys of a row with N doubles of scratch; no blocking,
 * no online rescaling, no reordering beyond the definition above.
 *
 * Inputs are float32 arrays holding the exact values the GPU sees (bf16
 * values are exactly representable in float32); every product, sum, exp and
 * log is taken in double.  Layout: contiguous [B,H,N,D] row-major, LSE
 * [B,H,N].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row.  `s` is caller scratch of at least N doubles. */
static void oracle_row(const float *Q, const float *K, const float *V,
                       int64_t N, int64_t D, int64_t head, int64_t i,
                       int64_t L, int causal, double scale, double *s,
                       double *o, double *lse)
{
    int64_t nkeys = L;
    if (causal && i + 1 < nkeys) nkeys = i + 1;
    if (nkeys <= 0) {
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    const float *q = Q + (head * N + i) * D;
    const float *k0 = K + head * N * D;
    const float *v0 = V + head * N * D;

    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const float *k = k0 + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += (double)q[d] * (double)k[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const float *v = v0 + j * D;
        for (int64_t d = 0; d < D; ++d) o[d] += s[j] * (double)v[d];
    }
    for (int64_t d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
}

static int64_t key_length(const int32_t *kv_len, int64_t b, int64_t N)
{
    if (!kv_len) return N;
    int64_t L = kv_len[b];
    if (L < 0) L = 0;
    if (L > N) L = N;
    return L;
}

/*
 * Selected rows: the same definition, for chosen rows only, so that a large
 * problem can be checked row by row.  rows[r] is the flat row index
 * (b*H + h)*N + i of batch b, head h, query i; the outputs
 * O_rows [nrows, D] and LSE_rows [nrows] are fp64.  Returns 0, or -1 on a bad
 * argument.  nthreads <= 0 means the OpenMP default.
 */
int oracle_attention_rows(const float *Q, const float *K, const float *V,
                          int64_t B, int64_t H, int64_t N, int64_t D,
                          int causal, double scale, const int32_t *kv_len,
                          const int64_t *rows, int64_t nrows,
                          double *O_rows, double *LSE_rows, int nthreads)
{
    if (!Q || !K || !V || !rows || !O_rows || !LSE_rows) return -1;
    if (B < 0 || H < 0 || N < 0 || D <= 0 || nrows < 0) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            int64_t flat = rows[r];
            int64_t i = flat % N;
            int64_t head = flat / N;
            int64_t b = head / H;
            oracle_row(Q, K, V, N, D, head, i, key_length(kv_len, b, N),
                       causal, scale, s, O_rows + r * D, LSE_rows + r);
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/* Every row: O [B,H,N,D] and LSE [B,H,N], both fp64. */
int oracle_attention(const float *Q, const float *K, const float *V,
                     double *O, double *LSE,
                     int64_t B, int64_t H, int64_t N, int64_t D,
                     int causal, double scale, const int32_t *kv_len,
                     int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return -1;
    if (B < 0 || H < 0 || N < 0 || D <= 0) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int64_t total = B * H * N;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t flat = 0; flat < total; ++flat) {
            if (!s) continue;
            int64_t i = flat % N;
            int64_t head = flat / N;
            int64_t b = head / H;
            oracle_row(Q, K, V, N, D, head, i, key_length(kv_len, b, N),
                       causal, scale, s, O + flat * D, LSE + flat);
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/* Threads an OpenMP parallel region of this library would use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Backward pass of the same attention, by recomputation ("FlashAttention"
 * module F08, Math: backward pass via recomputation and the identity
 * rowsum(dP * P) = rowsum(dO * O); "vectorized-flash-attention-kernel", Key
 * design decisions 4: the saved row statistics let the backward rebuild P).
 *
 * For one (b, h), with P the masked softmax of scale * Q K^T (rows with no
 * visible key are all zero), O = P V and an upstream gradient dO:
 *
 *   dV    = P^T dO
 *   dP    = dO V^T
 *   Delta = rowsum(dO * O)            (= rowsum(dP * P))
 *   dS    = P * (dP - Delta)          (elementwise, row-broadcast Delta)
 *   dQ    = scale * dS K
 *   dK    = scale * dS^T Q
 *
 * Plain fp64, one head per OpenMP iteration, O(N) scratch per query row plus
 * the head's fp64 accumulators for dK and dV.  Inputs are float32 arrays
 * holding the exact values the GPU sees; outputs fp64 [B,H,N,D].
 */
static void oracle_bwd_head(const float *Q, const float *K, const float *V, const float *dO,
                            double *dQ, double *dK, double *dV, int64_t N, int64_t D,
                            int64_t head, int64_t L, int causal, double scale, double *p,
                            double *dp, double *o)
{
    const int64_t base = head * N * D;
    for (int64_t t = 0; t < N * D; ++t) {
        dQ[base + t] = 0.0;
        dK[base + t] = 0.0;
        dV[base + t] = 0.0;
    }
    for (int64_t i = 0; i < N; ++i) {
        int64_t n_vis = L;
        if (causal && i + 1 < n_vis) n_vis = i + 1;
        if (n_vis <= 0) continue;                 /* P row is zero: no gradient */
        const float *q = Q + base + i * D;
        const float *g = dO + base + i * D;
        /* P row: two passes as in the forward definition */
        double m = -INFINITY;
        for (int64_t j = 0; j < n_vis; ++j) {
            const float *k = K + base + j * D;
            double qk = 0.0;
            for (int64_t d = 0; d < D; ++d) qk += (double)q[d] * (double)k[d];
            p[j] = scale * qk;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < n_vis; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (int64_t j = 0; j < n_vis; ++j) p[j] /= l;
        /* O row and Delta = rowsum(dO * O) */
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < n_vis; ++j) {
            const float *v = V + base + j * D;
            for (int64_t d = 0; d < D; ++d) o[d] += p[j] * (double)v[d];
        }
        double delta = 0.0;
        for (int64_t d = 0; d < D; ++d) delta += (double)g[d] * o[d];
        /* dP row = dO_i . V_j, dS row = P * (dP - Delta) */
        for (int64_t j = 0; j < n_vis; ++j) {
            const float *v = V + base + j * D;
            double s = 0.0;
            for (int64_t d = 0; d < D; ++d) s += (double)g[d] * (double)v[d];
            dp[j] = p[j] * (s - delta);
        }
        /* accumulate dV += P^T dO, dQ = scale dS K, dK += scale dS^T Q */
        for (int64_t j = 0; j < n_vis; ++j) {
            const float *k = K + base + j * D;
            double *dvj = dV + base + j * D;
            double *dkj = dK + base + j * D;
            double *dqi = dQ + base + i * D;
            for (int64_t d = 0; d < D; ++d) {
                dvj[d] += p[j] * (double)g[d];
                dqi[d] += scale * dp[j] * (double)k[d];
                dkj[d] += scale * dp[j] * (double)q[d];
            }
        }
    }
}

int oracle_attention_bwd(const float *Q, const float *K, const float *V, const float *dO,
                         double *dQ, double *dK, double *dV,
                         int64_t B, int64_t H, int64_t N, int64_t D,
                         int causal, double scale, const int32_t *kv_len, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return -1;
    if (B < 0 || H < 0 || N < 0 || D <= 0) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        if (!p || !dp || !o) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t head = 0; head < B * H; ++head) {
            if (!p || !dp || !o) continue;
            oracle_bwd_head(Q, K, V, dO, dQ, dK, dV, N, D, head, key_length(kv_len, head / H, N),
                            causal, scale, p, dp, o);
        }
        free(p);
        free(dp);
        free(o);
    }
    return bad ? -1 : 0;
}
