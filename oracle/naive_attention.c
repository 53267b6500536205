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
 * Selected rows.  rows[r] is the flat row index (b*H + h)*N + i; the outputs
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
