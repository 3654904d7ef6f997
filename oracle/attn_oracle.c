/*
 * attn_oracle.c -- FP64 CPU oracle for exact masked softmax attention.
 *
 * TEST INFRASTRUCTURE. This file is the slow, plain reference that the CUDA
 * path is compared against. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline / reference arm may load it. It shares no code,
 * header, constant or helper with the CUDA library, and the CUDA library never
 * loads it.
 *
 * Sources (the pages the method is taken from):
 *   P1  "Derive online softmax, prove it is exact, and explain why it makes
 *        FlashAttention fast without reducing FLOPs"
 *        (inferenceinterviews.com/q/online-softmax-derive-and-prove-flashattention)
 *   P2  "Implement online softmax for a whole tile of queries, not one query,
 *        and write the rescaling step in matrix form"
 *        (inferenceinterviews.com/q/online-softmax-query-tile-matrix-form)
 *   P3  "Online softmax" (interview.clozo.ai/blog/online-softmax.html)
 *
 * What is computed. The pages state that the blockwise method reaches exactly
 * the plain softmax-attention result (P1 "A strong answer": o = a / l is exact;
 * P2 "A strong answer": exactness carries over row by row; P3 "Trade-offs and
 * edge cases": exact, not approximate). So the oracle is that plain definition,
 * the three-pass "safe softmax" of P3 "Step 1" followed by the weighted sum of
 * value rows of P1 "A strong answer" (first equation):
 *
 *   for each query row i of head (b, h), over the visible keys j:
 *     1. s_j  = scale * sum_t q[i,t] k[j,t]
 *     2. m    = max_j s_j
 *     3. l    = sum_j exp(s_j - m)
 *     4. p_j  = exp(s_j - m) / l
 *     5. o[t] = sum_j p_j v[j,t]
 *     6. lse  = m + log(l)        (P1 "What interviewers probe next": the
 *                                  per-row log-sum-exp m + log l)
 *
 * Inputs are FP32 arrays (BF16 or FP32 values upcast exactly); all arithmetic
 * is in double. Layout: q [B,H,Nq,d], k and v [B,H,Nk,d], row-major.
 *
 * Readings where the pages leave a step open:
 *   - Masks. Causal (P2 code/causal test): key j is visible from query i iff
 *     j <= i, query i and key j at their own indices (top-left alignment).
 *     Sliding window of W keys (named, not defined, in P2 "How to approach it"
 *     and under the m_ref guard): visible iff i - W < j <= i, i.e. it implies
 *     the causal bound. Padding: keys j >= seqlens_k[b] are invisible
 *     (seqlens_k clamped to [0, Nk]). Masks combine by AND.
 *   - A row with no visible key (P2 discusses the per-block case under the
 *     m_ref guard but not the final output): o = 0 and lse = -inf, i.e. the
 *     empty sum gives l = 0 and log(0) = -inf, and the empty weighted sum is 0.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_WINDOW 2
#define ORACLE_MASK_PADDING 4

/* Visibility of key j from query i (readings above). */
static int oracle_key_visible(long long i, long long j, long long Lk,
                              int mask_kind, long long window)
{
    if (j >= Lk) return 0;                                   /* padding    */
    if ((mask_kind & (ORACLE_MASK_CAUSAL | ORACLE_MASK_WINDOW)) && j > i)
        return 0;                                            /* causal     */
    if ((mask_kind & ORACLE_MASK_WINDOW) && j <= i - window)
        return 0;                                            /* window     */
    return 1;
}

/* One query row, the six steps of the header, in order. */
static void oracle_one_row(const float* q_row, const float* k_head,
                           const float* v_head, long long i, int Nk, int d,
                           double scale, long long Lk, int mask_kind,
                           long long window, double* s, char* vis,
                           double* o_row, double* lse_out)
{
    long long n_visible = 0;
    /* step 1: scaled dot-product scores of the visible keys */
    for (long long j = 0; j < Nk; ++j) {
        vis[j] = (char)oracle_key_visible(i, j, Lk, mask_kind, window);
        if (!vis[j]) continue;
        const float* k_row = k_head + j * (long long)d;
        double dot = 0.0;
        for (int t = 0; t < d; ++t) dot += (double)q_row[t] * (double)k_row[t];
        s[j] = scale * dot;
        ++n_visible;
    }
    for (int t = 0; t < d; ++t) o_row[t] = 0.0;
    if (n_visible == 0) {           /* no visible key: o = 0, lse = -inf */
        *lse_out = -INFINITY;
        return;
    }
    /* step 2: row maximum */
    double m = -INFINITY;
    for (long long j = 0; j < Nk; ++j)
        if (vis[j] && s[j] > m) m = s[j];
    /* step 3: normalizer referenced to the maximum */
    double l = 0.0;
    for (long long j = 0; j < Nk; ++j)
        if (vis[j]) l += exp(s[j] - m);
    /* steps 4 and 5: normalized weights, weighted sum of value rows */
    for (long long j = 0; j < Nk; ++j) {
        if (!vis[j]) continue;
        double p = exp(s[j] - m) / l;
        const float* v_row = v_head + j * (long long)d;
        for (int t = 0; t < d; ++t) o_row[t] += p * (double)v_row[t];
    }
    /* step 6: log-sum-exp */
    *lse_out = m + log(l);
}

/*
 * oracle_attn_rows: evaluate the rows listed in `rows` (flat indices
 * (b*H + h)*Nq + i), or every row in order when rows == NULL (then
 * nrows must be B*H*Nq). Outputs: o [nrows, d] and lse [nrows], double.
 * seqlens_k is read only when mask_kind has the padding bit.
 * Returns 0 on success, a negative value on an invalid argument.
 */
int oracle_attn_rows(const float* q, const float* k, const float* v,
                     int B, int H, int Nq, int Nk, int d, double scale,
                     int mask_kind, int window, const int* seqlens_k,
                     const long long* rows, long long nrows,
                     double* o, double* lse, int nthreads)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if ((mask_kind & ORACLE_MASK_WINDOW) && window <= 0) return -2;
    if ((mask_kind & ORACLE_MASK_PADDING) && seqlens_k == NULL) return -3;
    long long total = (long long)B * H * Nq;
    if (rows == NULL && nrows != total) return -4;
    if (nthreads <= 0) nthreads = 1;
    int bad = 0;

#pragma omp parallel num_threads(nthreads) reduction(| : bad)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        char* vis = (char*)malloc((size_t)(Nk > 0 ? Nk : 1));
        if (s == NULL || vis == NULL) bad = 1;
#pragma omp for schedule(dynamic, 4)
        for (long long r = 0; r < nrows; ++r) {
            if (s == NULL || vis == NULL) continue;
            long long flat = rows ? rows[r] : r;
            if (flat < 0 || flat >= total) { bad = 1; continue; }
            long long i = flat % Nq;
            long long bh = flat / Nq;
            long long b = bh / H;
            long long Lk = Nk;
            if (mask_kind & ORACLE_MASK_PADDING) {
                long long L = seqlens_k[b];
                Lk = L < 0 ? 0 : (L > Nk ? Nk : L);
            }
            oracle_one_row(q + flat * (long long)d,
                           k + bh * (long long)Nk * d,
                           v + bh * (long long)Nk * d,
                           i, Nk, d, scale, Lk, mask_kind, window,
                           s, vis, o + r * (long long)d, lse + r);
        }
        free(s);
        free(vis);
    }
    return bad ? -5 : 0;
}

/* Number of threads OpenMP would use by default (for reporting). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * oracle_softmax_rows: row softmax of x [rows, n] (FP32 values upcast to
 * double), the three-pass "safe softmax" of P3 "Step 1": the row maximum,
 * the sum of exp(x - m), then each output exp(x_i - m) / sum. Also writes the
 * row's log-sum-exp m + log(sum). Outputs in double. A row whose entries
 * are all -inf (fully masked) gives y = 0 and lse = -inf, the same reading as
 * an attention row with no visible key.
 */
int oracle_softmax_rows(const float* x, long long rows, long long n, double* y, double* lse,
                        int nthreads)
{
    if (rows < 0 || n <= 0) return -1;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
    for (long long r = 0; r < rows; ++r) {
        const float* xr = x + r * n;
        double* yr = y + r * n;
        double mx = -INFINITY;                      /* pass 1: maximum   */
        for (long long i = 0; i < n; ++i)
            if ((double)xr[i] > mx) mx = (double)xr[i];
        if (mx == -INFINITY) {          /* every entry -inf: y = 0, lse = -inf */
            for (long long i = 0; i < n; ++i) yr[i] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;                           /* pass 2: normalizer */
        for (long long i = 0; i < n; ++i) sum += exp((double)xr[i] - mx);
        for (long long i = 0; i < n; ++i)           /* pass 3: outputs    */
            yr[i] = exp((double)xr[i] - mx) / sum;
        lse[r] = mx + log(sum);
    }
    return 0;
}
