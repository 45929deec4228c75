/*
 * attn_oracle.c -- fp64 CPU oracle for the fused attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker for the
 * CUDA path: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no code, header, table or helper with the
 * GPU library, and the GPU library never calls it.
 *
 * What it computes.  The pages split attention into three stages: the first
 * tensor-core stage Q K^T (T), a CUDA-core stage softmax (C) and the second
 * tensor-core stage P V (U) -- "Tawa: Automatic Warp Specialization for Modern
 * GPUs with Asynchronous References", Section III-D, Algorithm 1 (coarse-grained
 * CUDA/Tensor Core pipeline), where attention is the worked example of a
 * T -> C -> U loop.  The pages do not write the formula out; this file uses the
 * textbook definition of scaled-dot-product attention with an optional causal
 * (lower-triangular) mask and the per-row natural log-sum-exp of the scaled
 * logits:
 *
 *     s_ij   = scale * sum_d q[i,d] * k[j,d]              (stage T)
 *     J_i    = {0..S-1}            (no mask)
 *            = {0..i}              (causal mask, key j visible iff j <= i)
 *     m_i    = max_{j in J_i} s_ij                         (stage C)
 *     l_i    = sum_{j in J_i} exp(s_ij - m_i)
 *     LSE_i  = m_i + ln(l_i)
 *     O[i,:] = sum_{j in J_i} exp(s_ij - m_i) * v[j,:] / l_i   (stage U)
 *
 * It is evaluated exactly as written, in double precision, with a two-pass
 * (not online) softmax: first every logit of the row, then its maximum, then
 * the normaliser, then the weighted sum of V rows.  No tiling, no fusion, no
 * rescaling tricks.  Rows are independent, so OpenMP splits the rows of a call
 * across host threads; that changes no arithmetic of any single row.
 *
 * Layout: one (batch, head) slice at a time, row-major S x D doubles for K and
 * V, row-major n_rows x D doubles for the query rows that are evaluated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row i of one head.  s_buf holds n_keys doubles of scratch. */
static void oracle_one_row(const double *q_i, const double *k, const double *v,
                           int64_t n_keys, int64_t D, double scale,
                           double *s_buf, double *o_i, double *lse_i)
{
    int64_t j, d;
    double m, l;

    /* stage T: the scaled logits s_ij = scale * <q_i, k_j> for visible j */
    for (j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (d = 0; d < D; ++d)
            dot += q_i[d] * k[j * D + d];
        s_buf[j] = scale * dot;
    }

    /* stage C, pass 1: the row maximum over the visible keys */
    m = -INFINITY;
    for (j = 0; j < n_keys; ++j)
        if (s_buf[j] > m)
            m = s_buf[j];

    /* stage C, pass 2: unnormalised weights exp(s_ij - m_i) and their sum */
    l = 0.0;
    for (j = 0; j < n_keys; ++j) {
        s_buf[j] = exp(s_buf[j] - m);
        l += s_buf[j];
    }

    /* stage U: O[i,:] = sum_j w_ij v[j,:] / l_i */
    for (d = 0; d < D; ++d)
        o_i[d] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        const double w = s_buf[j];
        for (d = 0; d < D; ++d)
            o_i[d] += w * v[j * D + d];
    }
    for (d = 0; d < D; ++d)
        o_i[d] /= l;

    *lse_i = m + log(l);
}

/*
 * attn_oracle_rows -- evaluate selected rows of one (batch, head) slice.
 *
 *   q      n_rows x D   the query rows to evaluate (row r is query index rows[r])
 *   k, v   S x D        the full key and value matrices of the slice
 *   rows   n_rows       the query index i of each evaluated row, 0 <= i < S
 *   causal 0: every key visible; 1: key j visible to query i iff j <= i
 *   scale  the softmax scale applied to q.k
 *   o      n_rows x D   output rows
 *   lse    n_rows       output natural log-sum-exp of the scaled logits
 *
 * Returns 0 on success, 1 on a bad argument, 2 if scratch could not be had.
 */
int attn_oracle_rows(const double *q, const double *k, const double *v,
                     int64_t S, int64_t D, const int64_t *rows, int64_t n_rows,
                     int causal, double scale, double *o, double *lse)
{
    int64_t r;
    int failed = 0;

    if (S < 1 || D < 1 || n_rows < 0 || !q || !k || !v || !rows || !o || !lse)
        return 1;
    for (r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= S)
            return 1;

#pragma omp parallel reduction(| : failed)
    {
        double *s_buf = (double *)malloc((size_t)S * sizeof(double));
        if (!s_buf) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (r = 0; r < n_rows; ++r) {
                const int64_t i = rows[r];
                const int64_t n_keys = causal ? i + 1 : S;
                oracle_one_row(q + r * D, k, v, n_keys, D, scale, s_buf,
                               o + r * D, lse + r);
            }
            free(s_buf);
        }
    }
    return failed ? 2 : 0;
}

/*
 * attn_oracle_full -- every row of every (batch, head) slice.
 *
 *   q, k, v  BH x S x D   contiguous, one slice per (batch, head)
 *   o        BH x S x D
 *   lse      BH x S
 */
int attn_oracle_full(const double *q, const double *k, const double *v,
                     int64_t BH, int64_t S, int64_t D, int causal, double scale,
                     double *o, double *lse)
{
    int64_t bh, i;
    int rc = 0;
    int64_t *rows;

    if (BH < 0 || S < 1 || D < 1)
        return 1;
    rows = (int64_t *)malloc((size_t)S * sizeof(int64_t));
    if (!rows)
        return 2;
    for (i = 0; i < S; ++i)
        rows[i] = i;
    for (bh = 0; bh < BH && rc == 0; ++bh) {
        const int64_t off = bh * S * D;
        rc = attn_oracle_rows(q + off, k + off, v + off, S, D, rows, S, causal,
                              scale, o + off, lse + bh * S);
    }
    free(rows);
    return rc;
}

/* Number of host threads an oracle call will use (1 without OpenMP). */
int attn_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
