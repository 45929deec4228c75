/*
 * attn_oracle_bwd.c -- fp64 CPU oracle for the backward pass of attention.
 *
 * TEST INFRASTRUCTURE ONLY, like attn_oracle.c: only the test suite, the
 * smoke check and the benchmark's CPU leg load it, and it shares no code with
 * the GPU library.
 *
 * What it computes.  The gradients of the forward definition in attn_oracle.c
 * (O = softmax(scale * Q K^T [+ causal mask]) V) with respect to Q, K and V,
 * given the gradient dO of a loss with respect to O.  "Optimal Software
 * Pipelining and Warp Specialization for Tensor Core GPUs" schedules the
 * FlashAttention backward kernel as well as the forward one (Sections 6.3 and
 * 6.4: register-bound on Hopper, spilling on Blackwell) but does not write the
 * gradients out; this file writes out the chain rule of the definition, in
 * double precision, per (batch, head) slice:
 *
 *     p_ij    = exp(s_ij - m_i) / l_i             (the forward's softmax row)
 *     o_i     = sum_j p_ij v_j
 *     dV_j    = sum_i p_ij dO_i                    (O is linear in V)
 *     dP_ij   = dO_i . v_j                         (dL/dp_ij)
 *     delta_i = sum_j p_ij dP_ij  = dO_i . o_i
 *     dS_ij   = p_ij (dP_ij - delta_i)             (softmax Jacobian)
 *     dQ_i    = scale * sum_j dS_ij k_j
 *     dK_j    = scale * sum_i dS_ij q_i
 *
 * with j running over the keys visible to row i (j <= i under the causal
 * mask).  Every row's softmax is recomputed here from Q and K (two passes:
 * logits and maximum, then normaliser); nothing is taken from the GPU's
 * forward.  OpenMP splits the rows; each thread accumulates its own dK, dV
 * and the partial sums are added at the end, which changes no term, only the
 * order of fp64 additions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * attn_oracle_bwd_slice -- one (batch, head) slice.
 *
 *   q, k, v, dout   S x D row-major
 *   causal          0: every key visible; 1: key j visible to query i iff j <= i
 *   scale           the softmax scale of the forward
 *   dq, dk, dv      S x D row-major outputs
 *
 * Returns 0 on success, 1 on a bad argument, 2 if scratch could not be had.
 */
int attn_oracle_bwd_slice(const double *q, const double *k, const double *v,
                          const double *dout, int64_t S, int64_t D, int causal,
                          double scale, double *dq, double *dk, double *dv)
{
    int failed = 0;
    int64_t n;

    if (S < 1 || D < 1 || !q || !k || !v || !dout || !dq || !dk || !dv)
        return 1;
    n = S * D;
    memset(dk, 0, (size_t)n * sizeof(double));
    memset(dv, 0, (size_t)n * sizeof(double));

#pragma omp parallel reduction(| : failed)
    {
        double *p = (double *)malloc((size_t)S * sizeof(double));
        double *o = (double *)malloc((size_t)D * sizeof(double));
        double *dk_t = (double *)calloc((size_t)n, sizeof(double));
        double *dv_t = (double *)calloc((size_t)n, sizeof(double));
        const int have = p && o && dk_t && dv_t;
        int64_t i;
        if (!have)
            failed = 1;
        /* every thread reaches the work-sharing loop; one without scratch
           skips its rows, and the call reports the failure */
#pragma omp for schedule(dynamic, 4)
        for (i = 0; i < S; ++i) {
            const int64_t nk = causal ? i + 1 : S;
            const double *qi = q + i * D, *doi = dout + i * D;
            double m = -INFINITY, l = 0.0, delta = 0.0;
            int64_t j, d;
            if (!have)
                continue;

            /* the forward's softmax row: logits, maximum, normaliser */
            for (j = 0; j < nk; ++j) {
                double dot = 0.0;
                for (d = 0; d < D; ++d)
                    dot += qi[d] * k[j * D + d];
                p[j] = scale * dot;
                if (p[j] > m)
                    m = p[j];
            }
            for (j = 0; j < nk; ++j) {
                p[j] = exp(p[j] - m);
                l += p[j];
            }
            for (j = 0; j < nk; ++j)
                p[j] /= l;

            /* o_i and delta_i = dO_i . o_i */
            for (d = 0; d < D; ++d)
                o[d] = 0.0;
            for (j = 0; j < nk; ++j)
                for (d = 0; d < D; ++d)
                    o[d] += p[j] * v[j * D + d];
            for (d = 0; d < D; ++d)
                delta += doi[d] * o[d];

            /* dQ_i, and this row's share of dK and dV */
            for (d = 0; d < D; ++d)
                dq[i * D + d] = 0.0;
            for (j = 0; j < nk; ++j) {
                double dp = 0.0, ds;
                for (d = 0; d < D; ++d)
                    dp += doi[d] * v[j * D + d];
                ds = p[j] * (dp - delta);
                for (d = 0; d < D; ++d) {
                    dq[i * D + d] += scale * ds * k[j * D + d];
                    dk_t[j * D + d] += scale * ds * qi[d];
                    dv_t[j * D + d] += p[j] * doi[d];
                }
            }
        }
        if (have) {
#pragma omp critical
            {
                int64_t e;
                for (e = 0; e < n; ++e) {
                    dk[e] += dk_t[e];
                    dv[e] += dv_t[e];
                }
            }
        }
        free(p);
        free(o);
        free(dk_t);
        free(dv_t);
    }
    return failed ? 2 : 0;
}
