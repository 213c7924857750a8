/*
 * Oracle for the gated linear attention (GLA) prefill forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (plain definition, fp64 throughout, one (batch, head) at a time):
 *
 *     S_0 = h0            (or the zero matrix when h0 is NULL)
 *     for t = 0 .. T-1:
 *         S_t = diag(exp(g_t)) . S_{t-1} + k_t^T v_t       (Dk x Dv state)
 *         o_t = scale . q_t . S_t                          (row vector, Dv)
 *     hT = S_{T-1}
 *
 * Sources (page title, section):
 *   - "Linear Attention 在 GPU 上到底慢在哪", section 学长的反馈: the state update
 *     h <- h.g + k^T v with a D x D state (D = 128). The gate multiplies the state;
 *     read here as a per-key-dimension decay alpha_t = exp(g_t) acting on the rows
 *     (the key axis) of S, g_t being the log-gate.
 *   - "线性注意力GPU算子库的定义与技术解析", section 四 (工作原理): the plain
 *     recurrence accumulates outer(k[t], v[t]) into the state first and then reads
 *     o[t] = q[t] @ state, so token t sees its own key/value (causal, diagonal
 *     included).
 *   - "面向长序列大模型的线性注意力算子性能评测方法与优化实践", section 六.1: the
 *     correctness reference is a high-precision token-by-token recurrence.
 * The output scale is applied once to the final sum (q . S), which is the same
 * number as scaling q first, up to rounding.
 *
 * Inputs are float32 (bf16 inputs are widened exactly by the caller); all
 * arithmetic and outputs are double. Row strides are in elements.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (batch, head): q,k rows of Dk floats, v rows of Dv floats, g rows of Dk floats.
 * Consecutive tokens are sq / sk / sv / sg elements apart. h0 is a row-major Dk x Dv
 * block (or NULL). o receives T rows of Dv doubles, `so` elements apart. hT (or NULL)
 * receives the row-major Dk x Dv final state. Returns 0, or -1 if scratch allocation
 * fails. */
int gla_oracle_head(const float *q, const float *k, const float *v, const float *g,
                    int64_t T, int64_t Dk, int64_t Dv,
                    int64_t sq, int64_t sk, int64_t sv, int64_t sg,
                    double scale, const float *h0, double *o, int64_t so, double *hT)
{
    double *S = (double *)malloc((size_t)(Dk * Dv) * sizeof(double));
    double *alpha = (double *)malloc((size_t)Dk * sizeof(double));
    if (!S || !alpha) { free(S); free(alpha); return -1; }
    for (int64_t i = 0; i < Dk * Dv; ++i) S[i] = h0 ? (double)h0[i] : 0.0;

    for (int64_t t = 0; t < T; ++t) {
        const float *qt = q + t * sq, *kt = k + t * sk, *vt = v + t * sv, *gt = g + t * sg;
        for (int64_t d = 0; d < Dk; ++d) alpha[d] = exp((double)gt[d]);
        /* S <- diag(alpha) S + k^T v */
        for (int64_t d = 0; d < Dk; ++d) {
            const double a = alpha[d], kd = (double)kt[d];
            double *row = S + d * Dv;
            for (int64_t e = 0; e < Dv; ++e) row[e] = a * row[e] + kd * (double)vt[e];
        }
        /* o_t = scale * q_t S */
        double *ot = o + t * so;
        for (int64_t e = 0; e < Dv; ++e) ot[e] = 0.0;
        for (int64_t d = 0; d < Dk; ++d) {
            const double qd = (double)qt[d];
            const double *row = S + d * Dv;
            for (int64_t e = 0; e < Dv; ++e) ot[e] += qd * row[e];
        }
        for (int64_t e = 0; e < Dv; ++e) ot[e] *= scale;
    }
    if (hT) memcpy(hT, S, (size_t)(Dk * Dv) * sizeof(double));
    free(S);
    free(alpha);
    return 0;
}

/* All heads of a [B,T,H,D] contiguous batch. h0/hT are [B,H,Dk,Dv] (either may be NULL).
 * o is [B,T,H,Dv] double. The (b,h) pairs are independent and run in parallel.
 * Returns 0, or -1 if any head failed. */
int gla_oracle_batch(const float *q, const float *k, const float *v, const float *g,
                     double scale, const float *h0, double *o, double *hT,
                     int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv)
{
    int err = 0;
    const int64_t n = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < n; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        const int64_t offk = (b * T * H + h) * Dk, offv = (b * T * H + h) * Dv;
        err |= gla_oracle_head(q + offk, k + offk, v + offv, g + offk, T, Dk, Dv,
                               H * Dk, H * Dk, H * Dv, H * Dk, scale,
                               h0 ? h0 + bh * Dk * Dv : NULL,
                               o + offv, H * Dv,
                               hT ? hT + bh * Dk * Dv : NULL) != 0;
    }
    return err ? -1 : 0;
}

/* Number of threads an OpenMP parallel region will use (reported by the bench). */
int gla_oracle_num_threads(void)
{
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}
