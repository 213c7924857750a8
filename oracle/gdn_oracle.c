/*
 * Oracle for the gated delta rule forward pass, in plain C.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this file;
 * only the tests, the smoke check and the bench's CPU-baseline legs do. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes (fp64 throughout, one (batch, head) at a time):
 *
 *     S_0 = h0            (or the zero matrix when h0 is NULL)
 *     for t = 0 .. T-1:
 *         alpha = exp(g_t)
 *         S_t = alpha (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t   (Dk x Dv state)
 *         o_t = scale . q_t . S_t                                        (row vector, Dv)
 *     hT = S_{T-1}
 *
 * The gated delta rule: the gated-delta-network family that "面向长序列大模型的线性注意力
 * 算子性能评测方法与优化实践" (section 三.3) and "线性注意力GPU算子库的定义与技术解析"
 * (section 三) name, with the published recurrence (the pages print none). It is the same
 * token loop as oracle/gdn_ref.py's `recurrent`, written independently in C: the rank-one
 * projection is applied as S - beta k (k^T S) before the decay multiplies the result.
 *
 * Inputs are float32 (bf16 inputs are widened exactly by the caller); all arithmetic and
 * outputs are double. Row strides are in elements.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (batch, head): q, k rows of Dk floats, v rows of Dv floats, consecutive tokens sq / sk
 * / sv elements apart; g and beta one float per token, sg elements apart. h0 is a row-major
 * Dk x Dv block (or NULL). o receives T rows of Dv doubles, `so` elements apart. hT (or NULL)
 * receives the row-major Dk x Dv final state. Returns 0, or -1 if scratch allocation fails. */
int gdn_oracle_head(const float *q, const float *k, const float *v, const float *g,
                    const float *beta, int64_t T, int64_t Dk, int64_t Dv, int64_t sq, int64_t sk,
                    int64_t sv, int64_t sg, double scale, const float *h0, double *o, int64_t so,
                    double *hT)
{
    double *S = (double *)malloc((size_t)(Dk * Dv) * sizeof(double));
    double *kS = (double *)malloc((size_t)Dv * sizeof(double));
    if (!S || !kS) { free(S); free(kS); return -1; }
    for (int64_t i = 0; i < Dk * Dv; ++i) S[i] = h0 ? (double)h0[i] : 0.0;

    for (int64_t t = 0; t < T; ++t) {
        const float *qt = q + t * sq, *kt = k + t * sk, *vt = v + t * sv;
        const double alpha = exp((double)g[t * sg]), bt = (double)beta[t * sg];
        /* kS = k_t^T S_{t-1} (what the state returns under key k_t) */
        for (int64_t e = 0; e < Dv; ++e) kS[e] = 0.0;
        for (int64_t d = 0; d < Dk; ++d) {
            const double kd = (double)kt[d];
            const double *row = S + d * Dv;
            for (int64_t e = 0; e < Dv; ++e) kS[e] += kd * row[e];
        }
        /* S <- alpha (S - beta k kS) + beta k v */
        for (int64_t d = 0; d < Dk; ++d) {
            const double kd = (double)kt[d];
            double *row = S + d * Dv;
            for (int64_t e = 0; e < Dv; ++e)
                row[e] = alpha * (row[e] - bt * kd * kS[e]) + bt * kd * (double)vt[e];
        }
        /* o_t = scale * q_t S_t */
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
    free(kS);
    return 0;
}

/* All heads of a contiguous batch: q, k [B,T,H,Dk]; v [B,T,H,Dv]; g, beta [B,T,H]; h0 / hT
 * [B,H,Dk,Dv] (either may be NULL); o [B,T,H,Dv] double. The (b,h) pairs are independent
 * and run in parallel. Returns 0, or -1 if any head failed. */
int gdn_oracle_batch(const float *q, const float *k, const float *v, const float *g,
                     const float *beta, double scale, const float *h0, double *o, double *hT,
                     int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv)
{
    int err = 0;
    const int64_t n = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < n; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        const int64_t offk = (b * T * H + h) * Dk, offv = (b * T * H + h) * Dv;
        const int64_t offg = b * T * H + h;
        err |= gdn_oracle_head(q + offk, k + offk, v + offv, g + offg, beta + offg, T, Dk, Dv,
                               H * Dk, H * Dk, H * Dv, H, scale,
                               h0 ? h0 + bh * Dk * Dv : NULL, o + offv, H * Dv,
                               hT ? hT + bh * Dk * Dv : NULL) != 0;
    }
    return err ? -1 : 0;
}
