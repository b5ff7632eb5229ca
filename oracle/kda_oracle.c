/*
 * KDA reference oracle: float64, token by token, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do. It shares no code, header or constant
 * with the CUDA library.
 *
 * Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
 * (pwwt.cn/news/3763336), referred to below as the K3 essay.
 *
 *   - K3 essay §二.1: the state S_t is a d_k x d_v matrix and the read-out
 *     is o_t = S_t^T q_t (read after the update of token t).
 *   - K3 essay §三: the delta rule predicts v_hat = S^T k, forms the error
 *     e = v - v_hat and writes S + beta k e^T; the projector form
 *     (I - beta k k^T) S + beta k v^T is the same map.
 *   - K3 essay §四: KDA puts a per-channel gate in front of the delta rule,
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     with alpha_t in [0,1]^{d_k}.
 *
 * The oracle evaluates that update in its rank-1 expanded form: with
 * S' = Diag(alpha_t) S_{t-1}, the projector term is
 * S' - beta_t k_t (S'^T k_t)^T, so
 *     S_t = S' + beta_t k_t (v_t - S'^T k_t)^T,       o_t = S_t^T q_t.
 * This is the same matrix as the essay's §四 form, in O(d_k d_v) per token.
 * No chunking, blocking or reordering beyond that: token t is finished
 * before token t+1 starts, and every product is summed in index order.
 *
 * Layouts (row-major, contiguous; sequences packed along the token axis):
 *   q, k, alpha : [T_total, H, dk]      v, o : [T_total, H, dv]
 *   beta        : [T_total, H]
 *   s0, sT      : [N, H, dk, dv]        (d_v fastest)
 *   cu_seqlens  : [N + 1], sequence n owns tokens cu[n] .. cu[n+1]-1
 * s0 == NULL means a zero initial state; sT == NULL skips the final state.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (sequence, head) pair: T tokens starting at token index t0. */
static void kda_oracle_head(const double *q, const double *k, const double *v,
                            const double *alpha, const double *beta,
                            const double *s0, double *o, double *sT,
                            int64_t t0, int64_t T, int64_t H, int64_t h,
                            int64_t dk, int64_t dv, double *S, double *vhat)
{
    if (s0)
        memcpy(S, s0, (size_t)(dk * dv) * sizeof(double));
    else
        memset(S, 0, (size_t)(dk * dv) * sizeof(double));

    for (int64_t t = t0; t < t0 + T; ++t) {
        const double *kt = k + (t * H + h) * dk;
        const double *qt = q + (t * H + h) * dk;
        const double *at = alpha + (t * H + h) * dk;
        const double *vt = v + (t * H + h) * dv;
        const double bt = beta[t * H + h];
        double *ot = o + (t * H + h) * dv;

        /* S' = Diag(alpha_t) S_{t-1}  (row i of S is key channel i) */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                S[i * dv + j] *= at[i];

        /* v_hat = S'^T k_t */
        for (int64_t j = 0; j < dv; ++j)
            vhat[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                vhat[j] += S[i * dv + j] * kt[i];

        /* S_t = S' + beta_t k_t (v_t - v_hat)^T */
        for (int64_t i = 0; i < dk; ++i) {
            const double bk = bt * kt[i];
            for (int64_t j = 0; j < dv; ++j)
                S[i * dv + j] += bk * (vt[j] - vhat[j]);
        }

        /* o_t = S_t^T q_t */
        for (int64_t j = 0; j < dv; ++j)
            ot[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                ot[j] += S[i * dv + j] * qt[i];
    }

    if (sT)
        memcpy(sT, S, (size_t)(dk * dv) * sizeof(double));
}

/*
 * Runs every (sequence, head) pair. Returns 0 on success, -1 on bad
 * arguments (negative sizes, decreasing cu_seqlens), -2 when scratch
 * memory cannot be had. nthreads <= 0 lets OpenMP choose.
 */
int kda_oracle_run(const double *q, const double *k, const double *v,
                   const double *alpha, const double *beta,
                   const int32_t *cu_seqlens, int64_t N, int64_t H,
                   int64_t dk, int64_t dv, const double *s0, double *o,
                   double *sT, int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens)
        return -1;
    if (cu_seqlens[0] != 0)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -1;

    int failed = 0;
    const int64_t pairs = N * H;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *S = (double *)malloc((size_t)(dk * dv) * sizeof(double));
        double *vhat = (double *)malloc((size_t)dv * sizeof(double));
        if (!S || !vhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t p = 0; p < pairs; ++p) {
                const int64_t n = p / H, h = p % H;
                const int64_t t0 = cu_seqlens[n];
                const int64_t T = (int64_t)cu_seqlens[n + 1] - t0;
                const double *s0p = s0 ? s0 + p * dk * dv : NULL;
                double *sTp = sT ? sT + p * dk * dv : NULL;
                kda_oracle_head(q, k, v, alpha, beta, s0p, o, sTp, t0, T, H,
                                h, dk, dv, S, vhat);
            }
        }
        free(S);
        free(vhat);
    }
    (void)nthreads;
    return failed ? -2 : 0;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int kda_oracle_max_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}
