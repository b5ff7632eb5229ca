/*
 * KDA reference gradients: float64, token by token, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or
 * calls this file; only the tests and the benchmark's CPU-baseline leg do.
 * It shares no code, header or constant with the CUDA library, and none with
 * the forward oracle kda_oracle.c either (it is compiled on its own).
 *
 * Source of the map being differentiated: the web page
 * "研究KimiK3，我发现大模型正在学会“管理自己的计算”" (pwwt.cn/news/3763336),
 * the K3 essay, §四 (the KDA update) and §二.1 (the read-out). Per sequence
 * and head, for t = 1..T, in the rank-1 form of the §四 update:
 *
 *     S'_t = Diag(alpha_t) S_{t-1}
 *     e_t  = v_t - S'_t^T k_t
 *     S_t  = S'_t + beta_t k_t e_t^T
 *     o_t  = S_t^T q_t
 *
 * The pages give no gradients; the chain rule fixes them. With G the
 * gradient of the loss with respect to S_t (G = dS_T before the last token),
 * the reverse step for token t is
 *
 *     G      += q_t do_t^T                 (o_t = S_t^T q_t)
 *     dq_t    = S_t do_t
 *     w       = G^T k_t                    (d_v)
 *     dv_t    = beta_t w                   (through e_t)
 *     dbeta_t = w . e_t
 *     dk_t    = beta_t (G e_t - S'_t w)    (the write k e^T, and e's S'^T k)
 *     dS'     = G - beta_t k_t w^T
 *     dalpha_t[i] = sum_j dS'[i][j] S_{t-1}[i][j]
 *     G       = Diag(alpha_t) dS'          (now the gradient w.r.t. S_{t-1})
 *
 * and after the first token G is the gradient with respect to S_0.
 *
 * States are needed in reverse order. They are recomputed, never run
 * backwards: the forward pass keeps S at every KCK-th token, and each
 * stretch of KCK tokens is replayed from its checkpoint (the same float64
 * operations in the same order, so the same bits) before its reverse steps.
 *
 * Layouts as in kda_oracle.c (row-major, sequences packed along the tokens):
 *   q, k, alpha, dq, dk, dalpha : [T_total, H, dk]
 *   v, do, dv                   : [T_total, H, dv]
 *   beta, dbeta                 : [T_total, H]
 *   s0, dsT, ds0                : [N, H, dk, dv]       (d_v fastest)
 * s0 == NULL: zero initial state; dsT == NULL: no gradient on the final
 * state; ds0 == NULL: its gradient is not returned.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KCK 64

/* One forward token: S <- S_t from S_{t-1} (in place). */
static void fwd_token(double *S, const double *kt, const double *at, const double *vt, double bt,
                      int64_t dk, int64_t dv, double *tmp)
{
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
            S[i * dv + j] *= at[i];
    for (int64_t j = 0; j < dv; ++j)
        tmp[j] = 0.0;
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
            tmp[j] += S[i * dv + j] * kt[i];
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
            S[i * dv + j] += bt * kt[i] * (vt[j] - tmp[j]);
}

/* One (sequence, head) pair: T tokens from token index t0. */
static int bwd_head(const double *q, const double *k, const double *v, const double *alpha,
                    const double *beta, const double *s0, const double *dout, const double *dsT,
                    double *dq, double *dkk, double *dvv, double *dalpha, double *dbeta, double *ds0,
                    int64_t t0, int64_t T, int64_t H, int64_t h, int64_t dk, int64_t dv)
{
    const size_t SZ = (size_t)(dk * dv);
    const int64_t nck = T / KCK + 1;              /* checkpoints at t = 0, KCK, 2 KCK, ... */
    double *ck = (double *)malloc((size_t)nck * SZ * sizeof(double));
    double *seg = (double *)malloc((size_t)(KCK + 1) * SZ * sizeof(double));
    double *G = (double *)malloc(SZ * sizeof(double));
    double *Sp = (double *)malloc(SZ * sizeof(double));
    double *dSp = (double *)malloc(SZ * sizeof(double));
    double *e = (double *)malloc((size_t)dv * sizeof(double));
    double *w = (double *)malloc((size_t)dv * sizeof(double));
    double *tmp = (double *)malloc((size_t)dv * sizeof(double));
    int rc = 0;
    if (!ck || !seg || !G || !Sp || !dSp || !e || !w || !tmp) {
        rc = -2;
        goto done;
    }

    /* forward pass, keeping S at every KCK-th token */
    {
        double *S = seg;
        if (s0)
            memcpy(S, s0, SZ * sizeof(double));
        else
            memset(S, 0, SZ * sizeof(double));
        for (int64_t t = 0; t < T; ++t) {
            if (t % KCK == 0)
                memcpy(ck + (size_t)(t / KCK) * SZ, S, SZ * sizeof(double));
            const int64_t th = (t0 + t) * H + h;
            fwd_token(S, k + th * dk, alpha + th * dk, v + th * dv, beta[th], dk, dv, tmp);
        }
    }

    if (dsT)
        memcpy(G, dsT, SZ * sizeof(double));
    else
        memset(G, 0, SZ * sizeof(double));

    for (int64_t c = (T - 1) / KCK; T > 0 && c >= 0; --c) {
        const int64_t ta = c * KCK;
        const int64_t tb = ta + KCK < T ? ta + KCK : T;
        /* replay the stretch: seg[m] = S_{ta + m} */
        memcpy(seg, ck + (size_t)c * SZ, SZ * sizeof(double));
        for (int64_t t = ta; t < tb; ++t) {
            const int64_t th = (t0 + t) * H + h;
            double *nx = seg + (size_t)(t - ta + 1) * SZ;
            memcpy(nx, seg + (size_t)(t - ta) * SZ, SZ * sizeof(double));
            fwd_token(nx, k + th * dk, alpha + th * dk, v + th * dv, beta[th], dk, dv, tmp);
        }
        for (int64_t t = tb - 1; t >= ta; --t) {
            const int64_t th = (t0 + t) * H + h;
            const double *qt = q + th * dk, *kt = k + th * dk, *at = alpha + th * dk;
            const double *vt = v + th * dv, *dot = dout + th * dv;
            const double bt = beta[th];
            const double *Sprev = seg + (size_t)(t - ta) * SZ;   /* S_{t-1} */
            const double *Scur = seg + (size_t)(t - ta + 1) * SZ; /* S_t */

            /* G += q_t do_t^T */
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    G[i * dv + j] += qt[i] * dot[j];
            /* dq_t = S_t do_t */
            for (int64_t i = 0; i < dk; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < dv; ++j)
                    s += Scur[i * dv + j] * dot[j];
                dq[th * dk + i] = s;
            }
            /* S' = Diag(alpha_t) S_{t-1};  e = v_t - S'^T k_t */
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    Sp[i * dv + j] = at[i] * Sprev[i * dv + j];
            for (int64_t j = 0; j < dv; ++j)
                tmp[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    tmp[j] += Sp[i * dv + j] * kt[i];
            for (int64_t j = 0; j < dv; ++j)
                e[j] = vt[j] - tmp[j];
            /* w = G^T k_t */
            for (int64_t j = 0; j < dv; ++j)
                w[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    w[j] += G[i * dv + j] * kt[i];
            /* dv_t, dbeta_t */
            double db = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                dvv[th * dv + j] = bt * w[j];
                db += w[j] * e[j];
            }
            dbeta[th] = db;
            /* dk_t = beta_t (G e - S' w) */
            for (int64_t i = 0; i < dk; ++i) {
                double ge = 0.0, sw = 0.0;
                for (int64_t j = 0; j < dv; ++j) {
                    ge += G[i * dv + j] * e[j];
                    sw += Sp[i * dv + j] * w[j];
                }
                dkk[th * dk + i] = bt * (ge - sw);
            }
            /* dS' = G - beta_t k_t w^T; dalpha_t; G = Diag(alpha_t) dS' */
            for (int64_t i = 0; i < dk; ++i) {
                double da = 0.0;
                for (int64_t j = 0; j < dv; ++j) {
                    const double g = G[i * dv + j] - bt * kt[i] * w[j];
                    dSp[i * dv + j] = g;
                    da += g * Sprev[i * dv + j];
                }
                dalpha[th * dk + i] = da;
            }
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    G[i * dv + j] = at[i] * dSp[i * dv + j];
        }
    }
    if (ds0)
        memcpy(ds0, G, SZ * sizeof(double));

done:
    free(ck);
    free(seg);
    free(G);
    free(Sp);
    free(dSp);
    free(e);
    free(w);
    free(tmp);
    return rc;
}

/*
 * Gradients of sum_t <do_t, o_t> + <dsT, S_T> with respect to q, k, v, alpha,
 * beta and s0 for every (sequence, head) pair. Returns 0 on success, -1 on
 * bad arguments, -2 when memory cannot be had. nthreads <= 0 lets OpenMP
 * choose.
 */
int kda_oracle_backward(const double *q, const double *k, const double *v, const double *alpha,
                        const double *beta, const int32_t *cu_seqlens, int64_t N, int64_t H,
                        int64_t dk, int64_t dv, const double *s0, const double *dout,
                        const double *dsT, double *dq, double *dkk, double *dvv, double *dalpha,
                        double *dbeta, double *ds0, int nthreads)
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
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        const int64_t n = p / H, h = p % H;
        const int64_t t0 = cu_seqlens[n];
        const int64_t T = (int64_t)cu_seqlens[n + 1] - t0;
        const int r = bwd_head(q, k, v, alpha, beta, s0 ? s0 + p * dk * dv : NULL, dout,
                               dsT ? dsT + p * dk * dv : NULL, dq, dkk, dvv, dalpha, dbeta,
                               ds0 ? ds0 + p * dk * dv : NULL, t0, T, H, h, dk, dv);
        if (r != 0) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
    }
    (void)nthreads;
    return failed ? -2 : 0;
}
