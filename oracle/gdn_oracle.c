/*
 * Gated DeltaNet forward: CPU oracle in double precision.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the reference that the CUDA path is
 * checked against; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may build or call it. It shares no code with the GPU library.
 *
 * Sources (web pages on Gated DeltaNet):
 *  - "Lab3 GDN Prefill" (hpc101.zjusct.io), section "Linear Attention 与 Gated
 *    DeltaNet": the gated delta rule, S_bar = a_t S_{t-1};
 *    S_t = S_bar + b_t k_t^T (v_t - k_t S_bar); o_t = q_t S_t, with row vectors
 *    q_t, k_t in R^{1 x dk}, v_t in R^{1 x dv} and S in R^{dk x dv}.
 *  - Same page, section "计算过程描述" (computation description): the chunk
 *    form A = (I + StrictLower(B G K K^T G^-1))^-1, U = A B V, W = A B G K,
 *    S_[c+1] = g_l S_[c] + g_l K^T G^-1 (U - W S_[c]),
 *    O_[c] = (1/sqrt dk)[G Q S_[c] + G Lower(Q K^T) G^-1 (U - W S_[c])],
 *    valid length l_c = min(C, L - cC); g_l is the gate of the last valid token.
 *  - Same page, section "输入输出定义" (interface): raw_g = log(alpha), the
 *    gate prefix sum restarts at every chunk, gamma = exp(g_cumsum); GVA head
 *    map h_qk = floor(h_v / G) with G = Hv / Hq; optional initial state.
 *  - "sgl-qwen3-5-moe" (rainlin-net), decode node 7: the same rule applied one
 *    token at a time (decay, predict, correct, read with the updated state).
 *
 * Conventions of this oracle:
 *  - q, k: [T_total, Hq, dk]; v: [T_total, Hv, dv]; g, beta: [T_total, Hv];
 *    state: [N, Hv, dk, dv] row-major; out: [T_total, Hv, dv]. All double.
 *  - cu_seqlens: int64 [N+1] token offsets of N packed sequences; each
 *    sequence starts its own chunk grid (the pages are silent on packing; this
 *    is the plainest reading: a sequence is an independent problem).
 *  - `scale` multiplies every read-out term (the pages' 1/sqrt(dk)).
 *  - S0 == NULL means a zero initial state; final == NULL means not written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n <= 0: leave as is); returns the count
 * now in effect. Timing only: the results do not depend on it, since every
 * (sequence, head) pair is computed by one thread in a fixed order. */
int gdn_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Processors the OpenMP runtime sees on this host. */
int gdn_oracle_num_procs(void) {
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Recurrent form, token by token ("Lab3 GDN Prefill", Gated DeltaNet section).
 * For each token t of a sequence, with alpha_t = exp(g_t):
 *   S_bar = alpha_t S;  p = k_t S_bar;  S = S_bar + beta_t k_t^T (v_t - p);
 *   o_t = scale * q_t S.
 * ------------------------------------------------------------------------- */
void gdn_oracle_recurrent(int64_t N, const int64_t *cu_seqlens, int64_t Hq,
                          int64_t Hv, int64_t dk, int64_t dv, const double *q,
                          const double *k, const double *v, const double *g,
                          const double *beta, double scale, const double *S0,
                          double *out, double *final_state) {
    const int64_t G = Hv / Hq;
    int64_t pair;
#pragma omp parallel for schedule(dynamic, 1)
    for (pair = 0; pair < N * Hv; ++pair) {
        const int64_t n = pair / Hv, h = pair % Hv, hk = h / G;
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        double *p = (double *)malloc((size_t)dv * sizeof(double));
        if (S0) memcpy(S, S0 + (n * Hv + h) * dk * dv, (size_t)(dk * dv) * sizeof(double));
        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const double *kt = k + (t * Hq + hk) * dk;
            const double *qt = q + (t * Hq + hk) * dk;
            const double *vt = v + (t * Hv + h) * dv;
            const double alpha = exp(g[t * Hv + h]);
            const double b = beta[t * Hv + h];
            for (int64_t i = 0; i < dk * dv; ++i) S[i] *= alpha; /* S_bar */
            for (int64_t j = 0; j < dv; ++j) {                   /* p = k S_bar */
                double acc = 0.0;
                for (int64_t i = 0; i < dk; ++i) acc += kt[i] * S[i * dv + j];
                p[j] = acc;
            }
            for (int64_t i = 0; i < dk; ++i)                     /* rank-1 correction */
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += b * kt[i] * (vt[j] - p[j]);
            double *ot = out + (t * Hv + h) * dv;                /* read with updated S */
            for (int64_t j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < dk; ++i) acc += qt[i] * S[i * dv + j];
                ot[j] = scale * acc;
            }
        }
        if (final_state) memcpy(final_state + (n * Hv + h) * dk * dv, S, (size_t)(dk * dv) * sizeof(double));
        free(p);
        free(S);
    }
}

/* ---------------------------------------------------------------------------
 * Chunk form ("Lab3 GDN Prefill", section 计算过程描述), any chunk size C.
 * Per chunk of valid length l (rows/cols >= l never enter a sum):
 *   gc_r  = sum_{j<=r} g_j             (prefix sum restarted at the chunk)
 *   M_ij  = beta_i exp(gc_i - gc_j) (k_i . k_j)   for j < i   (StrictLower of
 *           B Gamma K K^T Gamma^-1; Gamma^-1 only ever enters as a masked
 *           exp of a difference, never on its own)
 *   A     = (I + M)^-1                 (unit lower triangular: forward
 *                                       substitution, column by column)
 *   U     = A diag(beta) V,  W = A diag(beta * gamma) K
 *   R     = U - W S
 *   O_r   = scale [ gamma_r q_r S + sum_{i<=r} exp(gc_r - gc_i)(q_r . k_i) R_i ]
 *   S    <- gamma_l S + sum_{i<l} exp(gc_l - gc_i) k_i^T R_i
 * where gamma_l is the gate of the chunk's last valid token.
 * ------------------------------------------------------------------------- */
void gdn_oracle_chunked(int64_t N, const int64_t *cu_seqlens, int64_t Hq,
                        int64_t Hv, int64_t dk, int64_t dv, int64_t C,
                        const double *q, const double *k, const double *v,
                        const double *g, const double *beta, double scale,
                        const double *S0, double *out, double *final_state) {
    const int64_t G = Hv / Hq;
    int64_t pair;
#pragma omp parallel for schedule(dynamic, 1)
    for (pair = 0; pair < N * Hv; ++pair) {
        const int64_t n = pair / Hv, h = pair % Hv, hk = h / G;
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        double *gc = (double *)malloc((size_t)C * sizeof(double));
        double *gam = (double *)malloc((size_t)C * sizeof(double));
        double *M = (double *)calloc((size_t)(C * C), sizeof(double));
        double *A = (double *)calloc((size_t)(C * C), sizeof(double));
        double *P = (double *)calloc((size_t)(C * C), sizeof(double));
        double *U = (double *)malloc((size_t)(C * dv) * sizeof(double));
        double *W = (double *)malloc((size_t)(C * dk) * sizeof(double));
        double *R = (double *)malloc((size_t)(C * dv) * sizeof(double));
        double *Snew = (double *)malloc((size_t)(dk * dv) * sizeof(double));
        if (S0) memcpy(S, S0 + (n * Hv + h) * dk * dv, (size_t)(dk * dv) * sizeof(double));
        const int64_t t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - cu_seqlens[n];
        for (int64_t c = 0; c * C < L; ++c) {
            const int64_t base = t0 + c * C;
            const int64_t l = (L - c * C < C) ? (L - c * C) : C;
#define KROW(i) (k + ((base + (i)) * Hq + hk) * dk)
#define QROW(i) (q + ((base + (i)) * Hq + hk) * dk)
#define VROW(i) (v + ((base + (i)) * Hv + h) * dv)
#define GATE(i) (g[(base + (i)) * Hv + h])
#define BETA(i) (beta[(base + (i)) * Hv + h])
            /* gate prefix sum, restarted at the chunk */
            double run = 0.0;
            for (int64_t r = 0; r < l; ++r) { run += GATE(r); gc[r] = run; }
            /* M = StrictLower(B Gamma K K^T Gamma^-1) on the valid block */
            for (int64_t i = 0; i < l; ++i)
                for (int64_t j = 0; j < l; ++j) {
                    double m = 0.0;
                    if (j < i) {
                        double kk = 0.0;
                        for (int64_t d = 0; d < dk; ++d) kk += KROW(i)[d] * KROW(j)[d];
                        m = BETA(i) * exp(gc[i] - gc[j]) * kk;
                    }
                    M[i * C + j] = m;
                }
            /* A = (I + M)^-1: for each column j solve (I + M) a = e_j */
            for (int64_t j = 0; j < l; ++j)
                for (int64_t i = 0; i < l; ++i) {
                    double a = (i == j) ? 1.0 : 0.0;
                    for (int64_t m = 0; m < i; ++m) a -= M[i * C + m] * A[m * C + j];
                    A[i * C + j] = a;
                }
            /* U = A diag(beta) V ;  W = A diag(beta gamma) K */
            for (int64_t j = 0; j < l; ++j) gam[j] = exp(gc[j]);
            for (int64_t i = 0; i < l; ++i) {
                for (int64_t e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < l; ++j) acc += A[i * C + j] * BETA(j) * VROW(j)[e];
                    U[i * dv + e] = acc;
                }
                for (int64_t d = 0; d < dk; ++d) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < l; ++j) acc += A[i * C + j] * BETA(j) * gam[j] * KROW(j)[d];
                    W[i * dk + d] = acc;
                }
            }
            /* R = U - W S */
            for (int64_t i = 0; i < l; ++i)
                for (int64_t e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int64_t d = 0; d < dk; ++d) acc += W[i * dk + d] * S[d * dv + e];
                    R[i * dv + e] = U[i * dv + e] - acc;
                }
            /* P = Gamma Lower(Q K^T) Gamma^-1 (diagonal included), masked
               before the exponential so that no Gamma^-1 is ever formed */
            for (int64_t r = 0; r < l; ++r)
                for (int64_t i = 0; i < l; ++i) {
                    double pr = 0.0;
                    if (i <= r) {
                        double qk = 0.0;
                        for (int64_t d = 0; d < dk; ++d) qk += QROW(r)[d] * KROW(i)[d];
                        pr = exp(gc[r] - gc[i]) * qk;
                    }
                    P[r * C + i] = pr;
                }
            /* O = scale [Gamma Q S + P R] */
            for (int64_t r = 0; r < l; ++r) {
                double *orow = out + ((base + r) * Hv + h) * dv;
                const double gr = exp(gc[r]);
                for (int64_t e = 0; e < dv; ++e) {
                    double inter = 0.0;
                    for (int64_t d = 0; d < dk; ++d) inter += QROW(r)[d] * S[d * dv + e];
                    double intra = 0.0;
                    for (int64_t i = 0; i <= r; ++i) intra += P[r * C + i] * R[i * dv + e];
                    orow[e] = scale * (gr * inter + intra);
                }
            }
            /* S <- gamma_l S + gamma_l K^T Gamma^-1 R */
            const double gl = gc[l - 1];
            for (int64_t i = 0; i < l; ++i) gam[i] = exp(gl - gc[i]); /* gamma_l / gamma_i */
            for (int64_t d = 0; d < dk; ++d)
                for (int64_t e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < l; ++i) acc += gam[i] * KROW(i)[d] * R[i * dv + e];
                    Snew[d * dv + e] = exp(gl) * S[d * dv + e] + acc;
                }
            memcpy(S, Snew, (size_t)(dk * dv) * sizeof(double));
#undef KROW
#undef QROW
#undef VROW
#undef GATE
#undef BETA
        }
        if (final_state) memcpy(final_state + (n * Hv + h) * dk * dv, S, (size_t)(dk * dv) * sizeof(double));
        free(Snew); free(R); free(W); free(U); free(P); free(A); free(M); free(gam); free(gc); free(S);
    }
}
