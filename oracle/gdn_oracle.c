/*
 * fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The CUDA operator never links or calls it, and
 * the two share no code.
 *
 * Every routine works on ONE (sequence, head): contiguous row-major arrays
 *   q, k : [T][K]     v, o : [T][V]     g, beta : [T]
 * and a recurrent state.  All arithmetic is plain fp64 in the order the
 * method is written, with no blocking, fusion or reordering.
 *
 * Sources (web pages on the subject):
 *  - "Research Sprint Day 1 - Verifying the flash-linear-attention Gated
 *    DeltaNet kernel on GB10", section "The GDN update": per token
 *        S <- alpha S;  v_old = S^T k;  S <- S + beta k (v - v_old)^T;
 *        o = S^T q
 *    with S of shape K x V.  gdn_oracle_fwd follows it, with the readout
 *    multiplied by `scale` (the cuLA issue #126 reproduction passes
 *    SCALE = D^-0.5 to the kernel; scale = 1 is the plain page-1 form).
 *  - "Research Sprint Day 2 - Rooflines", section "Building some intuition
 *    between attention and GDN", GDN update equation:
 *        S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T
 *    with S of shape V x K.  gdn_oracle_fwd_matrix_form evaluates it
 *    literally (a K x K transition matrix per token) as a cross-check.
 *  - alpha_t = exp(g_t) with g given in log space ("Research Sprint Day 2",
 *    GDN layer pseudocode, step 5).
 *
 * gdn_oracle_bwd is the reverse mode of the page-1 loop, derived by hand
 * (the pages list only which gradients exist: dq, dk, dv, dg, dbeta).  For
 * each token, with S' = alpha S_{t-1}, e = v - S'^T k, S_t = S' + beta k e^T,
 * o = scale S_t^T q, walking t = T..1 with dS = dL/dS_t:
 *     dS  += scale q dO^T
 *     dq   = scale S_t dO
 *     de   = beta dS^T k
 *     dbeta= k^T dS e
 *     dk   = beta dS e - S' de
 *     dv   = de
 *     dS'  = dS - k de^T
 *     dg   = <dS', S'>
 *     dS   = alpha dS'
 * The states S_{t-1} are recomputed from checkpoints taken every 64 tokens.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_CKPT 64

/* Returns 0 on success, -1 on allocation failure. */
int gdn_oracle_fwd(int T, int K, int V, double scale,
                   const double* q, const double* k, const double* v,
                   const double* g, const double* beta,
                   const double* S0, double* o, double* S) {
    double* v_old = (double*)malloc(sizeof(double) * (size_t)V);
    if (!v_old) return -1;
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)K * V);
    else memset(S, 0, sizeof(double) * (size_t)K * V);
    for (int t = 0; t < T; ++t) {
        const double* kt = k + (size_t)t * K;
        const double* qt = q + (size_t)t * K;
        const double* vt = v + (size_t)t * V;
        const double alpha = exp(g[t]);
        const double b = beta[t];
        /* forget */
        for (int i = 0; i < K * V; ++i) S[i] *= alpha;
        /* read what is stored for this key */
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * kt[i];
            v_old[j] = acc;
        }
        /* write the error */
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j)
                S[(size_t)i * V + j] += b * kt[i] * (vt[j] - v_old[j]);
        /* look up with the query */
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * qt[i];
            o[(size_t)t * V + j] = scale * acc;
        }
    }
    free(v_old);
    return 0;
}

/* Page-4 matrix form.  R is the V x K state (R = S^T of the page-1 form).
 * R0 may be NULL (zeros).  o_t = scale R_t q_t. */
int gdn_oracle_fwd_matrix_form(int T, int K, int V, double scale,
                               const double* q, const double* k, const double* v,
                               const double* g, const double* beta,
                               const double* R0, double* o, double* R) {
    double* M = (double*)malloc(sizeof(double) * (size_t)K * K);
    double* Rn = (double*)malloc(sizeof(double) * (size_t)V * K);
    if (!M || !Rn) { free(M); free(Rn); return -1; }
    if (R0) memcpy(R, R0, sizeof(double) * (size_t)V * K);
    else memset(R, 0, sizeof(double) * (size_t)V * K);
    for (int t = 0; t < T; ++t) {
        const double* kt = k + (size_t)t * K;
        const double* qt = q + (size_t)t * K;
        const double* vt = v + (size_t)t * V;
        const double alpha = exp(g[t]);
        const double b = beta[t];
        /* M = alpha (I - beta k k^T) */
        for (int a = 0; a < K; ++a)
            for (int c = 0; c < K; ++c)
                M[(size_t)a * K + c] = alpha * ((a == c ? 1.0 : 0.0) - b * kt[a] * kt[c]);
        /* Rn = R M + beta v k^T */
        for (int r = 0; r < V; ++r)
            for (int c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int a = 0; a < K; ++a) acc += R[(size_t)r * K + a] * M[(size_t)a * K + c];
                Rn[(size_t)r * K + c] = acc + b * vt[r] * kt[c];
            }
        memcpy(R, Rn, sizeof(double) * (size_t)V * K);
        for (int r = 0; r < V; ++r) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += R[(size_t)r * K + c] * qt[c];
            o[(size_t)t * V + r] = scale * acc;
        }
    }
    free(M);
    free(Rn);
    return 0;
}

/* One page-1 step applied to S in place (used by the backward's recompute). */
static void step_fwd(int K, int V, const double* kt, const double* vt, double alpha,
                     double b, double* S, double* v_old) {
    for (int i = 0; i < K * V; ++i) S[i] *= alpha;
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * kt[i];
        v_old[j] = acc;
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(size_t)i * V + j] += b * kt[i] * (vt[j] - v_old[j]);
}

/* Reverse mode of gdn_oracle_fwd.
 * dO: [T][V]; dS_final: K x V or NULL (zeros).
 * Outputs dq, dk [T][K]; dv [T][V]; dg, dbeta [T]; dS0 (K x V, may be NULL).
 * Returns 0 on success, -1 on allocation failure. */
int gdn_oracle_bwd(int T, int K, int V, double scale,
                   const double* q, const double* k, const double* v,
                   const double* g, const double* beta, const double* S0,
                   const double* dO, const double* dS_final,
                   double* dq, double* dk, double* dv, double* dg, double* dbeta,
                   double* dS0) {
    const size_t KV = (size_t)K * V;
    const int n_ckpt = (T + ORACLE_CKPT - 1) / ORACLE_CKPT + 1;
    double* ckpt = (double*)malloc(sizeof(double) * KV * (size_t)n_ckpt);
    double* hist = (double*)malloc(sizeof(double) * KV * ORACLE_CKPT); /* S_{t-1} */
    double* dS = (double*)malloc(sizeof(double) * KV);
    double* Sp = (double*)malloc(sizeof(double) * KV);   /* S' */
    double* St = (double*)malloc(sizeof(double) * KV);   /* S_t */
    double* e = (double*)malloc(sizeof(double) * (size_t)V);
    double* de = (double*)malloc(sizeof(double) * (size_t)V);
    double* tmp = (double*)malloc(sizeof(double) * (size_t)V);
    if (!ckpt || !hist || !dS || !Sp || !St || !e || !de || !tmp) {
        free(ckpt); free(hist); free(dS); free(Sp); free(St); free(e); free(de); free(tmp);
        return -1;
    }
    /* forward sweep, checkpoint S before every 64-token segment */
    double* S = St;
    if (S0) memcpy(S, S0, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);
    for (int t = 0; t < T; ++t) {
        if (t % ORACLE_CKPT == 0) memcpy(ckpt + (size_t)(t / ORACLE_CKPT) * KV, S, sizeof(double) * KV);
        step_fwd(K, V, k + (size_t)t * K, v + (size_t)t * V, exp(g[t]), beta[t], S, tmp);
    }
    if (dS_final) memcpy(dS, dS_final, sizeof(double) * KV);
    else memset(dS, 0, sizeof(double) * KV);

    const int n_seg = (T + ORACLE_CKPT - 1) / ORACLE_CKPT;
    for (int s = n_seg - 1; s >= 0; --s) {
        const int t0 = s * ORACLE_CKPT;
        const int t1 = (t0 + ORACLE_CKPT < T) ? t0 + ORACLE_CKPT : T;
        /* recompute S_{t-1} for t in [t0, t1) */
        memcpy(Sp, ckpt + (size_t)s * KV, sizeof(double) * KV);
        for (int t = t0; t < t1; ++t) {
            memcpy(hist + (size_t)(t - t0) * KV, Sp, sizeof(double) * KV);
            step_fwd(K, V, k + (size_t)t * K, v + (size_t)t * V, exp(g[t]), beta[t], Sp, tmp);
        }
        for (int t = t1 - 1; t >= t0; --t) {
            const double* kt = k + (size_t)t * K;
            const double* qt = q + (size_t)t * K;
            const double* vt = v + (size_t)t * V;
            const double* dot = dO + (size_t)t * V;
            const double alpha = exp(g[t]);
            const double b = beta[t];
            const double* Sprev = hist + (size_t)(t - t0) * KV;
            /* S' = alpha S_{t-1}; e = v - S'^T k; S_t = S' + beta k e^T */
            for (size_t i = 0; i < KV; ++i) Sp[i] = alpha * Sprev[i];
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) acc += Sp[(size_t)i * V + j] * kt[i];
                e[j] = vt[j] - acc;
            }
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j)
                    St[(size_t)i * V + j] = Sp[(size_t)i * V + j] + b * kt[i] * e[j];
            /* dS += scale q dO^T */
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j)
                    dS[(size_t)i * V + j] += scale * qt[i] * dot[j];
            /* dq = scale S_t dO */
            for (int i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) acc += St[(size_t)i * V + j] * dot[j];
                dq[(size_t)t * K + i] = scale * acc;
            }
            /* de = beta dS^T k */
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) acc += dS[(size_t)i * V + j] * kt[i];
                de[j] = b * acc;
            }
            /* dbeta = k^T dS e */
            {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) {
                    double r = 0.0;
                    for (int j = 0; j < V; ++j) r += dS[(size_t)i * V + j] * e[j];
                    acc += kt[i] * r;
                }
                dbeta[t] = acc;
            }
            /* dk = beta dS e - S' de */
            for (int i = 0; i < K; ++i) {
                double a1 = 0.0, a2 = 0.0;
                for (int j = 0; j < V; ++j) {
                    a1 += dS[(size_t)i * V + j] * e[j];
                    a2 += Sp[(size_t)i * V + j] * de[j];
                }
                dk[(size_t)t * K + i] = b * a1 - a2;
            }
            /* dv = de */
            for (int j = 0; j < V; ++j) dv[(size_t)t * V + j] = de[j];
            /* dS' = dS - k de^T ; dg = <dS', S'> ; dS = alpha dS' */
            {
                double acc = 0.0;
                for (int i = 0; i < K; ++i)
                    for (int j = 0; j < V; ++j) {
                        const double d = dS[(size_t)i * V + j] - kt[i] * de[j];
                        acc += d * Sp[(size_t)i * V + j];
                        dS[(size_t)i * V + j] = alpha * d;
                    }
                dg[t] = acc;
            }
        }
    }
    if (dS0) memcpy(dS0, dS, sizeof(double) * KV);
    free(ckpt); free(hist); free(dS); free(Sp); free(St); free(e); free(de); free(tmp);
    return 0;
}
