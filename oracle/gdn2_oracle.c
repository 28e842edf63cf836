/*
 * gdn2_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet-2 token-mixer core.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm may load or call this code. It shares nothing with the CUDA path and the CUDA path never
 * calls it.
 *
 * What it computes (burn-gdn2 0.1.5 docs, "Architecture", the per-token recurrence on the matrix
 * state S in R^{d_k x d_v}):
 *
 *     S_t = (I - k_t (b_t . k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t . v_t)^T,     o_t = S_t^T q_t
 *
 * with alpha_t = exp(g_t) per key channel, b_t the erase gate on the key axis and w_t the write
 * gate on the value axis ("." is the element-wise product). Readings where the page is silent:
 *   - o_t reads the post-update state S_t (the page prints "o_t = q_t^T S" without a subscript);
 *   - o_t is multiplied by `scale` (1.0 in every workload here);
 *   - q, k belong to key heads; g, b, v, w and the state to value heads; value head h uses key head
 *     h / (H_v / H_k) (contiguous groups);
 *   - an absent initial state means S_0 = 0.
 *
 * Three forms are provided; all take fp32 input arrays holding the exact stored values (bf16 values
 * widen exactly to fp32) and compute in double:
 *   form 0 "recurrent": the recurrence with the matrix product regrouped as a rank-1 update
 *          (S' = diag(alpha) S; r = S'^T (b.k); S = S' + k (w.v - r)^T), O(d_k d_v) per token;
 *   form 1 "literal":   the recurrence exactly as printed, building the d_k x d_k matrix
 *          E = (I - k (b.k)^T) diag(alpha) and computing S = E S + k (w.v)^T, O(d_k^2 d_v) per token;
 *   form 2 "chunked":   the chunked WY/UT form named by the same page ("chunked WY decomposition
 *          (training)"): per chunk of C tokens, cumulative log-decay, the strictly lower erase
 *          interaction matrix, its unit-lower inverse by forward substitution, the W/U factors,
 *          the inter-chunk state update and the intra-chunk causal output. The decay between two
 *          tokens, exp(G_i - G_j), is taken as the exponential of the gates summed over the
 *          tokens in between (no cancellation; exact when a gate is -inf, i.e. alpha = 0).
 *
 * Layouts (all row-major, innermost index last):
 *   q, k [B, T, H_k, d_k]; g, b [B, T, H_v, d_k]; v, w [B, T, H_v, d_v]; o [B, T, H_v, d_v];
 *   states S0 / S_T [B, H_v, d_k, d_v] (double).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float *q, *k, *v, *g, *b, *w;
    const double *s0;
    double *o, *sT;
    int B, T, Hk, Hv, dk, dv, C, form;
    double scale;
    int next;
    int failed;
    pthread_mutex_t mu;
} job_t;

#define QK(j, bi, t, h, i) (((size_t)((bi) * (j)->T + (t)) * (j)->Hk + (h)) * (j)->dk + (i))
#define GB(j, bi, t, h, i) (((size_t)((bi) * (j)->T + (t)) * (j)->Hv + (h)) * (j)->dk + (i))
#define VW(j, bi, t, h, c) (((size_t)((bi) * (j)->T + (t)) * (j)->Hv + (h)) * (j)->dv + (c))
#define ST(j, bi, h) ((size_t)((bi) * (j)->Hv + (h)) * (j)->dk * (j)->dv)

/* ---------------------------------------------------------------------------------------------- */
/* form 0: the recurrence, rank-1 grouping                                                         */

static int unit_recurrent(job_t* j, int bi, int hv, double* S) {
    const int dk = j->dk, dv = j->dv, hk = hv / (j->Hv / j->Hk);
    double* r = (double*)malloc(sizeof(double) * dv);
    double* d = (double*)malloc(sizeof(double) * dv);
    if (!r || !d) { free(r); free(d); return -1; }
    for (int t = 0; t < j->T; ++t) {
        const float* qt = j->q + QK(j, bi, t, hk, 0);
        const float* kt = j->k + QK(j, bi, t, hk, 0);
        const float* gt = j->g + GB(j, bi, t, hv, 0);
        const float* bt = j->b + GB(j, bi, t, hv, 0);
        const float* vt = j->v + VW(j, bi, t, hv, 0);
        const float* wt = j->w + VW(j, bi, t, hv, 0);
        /* S' = diag(alpha_t) S_{t-1} */
        for (int i = 0; i < dk; ++i) {
            const double a = exp((double)gt[i]);
            for (int c = 0; c < dv; ++c) S[(size_t)i * dv + c] *= a;
        }
        /* r = S'^T (b_t . k_t) */
        for (int c = 0; c < dv; ++c) r[c] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double bk = (double)bt[i] * (double)kt[i];
            for (int c = 0; c < dv; ++c) r[c] += S[(size_t)i * dv + c] * bk;
        }
        /* d = w_t . v_t - r ;  S_t = S' + k_t d^T */
        for (int c = 0; c < dv; ++c) d[c] = (double)wt[c] * (double)vt[c] - r[c];
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            for (int c = 0; c < dv; ++c) S[(size_t)i * dv + c] += ki * d[c];
        }
        /* o_t = scale * S_t^T q_t */
        if (j->o) {
            double* ot = j->o + VW(j, bi, t, hv, 0);
            for (int c = 0; c < dv; ++c) ot[c] = 0.0;
            for (int i = 0; i < dk; ++i) {
                const double qi = (double)qt[i];
                for (int c = 0; c < dv; ++c) ot[c] += S[(size_t)i * dv + c] * qi;
            }
            for (int c = 0; c < dv; ++c) ot[c] *= j->scale;
        }
    }
    free(r);
    free(d);
    return 0;
}

/* ---------------------------------------------------------------------------------------------- */
/* form 1: the recurrence as printed, with the explicit d_k x d_k transition                       */

static int unit_literal(job_t* j, int bi, int hv, double* S) {
    const int dk = j->dk, dv = j->dv, hk = hv / (j->Hv / j->Hk);
    double* E = (double*)malloc(sizeof(double) * dk * dk);
    double* N = (double*)malloc(sizeof(double) * dk * dv);
    if (!E || !N) { free(E); free(N); return -1; }
    for (int t = 0; t < j->T; ++t) {
        const float* qt = j->q + QK(j, bi, t, hk, 0);
        const float* kt = j->k + QK(j, bi, t, hk, 0);
        const float* gt = j->g + GB(j, bi, t, hv, 0);
        const float* bt = j->b + GB(j, bi, t, hv, 0);
        const float* vt = j->v + VW(j, bi, t, hv, 0);
        const float* wt = j->w + VW(j, bi, t, hv, 0);
        /* E = (I - k (b.k)^T) diag(alpha):  E[i][l] = (delta_il - k_i b_l k_l) alpha_l */
        for (int i = 0; i < dk; ++i)
            for (int l = 0; l < dk; ++l) {
                const double eye = (i == l) ? 1.0 : 0.0;
                const double outer = (double)kt[i] * ((double)bt[l] * (double)kt[l]);
                E[(size_t)i * dk + l] = (eye - outer) * exp((double)gt[l]);
            }
        /* S_t = E S_{t-1} + k (w.v)^T */
        for (int i = 0; i < dk; ++i)
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int l = 0; l < dk; ++l) acc += E[(size_t)i * dk + l] * S[(size_t)l * dv + c];
                N[(size_t)i * dv + c] = acc + (double)kt[i] * ((double)wt[c] * (double)vt[c]);
            }
        memcpy(S, N, sizeof(double) * dk * dv);
        if (j->o) {
            double* ot = j->o + VW(j, bi, t, hv, 0);
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + c] * (double)qt[i];
                ot[c] = j->scale * acc;
            }
        }
    }
    free(E);
    free(N);
    return 0;
}

/* ---------------------------------------------------------------------------------------------- */
/* form 2: chunked WY / UT form                                                                    */

static int unit_chunked(job_t* j, int bi, int hv, double* S) {
    const int dk = j->dk, dv = j->dv, C = j->C, hk = hv / (j->Hv / j->Hk);
    double* G = (double*)malloc(sizeof(double) * C * dk);      /* cumulative log-decay G_i        */
    double* Gs = (double*)malloc(sizeof(double) * C * dk);     /* decay from after token i to end */
    double* E = (double*)malloc(sizeof(double) * C * C * dk);  /* exp(sum_{j<s<=i} g_s), j <= i   */
    double* A = (double*)malloc(sizeof(double) * C * C);       /* erase interaction               */
    double* M = (double*)malloc(sizeof(double) * C * C);       /* causal q-k                      */
    double* Ti = (double*)malloc(sizeof(double) * C * C);      /* (I + A)^{-1}                    */
    double* W = (double*)malloc(sizeof(double) * C * dk);
    double* U = (double*)malloc(sizeof(double) * C * dv);
    double* O = (double*)malloc(sizeof(double) * C * dv);
    double* X = (double*)malloc(sizeof(double) * C * dk);
    double* Y = (double*)malloc(sizeof(double) * C * dv);
    int rc = 0;
    if (!G || !Gs || !E || !A || !M || !Ti || !W || !U || !O || !X || !Y) { rc = -1; goto done; }

    for (int t0 = 0; t0 < j->T; t0 += C) {
        const int n = (j->T - t0 < C) ? (j->T - t0) : C;
#define q_(i, c) ((double)j->q[QK(j, bi, t0 + (i), hk, c)])
#define k_(i, c) ((double)j->k[QK(j, bi, t0 + (i), hk, c)])
#define g_(i, c) ((double)j->g[GB(j, bi, t0 + (i), hv, c)])
#define b_(i, c) ((double)j->b[GB(j, bi, t0 + (i), hv, c)])
#define v_(i, c) ((double)j->v[VW(j, bi, t0 + (i), hv, c)])
#define w_(i, c) ((double)j->w[VW(j, bi, t0 + (i), hv, c)])
#define E_(i, jj, c) E[((size_t)(i) * C + (jj)) * dk + (c)]
        /* cumulative log-decay within the chunk (inclusive), G_i = sum_{s<=i} g_s, and the decay
           still to come after token i, sum_{i<s<n} g_s.  Decay factors between two tokens are
           taken as the exponential of the sum of the gates strictly after j up to i, which is
           G_i - G_j without the cancellation (and exact when a gate is -inf, alpha = 0).       */
        for (int c = 0; c < dk; ++c) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i) { acc += g_(i, c); G[i * dk + c] = acc; }
            acc = 0.0;
            for (int i = n - 1; i >= 0; --i) { Gs[i * dk + c] = acc; acc += g_(i, c); }
            for (int jj = 0; jj < n; ++jj) {
                double sum = 0.0;
                E_(jj, jj, c) = 1.0;
                for (int i = jj + 1; i < n; ++i) { sum += g_(i, c); E_(i, jj, c) = exp(sum); }
            }
        }
        /* A_ij = sum_c b_i k_i k_j e^{G_i - G_j} for j < i;  M_ij = sum_c q_i k_j e^{G_i - G_j}, j <= i */
        for (int i = 0; i < n; ++i)
            for (int jj = 0; jj < n; ++jj) {
                double a = 0.0, m = 0.0;
                if (jj <= i)
                    for (int c = 0; c < dk; ++c) {
                        const double e = E_(i, jj, c);
                        a += b_(i, c) * k_(i, c) * k_(jj, c) * e;
                        m += q_(i, c) * k_(jj, c) * e;
                    }
                A[i * C + jj] = (jj < i) ? a : 0.0;
                M[i * C + jj] = (jj <= i) ? m : 0.0;
            }
        /* T = (I + A)^{-1}, unit lower triangular, by forward substitution:
           row i:  T_i = e_i - sum_{j<i} A_ij T_j                                              */
        for (int i = 0; i < n; ++i) {
            for (int c = 0; c < n; ++c) Ti[i * C + c] = (c == i) ? 1.0 : 0.0;
            for (int jj = 0; jj < i; ++jj) {
                const double a = A[i * C + jj];
                for (int c = 0; c < n; ++c) Ti[i * C + c] -= a * Ti[jj * C + c];
            }
        }
        /* W = T (b . k . e^{G}),  U~ = T (w . v) */
        for (int i = 0; i < n; ++i) {
            for (int c = 0; c < dk; ++c) X[i * dk + c] = b_(i, c) * k_(i, c) * exp(G[i * dk + c]);
            for (int c = 0; c < dv; ++c) Y[i * dv + c] = w_(i, c) * v_(i, c);
        }
        for (int i = 0; i < n; ++i) {
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int jj = 0; jj <= i; ++jj) acc += Ti[i * C + jj] * X[jj * dk + c];
                W[i * dk + c] = acc;
            }
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int jj = 0; jj <= i; ++jj) acc += Ti[i * C + jj] * Y[jj * dv + c];
                U[i * dv + c] = acc;   /* U~ for now */
            }
        }
        /* U = U~ - W S_n */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int l = 0; l < dk; ++l) acc += W[i * dk + l] * S[(size_t)l * dv + c];
                U[i * dv + c] -= acc;
            }
        /* O = (q . e^{G}) S_n + M U */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int l = 0; l < dk; ++l) acc += q_(i, l) * exp(G[i * dk + l]) * S[(size_t)l * dv + c];
                for (int jj = 0; jj <= i; ++jj) acc += M[i * C + jj] * U[jj * dv + c];
                O[i * dv + c] = acc;
            }
        /* S_{n+1} = diag(e^{G_last}) S_n + (k . e^{G_last - G})^T U */
        for (int l = 0; l < dk; ++l) {
            const double gl = G[(n - 1) * dk + l];
            for (int c = 0; c < dv; ++c) {
                double acc = exp(gl) * S[(size_t)l * dv + c];
                for (int i = 0; i < n; ++i) acc += k_(i, l) * exp(Gs[i * dk + l]) * U[i * dv + c];
                S[(size_t)l * dv + c] = acc;
            }
        }
        if (j->o)
            for (int i = 0; i < n; ++i) {
                double* ot = j->o + VW(j, bi, t0 + i, hv, 0);
                for (int c = 0; c < dv; ++c) ot[c] = j->scale * O[i * dv + c];
            }
#undef q_
#undef k_
#undef g_
#undef b_
#undef v_
#undef w_
#undef E_
    }
done:
    free(G); free(Gs); free(E); free(A); free(M); free(Ti); free(W); free(U); free(O); free(X); free(Y);
    return rc;
}

/* ---------------------------------------------------------------------------------------------- */
/* threading over independent (batch, value head) units                                            */

static void* worker(void* arg) {
    job_t* j = (job_t*)arg;
    const size_t nst = (size_t)j->dk * j->dv;
    double* S = (double*)malloc(sizeof(double) * (nst ? nst : 1));
    if (!S) { pthread_mutex_lock(&j->mu); j->failed = 1; pthread_mutex_unlock(&j->mu); return NULL; }
    for (;;) {
        pthread_mutex_lock(&j->mu);
        const int u = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (u >= j->B * j->Hv) break;
        const int bi = u / j->Hv, hv = u % j->Hv;
        if (j->s0) memcpy(S, j->s0 + ST(j, bi, hv), sizeof(double) * nst);
        else memset(S, 0, sizeof(double) * nst);
        int rc = (j->form == 0) ? unit_recurrent(j, bi, hv, S)
               : (j->form == 1) ? unit_literal(j, bi, hv, S)
                                : unit_chunked(j, bi, hv, S);
        if (rc) { pthread_mutex_lock(&j->mu); j->failed = 1; pthread_mutex_unlock(&j->mu); }
        if (j->sT) memcpy(j->sT + ST(j, bi, hv), S, sizeof(double) * nst);
    }
    free(S);
    return NULL;
}

/*
 * gdn2_oracle_run -- run one form over all (batch, value head) units.
 *   form: 0 recurrent, 1 literal, 2 chunked (chunk length C >= 1).
 *   s0 may be NULL (zeros); o and sT may be NULL (not written).
 *   nthreads <= 0 means 1.
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int gdn2_oracle_run(int form, const float* q, const float* k, const float* v, const float* g,
                    const float* b, const float* w, const double* s0, double* o, double* sT,
                    int B, int T, int Hk, int Hv, int dk, int dv, int C, double scale, int nthreads) {
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk) return -1;
    if (form < 0 || form > 2 || (form == 2 && C < 1)) return -1;
    if (T > 0 && (!q || !k || !v || !g || !b || !w)) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.k = k; j.v = v; j.g = g; j.b = b; j.w = w; j.s0 = s0; j.o = o; j.sT = sT;
    j.B = B; j.T = T; j.Hk = Hk; j.Hv = Hv; j.dk = dk; j.dv = dv; j.C = C; j.form = form;
    j.scale = scale;
    pthread_mutex_init(&j.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B * Hv) nthreads = B * Hv > 0 ? B * Hv : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    int started = 0;
    if (th)
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, worker, &j)) break;
    if (started == 0) worker(&j);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.mu);
    return j.failed ? -1 : 0;
}
