/*
 * Float64 token-by-token recurrence for the gated delta-rule family of
 * linear attention, in plain C with one POSIX thread per group of heads.
 *
 * TEST INFRASTRUCTURE ONLY: built next to the CUDA library but linked by
 * nothing in it. Only the tests, the smoke check and the benchmark's CPU
 * baseline load it (through oracle/__init__.py).
 *
 * It computes exactly what oracle/recurrence.py computes (same definition,
 * same orientation: key-major S[dk][dv], o_t = S_t^T q_t) and is pinned to it
 * by the tests; it exists because the Python loop is too slow for full-length
 * sequences and for timing the CPU baseline.
 *
 *   mode 0 linear : S += k v^T                           ("Talk Linear Attention" 2.1)
 *   mode 1 elu1   : S += phi(k) v^T, z += phi(k), o = S^T phi(q) / z.phi(q)
 *                                                        (kernel-attention notes 13-14)
 *   mode 2 retnet : S = gamma_h S + k v^T, g[h] = log gamma_h
 *   mode 3 gla    : S = Diag(alpha_t) S + k v^T, g[b,h,t,c] ("Talk Linear Attention" 5.1)
 *   mode 4 scalar : S = alpha_t S + k v^T, g[b,h,t]
 *   mode 5 gdn    : S = alpha_t S; u = beta_t (v - S^T k); S += k u^T
 *                   (Gated DeltaNet: decay, then the delta rule)
 *   mode 6 kda    : S = Diag(alpha_t) S; u = beta_t (v - S^T k); S += k u^T
 *                   (Kimi Delta Attention: per-key-channel gate g[b,h,t,c])
 *   mode 7 outer  : S = (alpha_t beta_t^T) ⊙ S + k v^T, g[b,h,t,c] = log alpha,
 *                   beta[b,h,t,j] = log beta (outer-product gate,
 *                   "Talk Linear Attention" 5.4)
 *
 * Layouts: q,k [B,H,T,dk], v,o [B,H,T,dv], S0/S [B,H,dk,W] with W = dv+1 for
 * elu1 (z in column dv) and W = dv otherwise. g/beta/S0 may be NULL where the
 * mode allows it (NULL g in gdn means alpha = 1, NULL beta means beta = 1,
 * NULL S0 means a zero initial state).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *S0;
    double *o, *S;
    int B, H, T, dk, dv, mode;
    int head_begin, head_end;
} job_t;

static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

static void run_head(const job_t *J, int bh) {
    const int H = J->H, T = J->T, dk = J->dk, dv = J->dv, mode = J->mode;
    const int W = (mode == 1) ? dv + 1 : dv;
    const int h = bh % H;
    const double *q = J->q + (size_t)bh * T * dk;
    const double *k = J->k + (size_t)bh * T * dk;
    const double *v = J->v + (size_t)bh * T * dv;
    double *o = J->o + (size_t)bh * T * dv;
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *z = (double *)calloc((size_t)dk, sizeof(double));
    double *qh = (double *)malloc(sizeof(double) * dk);
    double *kh = (double *)malloc(sizeof(double) * dk);
    double *u = (double *)malloc(sizeof(double) * dv);

    if (J->S0) {
        const double *s0 = J->S0 + (size_t)bh * dk * W;
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] = s0[(size_t)c * W + j];
            if (mode == 1) z[c] = s0[(size_t)c * W + dv];
        }
    }

    for (int t = 0; t < T; ++t) {
        const double *qt = q + (size_t)t * dk, *kt = k + (size_t)t * dk, *vt = v + (size_t)t * dv;
        double *ot = o + (size_t)t * dv;
        if (mode == 1) {
            for (int c = 0; c < dk; ++c) { qh[c] = phi(qt[c]); kh[c] = phi(kt[c]); }
            qt = qh; kt = kh;
        }
        /* decay */
        if (mode == 2 || mode == 4 || (mode == 5 && J->g)) {
            double a;
            if (mode == 2) a = exp(J->g[h]);
            else a = exp(J->g[(size_t)bh * T + t]);
            for (size_t i = 0; i < (size_t)dk * dv; ++i) S[i] *= a;
        } else if (mode == 3 || mode == 6) {
            const double *gt = J->g + ((size_t)bh * T + t) * dk;
            for (int c = 0; c < dk; ++c) {
                double a = exp(gt[c]);
                for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
            }
        } else if (mode == 7) {
            const double *gt = J->g + ((size_t)bh * T + t) * dk;
            const double *bt = J->beta + ((size_t)bh * T + t) * dv;
            for (int c = 0; c < dk; ++c) {
                double a = exp(gt[c]);
                for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a * exp(bt[j]);
            }
        }
        /* write */
        if (mode == 5 || mode == 6) {
            double b = J->beta ? J->beta[(size_t)bh * T + t] : 1.0;
            for (int j = 0; j < dv; ++j) u[j] = 0.0;
            for (int c = 0; c < dk; ++c)
                for (int j = 0; j < dv; ++j) u[j] += S[(size_t)c * dv + j] * kt[c];
            for (int j = 0; j < dv; ++j) u[j] = b * (vt[j] - u[j]);
            for (int c = 0; c < dk; ++c)
                for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += kt[c] * u[j];
        } else {
            for (int c = 0; c < dk; ++c)
                for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += kt[c] * vt[j];
            if (mode == 1)
                for (int c = 0; c < dk; ++c) z[c] += kt[c];
        }
        /* read */
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j) ot[j] += S[(size_t)c * dv + j] * qt[c];
        if (mode == 1) {
            double den = 0.0;
            for (int c = 0; c < dk; ++c) den += z[c] * qt[c];
            for (int j = 0; j < dv; ++j) ot[j] /= den;
        }
    }

    if (J->S) {
        double *s = J->S + (size_t)bh * dk * W;
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) s[(size_t)c * W + j] = S[(size_t)c * dv + j];
            if (mode == 1) s[(size_t)c * W + dv] = z[c];
        }
    }
    free(S); free(z); free(qh); free(kh); free(u);
}

static void *worker(void *arg) {
    const job_t *J = (const job_t *)arg;
    for (int bh = J->head_begin; bh < J->head_end; ++bh) run_head(J, bh);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 if threads could not start. */
int la_oracle_fwd(const double *q, const double *k, const double *v, const double *g,
                  const double *beta, const double *S0, double *o, double *S,
                  int B, int H, int T, int dk, int dv, int mode, int nthreads) {
    if (!q || !k || !v || !o || B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || mode < 0 || mode > 7)
        return -1;
    if ((mode == 2 || mode == 3 || mode == 4 || mode == 6 || mode == 7) && !g) return -1;
    if (mode == 7 && !beta) return -1;
    const int BH = B * H;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = BH;
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int rc = 0, started = 0;
    for (int i = 0; i < nthreads; ++i) {
        job_t J = {q, k, v, g, beta, S0, o, S, B, H, T, dk, dv, mode,
                   (int)((long)BH * i / nthreads), (int)((long)BH * (i + 1) / nthreads)};
        jobs[i] = J;
    }
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &jobs[i]) != 0) { rc = -2; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(jobs); free(tid);
    return rc;
}

int la_oracle_threads_default(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
