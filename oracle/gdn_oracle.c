/*
 * Float64 CPU oracle for the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the package
 * smoke check and the CPU-baseline leg of the benchmark may load it; the
 * product library never links or calls it, and it shares no code, header or
 * constant with the CUDA sources.
 *
 * What it computes (token by token, per (batch, head) sequence):
 *
 *   S <- alpha_t * S                       forget first
 *   u <- beta_t * (v_t - S k_t)            error of the decayed state's prediction
 *   S <- S + u k_t^T                       rank-one write
 *   o_t <- S q_t                           read with the query after the write
 *
 * which is S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 * o_t = S_t q_t, with S in R^{V x K}.
 *
 * Sources:
 *  - "On State Reduction in Linear Attention" reading notes, Sec. 2.1,
 *    Eqs. (1)-(2): the DeltaNet update in its error-correction form and the
 *    read o_t = S_t q_t; Gated DeltaNet adds an input-dependent scalar decay.
 *  - "Linear Attention Architectures" reading notes, Sec. 2.1 (Eq. 8, the
 *    shared forget / predict / error / write / read skeleton) and Sec. 2.4
 *    (Eqs. 15-17): the decay is applied to the old state before the error is
 *    formed; an error against the undecayed state is not the GDN update.
 *
 * mode GDN_ORACLE_LINEAR replaces the error by the value itself (u = v),
 * which with alpha = 1 is the unnormalised linear attention of Sec. 2.1
 * (S_t = S_{t-1} + v_t k_t^T) of the state-reduction notes.  It exists only
 * so that a test can compare the two modes.
 *
 * Layouts (all dense, row-major, float64):
 *   q, k   [B, T, H, K]      v, o   [B, T, H, V]
 *   alpha, beta [B, T, H]    S0, ST [B, H, V, K]  (S0 may be NULL: zero state)
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define GDN_ORACLE_DELTA 0
#define GDN_ORACLE_LINEAR 1

typedef struct {
    const double *q, *k, *v, *alpha, *beta, *S0;
    double *o, *ST;
    int B, T, H, K, V, mode;
    int first, stride; /* sequences first, first+stride, ... */
} job_t;

static void run_sequence(const job_t *J, int seq, double *S, double *u) {
    const int b = seq / J->H, h = seq % J->H;
    const int H = J->H, K = J->K, V = J->V;
    const size_t state_off = (size_t)seq * V * K;
    if (J->S0)
        memcpy(S, J->S0 + state_off, sizeof(double) * V * K);
    else
        memset(S, 0, sizeof(double) * V * K);
    for (int t = 0; t < J->T; ++t) {
        const size_t th = ((size_t)b * J->T + t) * H + h; /* token-head index */
        const double a = J->alpha[th];
        const double be = J->beta[th];
        const double *kt = J->k + th * K;
        const double *qt = J->q + th * K;
        const double *vt = J->v + th * V;
        double *ot = J->o ? J->o + th * V : NULL;
        /* forget */
        for (int i = 0; i < V * K; ++i) S[i] *= a;
        /* error against the decayed state, one value channel (row) at a time */
        for (int i = 0; i < V; ++i) {
            if (J->mode == GDN_ORACLE_LINEAR) {
                u[i] = vt[i];
            } else {
                double pred = 0.0;
                for (int j = 0; j < K; ++j) pred += S[(size_t)i * K + j] * kt[j];
                u[i] = be * (vt[i] - pred);
            }
        }
        /* write */
        for (int i = 0; i < V; ++i)
            for (int j = 0; j < K; ++j) S[(size_t)i * K + j] += u[i] * kt[j];
        /* read with the query */
        if (ot) {
            for (int i = 0; i < V; ++i) {
                double r = 0.0;
                for (int j = 0; j < K; ++j) r += S[(size_t)i * K + j] * qt[j];
                ot[i] = r;
            }
        }
    }
    if (J->ST) memcpy(J->ST + state_off, S, sizeof(double) * V * K);
}

static void *worker(void *arg) {
    const job_t *J = (const job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->V * J->K);
    double *u = (double *)malloc(sizeof(double) * (size_t)J->V);
    if (S && u)
        for (int s = J->first; s < J->B * J->H; s += J->stride) run_sequence(J, s, S, u);
    free(S);
    free(u);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure. */
int gdn_oracle_recurrence(const double *q, const double *k, const double *v,
                          const double *alpha, const double *beta, const double *S0,
                          double *o, double *ST, int B, int T, int H, int K, int V,
                          int mode, int nthreads) {
    if (!k || !v || !alpha || !beta || B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0)
        return -1;
    if (o && !q) return -1;
    if (mode != GDN_ORACLE_DELTA && mode != GDN_ORACLE_LINEAR) return -1;
    const int nseq = B * H;
    if (nseq == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nseq) nthreads = nseq;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return -2;
    }
    int rc = 0, started = 0;
    for (int i = 0; i < nthreads; ++i) {
        job_t J = {q, k, v, alpha, beta, S0, o, ST, B, T, H, K, V, mode, i, nthreads};
        jobs[i] = J;
    }
    if (nthreads == 1) {
        worker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tid[i], NULL, worker, &jobs[i]) != 0) {
                rc = -2;
                break;
            }
            ++started;
        }
        for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    }
    free(jobs);
    free(tid);
    return rc;
}
