/*
 * Float64 CPU oracle for the channel-gated delta rules: Kimi Delta Attention
 * (KDA) and Gated DeltaNet-2 (GDN2).
 *
 * TEST INFRASTRUCTURE ONLY, like gdn_oracle.c: only the test suite may load
 * it; it shares no code, header or constant with the CUDA sources.
 *
 * "Linear Attention Architectures" reading notes, Sec. 2.5 (Eqs. 18-20) and
 * Sec. 2.6 (Eqs. 21-24).  The equations themselves are lost in the page's
 * extraction; the text fixes them:
 *  - KDA replaces the scalar decay by a per-key-channel decay D_alpha =
 *    diag(alpha_t), alpha_t in R^K, multiplied on the RIGHT of the state (it
 *    acts on the key-feature dimension, not the value dimension); alpha_t =
 *    a 1 gives Gated DeltaNet back.  Erase and write share the scalar beta_t.
 *  - GDN2 splits that control: a key-side vector b_t picks the direction the
 *    erase reads out along, e = b_t (.) k_t, and a value-side vector w_t
 *    scales the new content, z = w_t (.) v_t; the outer products keep the
 *    original key on their right (not e).  Written out, with the decayed
 *    state S~ = S D_alpha:  S_t = S~ (I - e k^T) + z k^T.  b = w = beta 1
 *    gives KDA back.
 *
 * Token by token, per (batch, head) sequence, S in R^{V x K}:
 *
 *   S[:, c] <- alpha_t[c] * S[:, c]        forget, per key channel
 *   e <- b_t (.) k_t     (KDA: beta_t k_t)
 *   z <- w_t (.) v_t     (KDA: beta_t v_t)
 *   u <- z - S e                           what the erase leaves to write
 *   S <- S + u k_t^T
 *   o_t <- S q_t
 *
 * Layouts (dense, row-major, float64):
 *   q, k, alpha, b  [B, T, H, K]     v, w, o  [B, T, H, V]
 *   beta [B, T, H] (KDA only)        S0, ST   [B, H, V, K] (S0 may be NULL)
 * gate 1 = KDA (b, w unused), 2 = GDN2 (beta unused).
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define GATED_KDA 1
#define GATED_GDN2 2

typedef struct {
    const double *q, *k, *v, *alpha, *beta, *bg, *wg, *S0;
    double *o, *ST;
    int B, T, H, K, V, gate;
    int first, stride;
} gjob_t;

static void gated_sequence(const gjob_t *J, int seq, double *S, double *e, double *z) {
    const int b = seq / J->H, h = seq % J->H;
    const int H = J->H, K = J->K, V = J->V;
    const size_t state_off = (size_t)seq * V * K;
    if (J->S0)
        memcpy(S, J->S0 + state_off, sizeof(double) * V * K);
    else
        memset(S, 0, sizeof(double) * V * K);
    for (int t = 0; t < J->T; ++t) {
        const size_t th = ((size_t)b * J->T + t) * H + h;
        const double *kt = J->k + th * K;
        const double *qt = J->q ? J->q + th * K : NULL;
        const double *vt = J->v + th * V;
        const double *at = J->alpha + th * K;
        /* forget: column c of S is key channel c */
        for (int i = 0; i < V; ++i)
            for (int c = 0; c < K; ++c) S[(size_t)i * K + c] *= at[c];
        /* erase direction and write content */
        if (J->gate == GATED_KDA) {
            const double be = J->beta[th];
            for (int c = 0; c < K; ++c) e[c] = be * kt[c];
            for (int i = 0; i < V; ++i) z[i] = be * vt[i];
        } else {
            const double *bt = J->bg + th * K;
            const double *wt = J->wg + th * V;
            for (int c = 0; c < K; ++c) e[c] = bt[c] * kt[c];
            for (int i = 0; i < V; ++i) z[i] = wt[i] * vt[i];
        }
        /* u = z - S e, then the write along the original key */
        for (int i = 0; i < V; ++i) {
            double read = 0.0;
            for (int c = 0; c < K; ++c) read += S[(size_t)i * K + c] * e[c];
            const double u = z[i] - read;
            for (int c = 0; c < K; ++c) S[(size_t)i * K + c] += u * kt[c];
        }
        if (J->o && qt) {
            double *ot = J->o + th * V;
            for (int i = 0; i < V; ++i) {
                double r = 0.0;
                for (int c = 0; c < K; ++c) r += S[(size_t)i * K + c] * qt[c];
                ot[i] = r;
            }
        }
    }
    if (J->ST) memcpy(J->ST + state_off, S, sizeof(double) * V * K);
}

static void *gated_worker(void *arg) {
    const gjob_t *J = (const gjob_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->V * J->K);
    double *e = (double *)malloc(sizeof(double) * (size_t)J->K);
    double *z = (double *)malloc(sizeof(double) * (size_t)J->V);
    if (S && e && z)
        for (int s = J->first; s < J->B * J->H; s += J->stride) gated_sequence(J, s, S, e, z);
    free(S);
    free(e);
    free(z);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure. */
int gdn_oracle_gated(const double *q, const double *k, const double *v, const double *alpha,
                     const double *beta, const double *bg, const double *wg, const double *S0,
                     double *o, double *ST, int B, int T, int H, int K, int V, int gate,
                     int nthreads) {
    if (!k || !v || !alpha || B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return -1;
    if (gate == GATED_KDA && !beta) return -1;
    if (gate == GATED_GDN2 && (!bg || !wg)) return -1;
    if (gate != GATED_KDA && gate != GATED_GDN2) return -1;
    if (o && !q) return -1;
    const int nseq = B * H;
    if (nseq == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nseq) nthreads = nseq;
    gjob_t *jobs = (gjob_t *)calloc((size_t)nthreads, sizeof(gjob_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return -2;
    }
    int rc = 0, started = 0;
    for (int i = 0; i < nthreads; ++i) {
        gjob_t J = {q, k, v, alpha, beta, bg, wg, S0, o, ST, B, T, H, K, V, gate, i, nthreads};
        jobs[i] = J;
    }
    if (nthreads == 1) {
        gated_worker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tid[i], NULL, gated_worker, &jobs[i]) != 0) {
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
