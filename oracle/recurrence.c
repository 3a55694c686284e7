/*
 * DeltaProduct forward recurrence: plain sequential fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it. It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (DeltaProduct: Improving State-Tracking in Linear RNNs via
 * Householder Products, Sec.4 Eq.(2)-(3) and the gated variant in Sec.4 with
 * its per-token pseudocode, Appendix B.1):
 *
 *   H = H0                      (zeros when no initial state is given)
 *   for every token t:
 *       H = g_t * H             (gated variant only; once per token, before
 *                                the n_h sub-steps)
 *       for j = 0 .. n_h-1:     (ordered generalised-Householder steps)
 *           e = v_{t,j} - H^T k_{t,j}          prediction error (Eq.(2))
 *           H = H + beta_{t,j} k_{t,j} e^T     delta write
 *                                             = (I - b k k^T) H + b k v^T (Eq.(3))
 *       o_t = H^T q_t           readout of the post-update state
 *
 * State H is D_k x D_v (rows indexed by the key dimension). Time is strictly
 * sequential; threads only split the independent (batch, head) pairs.
 *
 * Layouts (row-major, contiguous):
 *   q    [B, T, H, Dk]          k    [B, T, H, nh, Dk]
 *   v    [B, T, H, nh, Dv]      beta [B, T, H, nh]
 *   g    [B, T, H]   (may be NULL: ungated)
 *   h0   [B, H, Dk, Dv] (may be NULL: zero initial state)
 *   o    [B, T, H, Dv]          h_final [B, H, Dk, Dv] (may be NULL)
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, T, H, Dk, Dv, nh;
    const double *q, *k, *v, *beta, *g, *h0;
    double *o, *h_final;
    int next;               /* next (b,h) pair to take; guarded by lock */
    int failed;
    pthread_mutex_t lock;
} oracle_job;

static int run_pair(oracle_job *J, int b, int h, double *S, double *e)
{
    const int T = J->T, H = J->H, Dk = J->Dk, Dv = J->Dv, nh = J->nh;
    const size_t state_off = ((size_t)b * H + h) * (size_t)Dk * Dv;

    if (J->h0)
        memcpy(S, J->h0 + state_off, sizeof(double) * (size_t)Dk * Dv);
    else
        memset(S, 0, sizeof(double) * (size_t)Dk * Dv);

    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;   /* (b,t,h) index */
        if (J->g) {
            const double gt = J->g[tok];
            for (size_t x = 0; x < (size_t)Dk * Dv; ++x) S[x] *= gt;
        }
        for (int j = 0; j < nh; ++j) {
            const double *kk = J->k + (tok * nh + j) * (size_t)Dk;
            const double *vv = J->v + (tok * nh + j) * (size_t)Dv;
            const double bt = J->beta[tok * nh + j];
            /* e = v - H^T k  (accumulated row by row of H) */
            for (int c = 0; c < Dv; ++c) e[c] = vv[c];
            for (int r = 0; r < Dk; ++r) {
                const double *row = S + (size_t)r * Dv;
                for (int c = 0; c < Dv; ++c) e[c] -= row[c] * kk[r];
            }
            /* H += beta k e^T */
            for (int r = 0; r < Dk; ++r) {
                const double br = bt * kk[r];
                double *row = S + (size_t)r * Dv;
                for (int c = 0; c < Dv; ++c) row[c] += br * e[c];
            }
        }
        /* o_t = H^T q_t */
        const double *qq = J->q + tok * (size_t)Dk;
        double *oo = J->o + tok * (size_t)Dv;
        for (int c = 0; c < Dv; ++c) oo[c] = 0.0;
        for (int r = 0; r < Dk; ++r) {
            const double *row = S + (size_t)r * Dv;
            for (int c = 0; c < Dv; ++c) oo[c] += row[c] * qq[r];
        }
    }
    if (J->h_final)
        memcpy(J->h_final + state_off, S, sizeof(double) * (size_t)Dk * Dv);
    return 0;
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->Dk * J->Dv);
    double *e = (double *)malloc(sizeof(double) * (size_t)J->Dv);
    if (!S || !e) {
        pthread_mutex_lock(&J->lock);
        J->failed = 1;
        pthread_mutex_unlock(&J->lock);
        free(S);
        free(e);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int pair = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (pair >= J->B * J->H) break;
        run_pair(J, pair / J->H, pair % J->H, S, e);
    }
    free(S);
    free(e);
    return NULL;
}

/* Returns 0 on success, -1 on bad sizes, -2 on allocation/thread failure. */
int oracle_forward(int B, int T, int H, int Dk, int Dv, int nh,
                   const double *q, const double *k, const double *v,
                   const double *beta, const double *g, const double *h0,
                   double *o, double *h_final, int n_threads)
{
    if (B < 0 || T < 0 || H < 0 || Dk <= 0 || Dv <= 0 || nh <= 0) return -1;
    if ((B * H > 0) && (!beta || !o || (T > 0 && (!q || !k || !v)))) return -1;
    oracle_job J;
    J.B = B; J.T = T; J.H = H; J.Dk = Dk; J.Dv = Dv; J.nh = nh;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.o = o; J.h_final = h_final;
    J.next = 0;
    J.failed = 0;
    pthread_mutex_init(&J.lock, NULL);

    int nt = n_threads < 1 ? 1 : n_threads;
    if (nt > B * H) nt = B * H > 0 ? B * H : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return -2;
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? -2 : 0;
}
