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
    const double *kw;       /* write keys (OSDN variant), or NULL: write with k */
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
            const double *kwr = J->kw ? J->kw + (tok * nh + j) * (size_t)Dk : kk;
            const double *vv = J->v + (tok * nh + j) * (size_t)Dv;
            const double bt = J->beta[tok * nh + j];
            /* e = v - H^T k  (accumulated row by row of H) */
            for (int c = 0; c < Dv; ++c) e[c] = vv[c];
            for (int r = 0; r < Dk; ++r) {
                const double *row = S + (size_t)r * Dv;
                for (int c = 0; c < Dv; ++c) e[c] -= row[c] * kk[r];
            }
            /* H += beta k e^T (OSDN: beta k~ e^T, the write key) */
            for (int r = 0; r < Dk; ++r) {
                const double br = bt * kwr[r];
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

/* Returns 0 on success, -1 on bad sizes, -2 on allocation/thread failure.
 * kw: write keys [B,T,H,nh,Dk] (OSDN, Sec.4.1 / Eq.(5) of the OSDN paper:
 * the state is written along k~ = d (.) k while the residual still reads
 * with k), or NULL for the plain recurrence. */
int oracle_forward_wk(int B, int T, int H, int Dk, int Dv, int nh,
                      const double *q, const double *k, const double *kw, const double *v,
                      const double *beta, const double *g, const double *h0,
                      double *o, double *h_final, int n_threads);

int oracle_forward(int B, int T, int H, int Dk, int Dv, int nh,
                   const double *q, const double *k, const double *v,
                   const double *beta, const double *g, const double *h0,
                   double *o, double *h_final, int n_threads)
{
    return oracle_forward_wk(B, T, H, Dk, Dv, nh, q, k, NULL, v, beta, g, h0, o, h_final, n_threads);
}

int oracle_forward_wk(int B, int T, int H, int Dk, int Dv, int nh,
                      const double *q, const double *k, const double *kw, const double *v,
                      const double *beta, const double *g, const double *h0,
                      double *o, double *h_final, int n_threads)
{
    if (B < 0 || T < 0 || H < 0 || Dk <= 0 || Dv <= 0 || nh <= 0) return -1;
    if ((B * H > 0) && (!beta || !o || (T > 0 && (!q || !k || !v)))) return -1;
    oracle_job J;
    J.B = B; J.T = T; J.H = H; J.Dk = Dk; J.Dv = Dv; J.nh = nh;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.kw = kw;
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

/*
 * Backward pass (reverse-mode gradients) of the same recurrence, fp64.
 *
 * Each sub-step is H' = H + k u^T with u = beta (v - H^T k) (the prediction
 * error scaled by beta, Eq.(2)); the token's gate multiplies H once before
 * its sub-steps and the readout o_t = H^T q_t reads the post-update state.
 * Given dH' (the gradient of the loss with respect to H'):
 *
 *   du     = dH'^T k                       (through k u^T)
 *   dv     = beta du                       (u depends on v linearly)
 *   dbeta  = du . (v - H^T k)
 *   dk     = dH' u - beta H du             (k u^T, and -H^T k inside u)
 *   dH     = dH' - beta k du^T             (= (I - beta k k^T) dH')
 *
 * readout: dq_t = H do_t and dH += q_t do_t^T;
 * gate:    dg_t = <dH_gated, H_before_gate> (Frobenius), dH_before = g_t dH_gated.
 *
 * Plain strategy: the forward stores the state at the start of every token
 * (before its gate); the backward walks the tokens in reverse, recomputes the
 * token's sub-step states from that copy, then applies the rules above in
 * reverse order. Memory: (T + 1) D_k D_v doubles per (batch, head).
 *
 * Extra layouts: do [B,T,H,Dv]; dh_final [B,H,Dk,Dv] or NULL (zero);
 * outputs dq [B,T,H,Dk], dk [B,T,H,nh,Dk], dv [B,T,H,nh,Dv],
 * dbeta [B,T,H,nh], dg [B,T,H] (NULL when ungated), dh0 [B,H,Dk,Dv] or NULL.
 */
typedef struct {
    int B, T, H, Dk, Dv, nh;
    const double *q, *k, *v, *beta, *g, *h0, *d_o, *dh_final;
    double *dq, *dk, *dv, *dbeta, *dg, *dh0;
    int next;
    int failed;
    pthread_mutex_t lock;
} oracle_bwd_job;

static int run_pair_bwd(oracle_bwd_job *J, int b, int h)
{
    const int T = J->T, H = J->H, Dk = J->Dk, Dv = J->Dv, nh = J->nh;
    const size_t SZ = (size_t)Dk * Dv;
    const size_t state_off = ((size_t)b * H + h) * SZ;
    double *Stok = (double *)malloc(sizeof(double) * SZ * (size_t)(T + 1));
    double *Ssub = (double *)malloc(sizeof(double) * SZ * (size_t)(nh + 1));
    double *dS = (double *)malloc(sizeof(double) * SZ);
    double *e = (double *)malloc(sizeof(double) * (size_t)Dv * (nh > 0 ? nh : 1));
    double *du = (double *)malloc(sizeof(double) * (size_t)Dv);
    if (!Stok || !Ssub || !dS || !e || !du) {
        free(Stok); free(Ssub); free(dS); free(e); free(du);
        return -2;
    }

    /* forward: Stok[t] = state at the start of token t (before its gate) */
    if (J->h0)
        memcpy(Stok, J->h0 + state_off, sizeof(double) * SZ);
    else
        memset(Stok, 0, sizeof(double) * SZ);
    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        double *S = Stok + (size_t)(t + 1) * SZ;
        memcpy(S, Stok + (size_t)t * SZ, sizeof(double) * SZ);
        if (J->g)
            for (size_t x = 0; x < SZ; ++x) S[x] *= J->g[tok];
        for (int j = 0; j < nh; ++j) {
            const double *kk = J->k + (tok * nh + j) * (size_t)Dk;
            const double *vv = J->v + (tok * nh + j) * (size_t)Dv;
            const double bt = J->beta[tok * nh + j];
            for (int c = 0; c < Dv; ++c) e[c] = vv[c];
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c) e[c] -= S[(size_t)r * Dv + c] * kk[r];
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c) S[(size_t)r * Dv + c] += bt * kk[r] * e[c];
        }
    }

    /* backward */
    if (J->dh_final)
        memcpy(dS, J->dh_final + state_off, sizeof(double) * SZ);
    else
        memset(dS, 0, sizeof(double) * SZ);
    for (int t = T - 1; t >= 0; --t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const double gt = J->g ? J->g[tok] : 1.0;
        /* the token's sub-step states Ssub[0] (gated) .. Ssub[nh] and errors e_j */
        for (size_t x = 0; x < SZ; ++x) Ssub[x] = gt * Stok[(size_t)t * SZ + x];
        for (int j = 0; j < nh; ++j) {
            const double *kk = J->k + (tok * nh + j) * (size_t)Dk;
            const double *vv = J->v + (tok * nh + j) * (size_t)Dv;
            const double bt = J->beta[tok * nh + j];
            const double *S0 = Ssub + (size_t)j * SZ;
            double *S1 = Ssub + (size_t)(j + 1) * SZ;
            double *ej = e + (size_t)j * Dv;
            for (int c = 0; c < Dv; ++c) ej[c] = vv[c];
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c) ej[c] -= S0[(size_t)r * Dv + c] * kk[r];
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c)
                    S1[(size_t)r * Dv + c] = S0[(size_t)r * Dv + c] + bt * kk[r] * ej[c];
        }
        /* readout o_t = Ssub[nh]^T q_t */
        const double *qq = J->q + tok * (size_t)Dk;
        const double *dd = J->d_o + tok * (size_t)Dv;
        const double *Sn = Ssub + (size_t)nh * SZ;
        double *dqq = J->dq + tok * (size_t)Dk;
        for (int r = 0; r < Dk; ++r) {
            double acc = 0.0;
            for (int c = 0; c < Dv; ++c) acc += Sn[(size_t)r * Dv + c] * dd[c];
            dqq[r] = acc;
            for (int c = 0; c < Dv; ++c) dS[(size_t)r * Dv + c] += qq[r] * dd[c];
        }
        /* sub-steps in reverse */
        for (int j = nh - 1; j >= 0; --j) {
            const double *kk = J->k + (tok * nh + j) * (size_t)Dk;
            const double bt = J->beta[tok * nh + j];
            const double *S0 = Ssub + (size_t)j * SZ;
            const double *ej = e + (size_t)j * Dv;
            double *dkk = J->dk + (tok * nh + j) * (size_t)Dk;
            double *dvv = J->dv + (tok * nh + j) * (size_t)Dv;
            double db = 0.0;
            for (int c = 0; c < Dv; ++c) du[c] = 0.0;
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c) du[c] += dS[(size_t)r * Dv + c] * kk[r];
            for (int c = 0; c < Dv; ++c) {
                dvv[c] = bt * du[c];
                db += du[c] * ej[c];
            }
            J->dbeta[tok * nh + j] = db;
            for (int r = 0; r < Dk; ++r) {
                double acc = 0.0;
                for (int c = 0; c < Dv; ++c)
                    acc += dS[(size_t)r * Dv + c] * (bt * ej[c]) - bt * S0[(size_t)r * Dv + c] * du[c];
                dkk[r] = acc;
            }
            for (int r = 0; r < Dk; ++r)
                for (int c = 0; c < Dv; ++c) dS[(size_t)r * Dv + c] -= bt * kk[r] * du[c];
        }
        /* gate */
        if (J->g) {
            double acc = 0.0;
            for (size_t x = 0; x < SZ; ++x) acc += dS[x] * Stok[(size_t)t * SZ + x];
            J->dg[tok] = acc;
            for (size_t x = 0; x < SZ; ++x) dS[x] *= gt;
        }
    }
    if (J->dh0) memcpy(J->dh0 + state_off, dS, sizeof(double) * SZ);
    free(Stok); free(Ssub); free(dS); free(e); free(du);
    return 0;
}

static void *worker_bwd(void *arg)
{
    oracle_bwd_job *J = (oracle_bwd_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int pair = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (pair >= J->B * J->H) break;
        if (run_pair_bwd(J, pair / J->H, pair % J->H) != 0) {
            pthread_mutex_lock(&J->lock);
            J->failed = 1;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/* Returns 0 on success, -1 on bad sizes, -2 on allocation/thread failure. */
int oracle_backward(int B, int T, int H, int Dk, int Dv, int nh,
                    const double *q, const double *k, const double *v,
                    const double *beta, const double *g, const double *h0,
                    const double *d_o, const double *dh_final,
                    double *dq, double *dk, double *dv, double *dbeta, double *dg,
                    double *dh0, int n_threads)
{
    if (B < 0 || T < 0 || H < 0 || Dk <= 0 || Dv <= 0 || nh <= 0) return -1;
    if (B * H > 0 && T > 0 && (!q || !k || !v || !beta || !d_o || !dq || !dk || !dv || !dbeta))
        return -1;
    if (g && !dg && T > 0) return -1;
    oracle_bwd_job J;
    J.B = B; J.T = T; J.H = H; J.Dk = Dk; J.Dv = Dv; J.nh = nh;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.d_o = d_o; J.dh_final = dh_final;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dbeta = dbeta; J.dg = dg; J.dh0 = dh0;
    J.next = 0;
    J.failed = 0;
    pthread_mutex_init(&J.lock, NULL);
    int nt = n_threads < 1 ? 1 : n_threads;
    if (nt > B * H) nt = B * H > 0 ? B * H : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return -2;
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker_bwd, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker_bwd(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? -2 : 0;
}
