/*
 * KDA oracle, gradients of the token recurrence (reverse mode), fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table
 * or constant with the CUDA library.
 *
 * The forward map is the recurrence of kda_recurrent.c (Kimi Delta
 * Attention: one fixed-size state per head, updated by every token; "Kimi K3
 * 的三個系統設計", section "第一個設計"; the pages mention that K3 trains
 * with KDA, "Kimi K3 開源基礎設施"):
 *
 *   S' = Diag(a_t) S_{t-1},  a_t = exp(g_t)
 *   u  = S'^T k_t,  w = v_t - u
 *   S_t = S' + beta_t k_t w^T
 *   o_t = scale S_t^T q_t
 *
 * Given dO = dL/do_t for every token and dS_T = dL/d(final state) (or 0),
 * this walks every sequence backwards, holding dS = dL/dS_t:
 *
 *   dS   += scale q_t dO_t^T                (o_t reads S_t)
 *   dq_t  = scale S_t dO_t
 *   x     = dS^T k_t
 *   dv_t  = beta_t x
 *   dbeta = w . x
 *   dk_t  = beta_t (dS w - S' x)
 *   dS'   = dS - beta_t k_t x^T
 *   dg_t  = a_t * rowsum(dS' o S_{t-1})     (o: elementwise)
 *   dS    = Diag(a_t) dS'                   (= dL/dS_{t-1})
 *
 * and ends with dL/d(initial state) = dS. Each line is the derivative of
 * one line of the forward map above. The states S_{t-1} are kept from a
 * forward pass over the sequence (no recomputation), which also yields o and
 * the final state: the pin tests compare those with kda_recurrent.c and the
 * gradients with central differences of this forward pass.
 *
 * All inputs and outputs are double. Layouts as in kda_recurrent.c:
 * q,k,g [T, H, K]; v [T, H, V]; beta [T, H]; s0 [N, H, K, V] or NULL;
 * cu [N+1]; dout [T, H, V]; dsf [N, H, K, V] or NULL (zero). Outputs: o
 * [T, H, V] and fs [N, H, K, V] (each may be NULL), dq, dk, dg [T, H, K], dv
 * [T, H, V], dbeta [T, H], ds0 [N, H, K, V].
 *
 * `mutation` plants a known mistake in the reverse pass (0 = none), so the
 * pin tests can show that the finite-difference pins catch it:
 *   1: the S' x term of dk dropped
 *   2: dS passed back without the decay a_t
 *   3: the erase term of dS' added instead of subtracted
 *   4: dq from S_{t-1} instead of S_t
 *   5: dg without the factor a_t
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *s0, *dout, *dsf;
    const int64_t *cu;
    int64_t N, H, K, V, Lmax;
    double scale;
    double *o, *fs, *dq, *dk, *dv, *dg, *dbeta, *ds0;
    int mutation;
    int64_t next;
    pthread_mutex_t mu;
    int err;
} bwd_ctx;

/* One (sequence n, head h): forward with every state kept, then reverse. */
static void bwd_one(const bwd_ctx *c, int64_t n, int64_t h, double *hist, double *dS, double *Sp,
                    double *St, double *a, double *w, double *x)
{
    const int64_t H = c->H, K = c->K, V = c->V, KV = K * V;
    const double *q = c->q, *k = c->k, *v = c->v, *g = c->g, *beta = c->beta;
    const double scale = c->scale;
    const int mutation = c->mutation;
    const int64_t t0 = c->cu[n], L = c->cu[n + 1] - c->cu[n];

    /* ---- forward: hist[j] = state before token t0 + j */
    if (c->s0)
        memcpy(hist, c->s0 + (n * H + h) * KV, sizeof(double) * (size_t)KV);
    else
        memset(hist, 0, sizeof(double) * (size_t)KV);
    for (int64_t j = 0; j < L; ++j) {
        const int64_t t = t0 + j;
        const double *kt = k + (t * H + h) * K, *vt = v + (t * H + h) * V;
        const double *gt = g + (t * H + h) * K, *qt = q + (t * H + h) * K;
        const double b = beta[t * H + h];
        const double *S0 = hist + j * KV;
        double *S1 = hist + (j + 1) * KV;
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) S1[i * V + cc] = exp(gt[i]) * S0[i * V + cc];
        for (int64_t cc = 0; cc < V; ++cc) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) acc += S1[i * V + cc] * kt[i];
            w[cc] = vt[cc] - acc;
        }
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) S1[i * V + cc] += b * kt[i] * w[cc];
        if (c->o) {
            double *ot = c->o + (t * H + h) * V;
            for (int64_t cc = 0; cc < V; ++cc) {
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i) acc += S1[i * V + cc] * qt[i];
                ot[cc] = scale * acc;
            }
        }
    }
    if (c->fs) memcpy(c->fs + (n * H + h) * KV, hist + L * KV, sizeof(double) * (size_t)KV);

    /* ---- reverse */
    if (c->dsf)
        memcpy(dS, c->dsf + (n * H + h) * KV, sizeof(double) * (size_t)KV);
    else
        memset(dS, 0, sizeof(double) * (size_t)KV);
    for (int64_t j = L - 1; j >= 0; --j) {
        const int64_t t = t0 + j;
        const double *kt = k + (t * H + h) * K, *vt = v + (t * H + h) * V;
        const double *gt = g + (t * H + h) * K, *qt = q + (t * H + h) * K;
        const double *dot = c->dout + (t * H + h) * V;
        const double b = beta[t * H + h];
        const double *Sprev = hist + j * KV;
        for (int64_t i = 0; i < K; ++i) a[i] = exp(gt[i]);
        /* S', w, S_t again (the forward lines) */
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) Sp[i * V + cc] = a[i] * Sprev[i * V + cc];
        for (int64_t cc = 0; cc < V; ++cc) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) acc += Sp[i * V + cc] * kt[i];
            w[cc] = vt[cc] - acc;
        }
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) St[i * V + cc] = Sp[i * V + cc] + b * kt[i] * w[cc];
        /* o_t = scale S_t^T q_t */
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) dS[i * V + cc] += scale * qt[i] * dot[cc];
        const double *Sq = (mutation == 4) ? Sprev : St;
        for (int64_t i = 0; i < K; ++i) {
            double acc = 0.0;
            for (int64_t cc = 0; cc < V; ++cc) acc += Sq[i * V + cc] * dot[cc];
            c->dq[(t * H + h) * K + i] = scale * acc;
        }
        /* S_t = S' + beta k w^T, w = v - S'^T k */
        for (int64_t cc = 0; cc < V; ++cc) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) acc += dS[i * V + cc] * kt[i];
            x[cc] = acc;
            c->dv[(t * H + h) * V + cc] = b * acc;
        }
        {
            double acc = 0.0;
            for (int64_t cc = 0; cc < V; ++cc) acc += w[cc] * x[cc];
            c->dbeta[t * H + h] = acc;
        }
        for (int64_t i = 0; i < K; ++i) {
            double dsw = 0.0, spx = 0.0;
            for (int64_t cc = 0; cc < V; ++cc) {
                dsw += dS[i * V + cc] * w[cc];
                spx += Sp[i * V + cc] * x[cc];
            }
            c->dk[(t * H + h) * K + i] = (mutation == 1) ? b * dsw : b * (dsw - spx);
        }
        for (int64_t i = 0; i < K; ++i)
            for (int64_t cc = 0; cc < V; ++cc) {
                const double e = b * kt[i] * x[cc];
                dS[i * V + cc] += (mutation == 3) ? e : -e;
            }
        /* S' = Diag(a) S_{t-1} */
        for (int64_t i = 0; i < K; ++i) {
            double acc = 0.0;
            for (int64_t cc = 0; cc < V; ++cc) acc += dS[i * V + cc] * Sprev[i * V + cc];
            c->dg[(t * H + h) * K + i] = (mutation == 5) ? acc : a[i] * acc;
        }
        if (mutation != 2)
            for (int64_t i = 0; i < K; ++i)
                for (int64_t cc = 0; cc < V; ++cc) dS[i * V + cc] *= a[i];
    }
    memcpy(c->ds0 + (n * H + h) * KV, dS, sizeof(double) * (size_t)KV);
}

static void *bwd_worker(void *arg)
{
    bwd_ctx *c = (bwd_ctx *)arg;
    const int64_t KV = c->K * c->V;
    double *hist = (double *)malloc(sizeof(double) * (size_t)((c->Lmax + 1) * KV));
    double *dS = (double *)malloc(sizeof(double) * (size_t)KV);
    double *Sp = (double *)malloc(sizeof(double) * (size_t)KV);
    double *St = (double *)malloc(sizeof(double) * (size_t)KV);
    double *a = (double *)malloc(sizeof(double) * (size_t)c->K);
    double *w = (double *)malloc(sizeof(double) * (size_t)c->V);
    double *x = (double *)malloc(sizeof(double) * (size_t)c->V);
    if (!hist || !dS || !Sp || !St || !a || !w || !x) {
        pthread_mutex_lock(&c->mu);
        c->err = 1;
        pthread_mutex_unlock(&c->mu);
    } else {
        for (;;) {
            pthread_mutex_lock(&c->mu);
            const int64_t u = c->next++;
            pthread_mutex_unlock(&c->mu);
            if (u >= c->N * c->H) break;
            bwd_one(c, u / c->H, u % c->H, hist, dS, Sp, St, a, w, x);
        }
    }
    free(hist); free(dS); free(Sp); free(St); free(a); free(w); free(x);
    return NULL;
}

/* Returns 0 on success, 1 on a bad argument, 2 on an allocation failure.
 * n_threads <= 0 uses every online core; each (sequence, head) is one task. */
int kda_oracle_backward(const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const double *s0, const int64_t *cu, int64_t N,
                        int64_t H, int64_t K, int64_t V, double scale, const double *dout,
                        const double *dsf, double *o, double *fs, double *dq, double *dk,
                        double *dv, double *dg, double *dbeta, double *ds0, int n_threads,
                        int mutation)
{
    if (!q || !k || !v || !g || !beta || !cu || !dout || !dq || !dk || !dv || !dg || !dbeta ||
        !ds0 || N < 0 || H <= 0 || K <= 0 || V <= 0)
        return 1;
    bwd_ctx c;
    memset(&c, 0, sizeof(c));
    for (int64_t n = 0; n < N; ++n) {
        if (cu[n + 1] < cu[n]) return 1;
        if (cu[n + 1] - cu[n] > c.Lmax) c.Lmax = cu[n + 1] - cu[n];
    }
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = s0; c.dout = dout; c.dsf = dsf;
    c.cu = cu; c.N = N; c.H = H; c.K = K; c.V = V; c.scale = scale;
    c.o = o; c.fs = fs; c.dq = dq; c.dk = dk; c.dv = dv; c.dg = dg; c.dbeta = dbeta; c.ds0 = ds0;
    c.mutation = mutation;
    pthread_mutex_init(&c.mu, NULL);
    const int64_t work = N * H;
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > work) n_threads = (int)(work > 0 ? work : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return 2;
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, bwd_worker, &c) != 0) break;
        ++started;
    }
    if (started == 0) bwd_worker(&c);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&c.mu);
    return c.err ? 2 : 0;
}
