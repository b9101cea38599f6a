/*
 * KDA oracle, token-by-token recurrence, fp64.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against. Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no
 * code, header, table or constant with the CUDA library.
 *
 * What it computes (Kimi Delta Attention; the pages "Kimi K3 的三個系統設計",
 * section "第一個設計", and "Kimi K3 開源基礎設施", section "FlashKDA", state
 * that KDA keeps one fixed-size recurrent state per head that every new token
 * updates; the update rule itself is the gated delta rule with a per-channel
 * decay):
 *
 *   for every sequence n and head h, S starts at initial_state[n,h] (or 0):
 *     for each token t of the sequence:
 *       S <- Diag(exp(g_t)) S                    (decay acts on the key rows)
 *       S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T
 *       o_t = scale * S^T q_t                    (post-update state)
 *     final_state[n,h] = S
 *
 * S is K x V (row = key channel, column = value channel), row-major.
 * Inputs are fp32 arrays holding exactly the values the GPU sees (bf16 q/k/v
 * promote to fp32 without change); all arithmetic is in double.
 *
 * Layouts: q,k,g [T_total, H, K]; v [T_total, H, V]; beta [T_total, H];
 * s0 [N, H, K, V] or NULL; cu [N+1] token offsets of the packed sequences;
 * out [out_tokens, H, V] (only tokens t < out_tokens are written);
 * final_state [N, H, K, V].
 *
 * `flags` asks for the input preprocessing that the library can do inside
 * its kernels (the pages leave the production of q, k and g to the model, so
 * these are readings, not page text): bit 1 = q and k are raw, use
 * x / sqrt(sum_i x_i^2 + 1e-6) per (token, head); bit 2 = g holds gate
 * logits x, use the log decay logsigmoid(x) = -log(1 + exp(-x)).
 *
 * `mutation` plants a known mistake (0 = none). It exists so the pin tests
 * can show that each pin catches the mistakes it is meant to catch:
 *   1: o_t from the pre-update state S_{t-1}
 *   2: decay applied to the value columns instead of the key rows (K == V)
 *   3: delta term added with the wrong sign
 *   4: beta dropped from the erase term (S - k k^T S)
 *   5: decay applied after the delta update instead of before
 *   6: scale applied twice
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v, *g, *beta;
    const double *s0;
    const int64_t *cu;
    int64_t N, H, K, V, out_tokens;
    double scale;
    double *out, *final_state;
    int flags;
    int mutation;
    int64_t next;
    pthread_mutex_t mu;
    int err;
} rec_ctx;

/* logsigmoid(x) = -log(1 + e^-x), written so that neither branch overflows */
static double log_sigmoid(double x)
{
    return x >= 0.0 ? -log1p(exp(-x)) : x - log1p(exp(x));
}

/* 1 / sqrt(sum x_i^2 + 1e-6), or 1 when the inputs are used as given */
static double inv_norm(const float *x, int64_t n, int on)
{
    if (!on) return 1.0;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
    return 1.0 / sqrt(ss + 1e-6);
}

static void rec_one(rec_ctx *c, int64_t n, int64_t h, double *S, double *kS, double *dec)
{
    const int64_t K = c->K, V = c->V, H = c->H;
    const int m = c->mutation;
    if (c->s0)
        memcpy(S, c->s0 + (n * H + h) * K * V, sizeof(double) * K * V);
    else
        memset(S, 0, sizeof(double) * K * V);

    for (int64_t t = c->cu[n]; t < c->cu[n + 1]; ++t) {
        const float *qt = c->q + (t * H + h) * K;
        const float *kt = c->k + (t * H + h) * K;
        const float *gt = c->g + (t * H + h) * K;
        const float *vt = c->v + (t * H + h) * V;
        const double b = (double)c->beta[t * H + h];
        const double rq = inv_norm(qt, K, c->flags & 1), rk = inv_norm(kt, K, c->flags & 1);

        for (int64_t i = 0; i < K; ++i)
            dec[i] = exp((c->flags & 2) ? log_sigmoid((double)gt[i]) : (double)gt[i]);

        /* pre-update output, for mutation 1 only */
        if (m == 1 && t < c->out_tokens) {
            double *ot = c->out + (t * H + h) * V;
            for (int64_t j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i) acc += S[i * V + j] * (double)qt[i] * rq;
                ot[j] = c->scale * acc;
            }
        }

        /* S <- Diag(exp g_t) S */
        if (m != 5) {
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    S[i * V + j] *= (m == 2) ? dec[j] : dec[i];
        }

        /* kS = k_t^T S */
        for (int64_t j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) acc += (double)kt[i] * rk * S[i * V + j];
            kS[j] = acc;
        }

        /* S <- S - beta k (k^T S) + beta k v^T */
        for (int64_t i = 0; i < K; ++i) {
            const double ki = (double)kt[i] * rk;
            for (int64_t j = 0; j < V; ++j) {
                double erase = (m == 4) ? ki * kS[j] : b * ki * kS[j];
                double write = b * ki * (double)vt[j];
                if (m == 3)
                    S[i * V + j] += erase - write;
                else
                    S[i * V + j] += write - erase;
            }
        }

        if (m == 5) {
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) S[i * V + j] *= dec[i];
        }

        /* o_t = scale * S^T q_t */
        if (m != 1 && t < c->out_tokens) {
            double *ot = c->out + (t * H + h) * V;
            for (int64_t j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i) acc += S[i * V + j] * (double)qt[i] * rq;
                ot[j] = (m == 6) ? c->scale * c->scale * acc : c->scale * acc;
            }
        }
    }
    if (c->final_state)
        memcpy(c->final_state + (n * H + h) * K * V, S, sizeof(double) * K * V);
}

static void *rec_worker(void *arg)
{
    rec_ctx *c = (rec_ctx *)arg;
    double *S = (double *)malloc(sizeof(double) * c->K * c->V);
    double *kS = (double *)malloc(sizeof(double) * c->V);
    double *dec = (double *)malloc(sizeof(double) * (c->K > c->V ? c->K : c->V));
    if (!S || !kS || !dec) {
        pthread_mutex_lock(&c->mu);
        c->err = 1;
        pthread_mutex_unlock(&c->mu);
        free(S); free(kS); free(dec);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&c->mu);
        int64_t w = c->next++;
        pthread_mutex_unlock(&c->mu);
        if (w >= c->N * c->H) break;
        rec_one(c, w / c->H, w % c->H, S, kS, dec);
    }
    free(S); free(kS); free(dec);
    return NULL;
}

/* Returns 0 on success, nonzero on a bad argument or an allocation failure. */
int kda_oracle_recurrent(const float *q, const float *k, const float *v, const float *g,
                         const float *beta, const double *s0, const int64_t *cu,
                         int64_t N, int64_t H, int64_t K, int64_t V, double scale,
                         double *out, int64_t out_tokens, double *final_state,
                         int n_threads, int flags, int mutation)
{
    if (!q || !k || !v || !g || !beta || !cu || N < 0 || H <= 0 || K <= 0 || V <= 0) return 1;
    if (out_tokens > 0 && !out) return 1;
    if (mutation == 2 && K != V) return 1;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 1;

    rec_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = s0; c.cu = cu;
    c.N = N; c.H = H; c.K = K; c.V = V; c.out_tokens = out ? out_tokens : 0;
    c.scale = scale; c.out = out; c.final_state = final_state; c.mutation = mutation;
    c.flags = flags;
    pthread_mutex_init(&c.mu, NULL);

    int64_t work = N * H;
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > work) n_threads = (int)(work > 0 ? work : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return 2;
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, rec_worker, &c) != 0) break;
        ++started;
    }
    if (started == 0) rec_worker(&c);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&c.mu);
    return c.err ? 2 : 0;
}
