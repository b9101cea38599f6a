/*
 * KDA oracle, chunked WY form, fp64.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as kda_recurrent.c; the two files share
 * no code with each other or with the CUDA library).
 *
 * This is the second, independently written form of the same result. It
 * follows the chunked algorithm the pages outline ("Kimi K3 的三個系統設計",
 * section "為什麼 FlashKDA 選擇 16-token chunks": cut the sequence into
 * 16-token chunks, invert a small triangular matrix per chunk, and propagate
 * the state from chunk to chunk), written out with exact per-pair
 * exponentials and no factoring, blocking or reordering:
 *
 *   chunk of L <= C tokens r = 0..L-1, state S (K x V) entering the chunk:
 *     G_r    = sum_{i<=r} g_i                    chunk-local cumulative log decay
 *     A[r,i] = beta_r sum_c k_rc k_ic exp(G_rc - G_ic)        for i < r
 *     Tm     = (I + A)^{-1}                      forward substitution
 *     W      = Tm diag(beta) (K . exp(G))        L x K
 *     Ut     = Tm diag(beta) V                   L x V
 *     U      = Ut - W S
 *     P[r,i] = sum_c q_rc k_ic exp(G_rc - G_ic)               for i <= r
 *     o_r    = scale ( (q_r . exp(G_r))^T S + sum_{i<=r} P[r,i] U_i )
 *     S     <- Diag(exp(G_{L-1})) S + sum_r (k_r . exp(G_{L-1} - G_r)) U_r^T
 *
 * Layouts and arguments are those of kda_oracle_recurrent, plus the chunk
 * size C (the method uses 16; other sizes are accepted so tests can check the
 * algebra at several sizes).
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
    int64_t N, H, K, V, C, out_tokens;
    double scale;
    double *out, *final_state;
    int64_t next;
    pthread_mutex_t mu;
    int err;
} chk_ctx;

typedef struct {
    double *S, *G, *A, *Tm, *W, *Ut, *U, *P;
} chk_buf;

static int chk_alloc(chk_buf *b, int64_t K, int64_t V, int64_t C)
{
    b->S = (double *)malloc(sizeof(double) * K * V);
    b->G = (double *)malloc(sizeof(double) * C * K);
    b->A = (double *)malloc(sizeof(double) * C * C);
    b->Tm = (double *)malloc(sizeof(double) * C * C);
    b->W = (double *)malloc(sizeof(double) * C * K);
    b->Ut = (double *)malloc(sizeof(double) * C * V);
    b->U = (double *)malloc(sizeof(double) * C * V);
    b->P = (double *)malloc(sizeof(double) * C * C);
    return b->S && b->G && b->A && b->Tm && b->W && b->Ut && b->U && b->P;
}

static void chk_free(chk_buf *b)
{
    free(b->S); free(b->G); free(b->A); free(b->Tm);
    free(b->W); free(b->Ut); free(b->U); free(b->P);
}

static void chk_one(chk_ctx *c, int64_t n, int64_t h, chk_buf *b)
{
    const int64_t K = c->K, V = c->V, H = c->H, C = c->C;
    double *S = b->S, *G = b->G, *A = b->A, *Tm = b->Tm;
    double *W = b->W, *Ut = b->Ut, *U = b->U, *P = b->P;

    if (c->s0)
        memcpy(S, c->s0 + (n * H + h) * K * V, sizeof(double) * K * V);
    else
        memset(S, 0, sizeof(double) * K * V);

    for (int64_t t0 = c->cu[n]; t0 < c->cu[n + 1]; t0 += C) {
        int64_t L = c->cu[n + 1] - t0;
        if (L > C) L = C;
#define KR(r, ch) ((double)c->k[((t0 + (r)) * H + h) * K + (ch)])
#define QR(r, ch) ((double)c->q[((t0 + (r)) * H + h) * K + (ch)])
#define VR(r, j) ((double)c->v[((t0 + (r)) * H + h) * V + (j)])
#define BR(r) ((double)c->beta[(t0 + (r)) * H + h])

        /* a1: chunk-local cumulative log decay */
        for (int64_t ch = 0; ch < K; ++ch) {
            double acc = 0.0;
            for (int64_t r = 0; r < L; ++r) {
                acc += (double)c->g[((t0 + r) * H + h) * K + ch];
                G[r * K + ch] = acc;
            }
        }

        /* a2: gated Gram A (strictly lower) and scores P (lower incl. diagonal) */
        for (int64_t r = 0; r < L; ++r)
            for (int64_t i = 0; i < L; ++i) {
                double a = 0.0, p = 0.0;
                if (i <= r) {
                    for (int64_t ch = 0; ch < K; ++ch) {
                        double e = exp(G[r * K + ch] - G[i * K + ch]);
                        a += KR(r, ch) * KR(i, ch) * e;
                        p += QR(r, ch) * KR(i, ch) * e;
                    }
                }
                A[r * C + i] = (i < r) ? BR(r) * a : 0.0;
                P[r * C + i] = (i <= r) ? p : 0.0;
            }

        /* a3: Tm = (I + A)^{-1}; row r of (I + A) Tm = I gives
         *     Tm[r, :] = e_r - sum_{i<r} A[r, i] Tm[i, :]                      */
        for (int64_t r = 0; r < L; ++r)
            for (int64_t j = 0; j < L; ++j) {
                double acc = (r == j) ? 1.0 : 0.0;
                for (int64_t i = 0; i < r; ++i) acc -= A[r * C + i] * Tm[i * C + j];
                Tm[r * C + j] = acc;
            }

        /* a4: WY tiles */
        for (int64_t r = 0; r < L; ++r) {
            for (int64_t ch = 0; ch < K; ++ch) {
                double acc = 0.0;
                for (int64_t i = 0; i < L; ++i)
                    acc += Tm[r * C + i] * BR(i) * KR(i, ch) * exp(G[i * K + ch]);
                W[r * K + ch] = acc;
            }
            for (int64_t j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < L; ++i) acc += Tm[r * C + i] * BR(i) * VR(i, j);
                Ut[r * V + j] = acc;
            }
        }

        /* a5: U = Ut - W S */
        for (int64_t r = 0; r < L; ++r)
            for (int64_t j = 0; j < V; ++j) {
                double acc = Ut[r * V + j];
                for (int64_t ch = 0; ch < K; ++ch) acc -= W[r * K + ch] * S[ch * V + j];
                U[r * V + j] = acc;
            }

        /* a5: outputs, from the state entering the chunk plus intra-chunk scores */
        for (int64_t r = 0; r < L; ++r) {
            int64_t t = t0 + r;
            if (t >= c->out_tokens) continue;
            double *ot = c->out + (t * H + h) * V;
            for (int64_t j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int64_t ch = 0; ch < K; ++ch)
                    acc += QR(r, ch) * exp(G[r * K + ch]) * S[ch * V + j];
                for (int64_t i = 0; i <= r; ++i) acc += P[r * C + i] * U[i * V + j];
                ot[j] = c->scale * acc;
            }
        }

        /* a5: state to the next chunk */
        for (int64_t ch = 0; ch < K; ++ch) {
            double gl = G[(L - 1) * K + ch];
            double dl = exp(gl);
            for (int64_t j = 0; j < V; ++j) {
                double acc = dl * S[ch * V + j];
                for (int64_t r = 0; r < L; ++r)
                    acc += KR(r, ch) * exp(gl - G[r * K + ch]) * U[r * V + j];
                S[ch * V + j] = acc;
            }
        }
#undef KR
#undef QR
#undef VR
#undef BR
    }
    if (c->final_state)
        memcpy(c->final_state + (n * H + h) * K * V, S, sizeof(double) * K * V);
}

static void *chk_worker(void *arg)
{
    chk_ctx *c = (chk_ctx *)arg;
    chk_buf b;
    if (!chk_alloc(&b, c->K, c->V, c->C)) {
        pthread_mutex_lock(&c->mu);
        c->err = 1;
        pthread_mutex_unlock(&c->mu);
        chk_free(&b);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&c->mu);
        int64_t w = c->next++;
        pthread_mutex_unlock(&c->mu);
        if (w >= c->N * c->H) break;
        chk_one(c, w / c->H, w % c->H, &b);
    }
    chk_free(&b);
    return NULL;
}

int kda_oracle_chunked(const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const double *s0, const int64_t *cu,
                       int64_t N, int64_t H, int64_t K, int64_t V, int64_t C, double scale,
                       double *out, int64_t out_tokens, double *final_state, int n_threads)
{
    if (!q || !k || !v || !g || !beta || !cu || N < 0 || H <= 0 || K <= 0 || V <= 0 || C <= 0)
        return 1;
    if (out_tokens > 0 && !out) return 1;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 1;

    chk_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = s0; c.cu = cu;
    c.N = N; c.H = H; c.K = K; c.V = V; c.C = C; c.out_tokens = out ? out_tokens : 0;
    c.scale = scale; c.out = out; c.final_state = final_state;
    pthread_mutex_init(&c.mu, NULL);

    int64_t work = N * H;
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > work) n_threads = (int)(work > 0 ? work : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return 2;
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, chk_worker, &c) != 0) break;
        ++started;
    }
    if (started == 0) chk_worker(&c);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&c.mu);
    return c.err ? 2 : 0;
}
