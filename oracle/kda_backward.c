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
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

int kda_oracle_backward(const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const double *s0, const int64_t *cu, int64_t N,
                        int64_t H, int64_t K, int64_t V, double scale, const double *dout,
                        const double *dsf, double *o, double *fs, double *dq, double *dk,
                        double *dv, double *dg, double *dbeta, double *ds0, int mutation)
{
    if (!q || !k || !v || !g || !beta || !cu || !dout || !dq || !dk || !dv || !dg || !dbeta ||
        !ds0 || N < 0 || H <= 0 || K <= 0 || V <= 0)
        return 1;
    int64_t Lmax = 0;
    for (int64_t n = 0; n < N; ++n) {
        if (cu[n + 1] < cu[n]) return 1;
        if (cu[n + 1] - cu[n] > Lmax) Lmax = cu[n + 1] - cu[n];
    }
    const int64_t KV = K * V;
    /* states before every token of one sequence, plus the final one */
    double *hist = (double *)malloc(sizeof(double) * (size_t)((Lmax + 1) * KV));
    double *dS = (double *)malloc(sizeof(double) * (size_t)KV);
    double *Sp = (double *)malloc(sizeof(double) * (size_t)KV);   /* S' */
    double *St = (double *)malloc(sizeof(double) * (size_t)KV);   /* S_t */
    double *a = (double *)malloc(sizeof(double) * (size_t)K);
    double *u = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *x = (double *)malloc(sizeof(double) * (size_t)V);
    if (!hist || !dS || !Sp || !St || !a || !u || !w || !x) {
        free(hist); free(dS); free(Sp); free(St); free(a); free(u); free(w); free(x);
        return 2;
    }
    for (int64_t n = 0; n < N; ++n) {
        const int64_t t0 = cu[n], L = cu[n + 1] - cu[n];
        for (int64_t h = 0; h < H; ++h) {
            /* ---- forward: hist[j] = state before token t0 + j */
            if (s0)
                memcpy(hist, s0 + (n * H + h) * KV, sizeof(double) * (size_t)KV);
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
                    for (int64_t c = 0; c < V; ++c) S1[i * V + c] = exp(gt[i]) * S0[i * V + c];
                for (int64_t c = 0; c < V; ++c) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < K; ++i) acc += S1[i * V + c] * kt[i];
                    w[c] = vt[c] - acc;
                }
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t c = 0; c < V; ++c) S1[i * V + c] += b * kt[i] * w[c];
                if (o) {
                    double *ot = o + (t * H + h) * V;
                    for (int64_t c = 0; c < V; ++c) {
                        double acc = 0.0;
                        for (int64_t i = 0; i < K; ++i) acc += S1[i * V + c] * qt[i];
                        ot[c] = scale * acc;
                    }
                }
            }
            if (fs) memcpy(fs + (n * H + h) * KV, hist + L * KV, sizeof(double) * (size_t)KV);

            /* ---- reverse */
            if (dsf)
                memcpy(dS, dsf + (n * H + h) * KV, sizeof(double) * (size_t)KV);
            else
                memset(dS, 0, sizeof(double) * (size_t)KV);
            for (int64_t j = L - 1; j >= 0; --j) {
                const int64_t t = t0 + j;
                const double *kt = k + (t * H + h) * K, *vt = v + (t * H + h) * V;
                const double *gt = g + (t * H + h) * K, *qt = q + (t * H + h) * K;
                const double *dot = dout + (t * H + h) * V;
                const double b = beta[t * H + h];
                const double *Sprev = hist + j * KV;
                for (int64_t i = 0; i < K; ++i) a[i] = exp(gt[i]);
                /* S', u, w, S_t again (the forward lines) */
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t c = 0; c < V; ++c) Sp[i * V + c] = a[i] * Sprev[i * V + c];
                for (int64_t c = 0; c < V; ++c) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < K; ++i) acc += Sp[i * V + c] * kt[i];
                    u[c] = acc;
                    w[c] = vt[c] - acc;
                }
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t c = 0; c < V; ++c)
                        St[i * V + c] = Sp[i * V + c] + b * kt[i] * w[c];
                /* o_t = scale S_t^T q_t */
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t c = 0; c < V; ++c) dS[i * V + c] += scale * qt[i] * dot[c];
                const double *Sq = (mutation == 4) ? Sprev : St;
                for (int64_t i = 0; i < K; ++i) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < V; ++c) acc += Sq[i * V + c] * dot[c];
                    dq[t * H * K + h * K + i] = scale * acc;
                }
                /* S_t = S' + beta k w^T, w = v - S'^T k */
                for (int64_t c = 0; c < V; ++c) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < K; ++i) acc += dS[i * V + c] * kt[i];
                    x[c] = acc;
                    dv[(t * H + h) * V + c] = b * acc;
                }
                {
                    double acc = 0.0;
                    for (int64_t c = 0; c < V; ++c) acc += w[c] * x[c];
                    dbeta[t * H + h] = acc;
                }
                for (int64_t i = 0; i < K; ++i) {
                    double dsw = 0.0, spx = 0.0;
                    for (int64_t c = 0; c < V; ++c) {
                        dsw += dS[i * V + c] * w[c];
                        spx += Sp[i * V + c] * x[c];
                    }
                    dk[(t * H + h) * K + i] = (mutation == 1) ? b * dsw : b * (dsw - spx);
                }
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t c = 0; c < V; ++c) {
                        const double e = b * kt[i] * x[c];
                        dS[i * V + c] += (mutation == 3) ? e : -e;
                    }
                /* S' = Diag(a) S_{t-1} */
                for (int64_t i = 0; i < K; ++i) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < V; ++c) acc += dS[i * V + c] * Sprev[i * V + c];
                    dg[(t * H + h) * K + i] = (mutation == 5) ? acc : a[i] * acc;
                }
                if (mutation != 2)
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t c = 0; c < V; ++c) dS[i * V + c] *= a[i];
            }
            memcpy(ds0 + (n * H + h) * KV, dS, sizeof(double) * (size_t)KV);
        }
    }
    free(hist); free(dS); free(Sp); free(St); free(a); free(u); free(w); free(x);
    return 0;
}
