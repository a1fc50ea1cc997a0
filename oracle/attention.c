/*
 * attention.c -- plain fp64 statement of scaled dot-product attention and its
 * gradients, the computation of "I built a GPT-2 in the browser, then made it
 * 2.6x-12.1x faster", section "Flash Attention 2".  TEST INFRASTRUCTURE ONLY,
 * like oracle.c: the product library never links or calls it.
 *
 * That section states the algorithm it accelerates without printing it:
 * attention rows S = q k^T, a softmax over each row, O = P V; the forward keeps
 * L = m + log(l) per query row (m the row maximum, l the sum of exp(S - m)),
 * and the backward rebuilds P = exp(S - L) from q and k.  Here every step is
 * the plain definition, in double, with the whole T x T score matrix of a head
 * formed explicitly -- no blocking, no online rescaling:
 *
 *   S[i][k] = scale * sum_d Q[i][d] K[k][d]      (k <= i when causal)
 *   L[i]    = m_i + log(sum_k exp(S[i][k] - m_i)),   m_i = max_k S[i][k]
 *   P[i][k] = exp(S[i][k] - L[i])                (0 for masked k)
 *   O[i][d] = sum_k P[i][k] V[k][d]
 *
 * and for a loss whose gradient with respect to O is dO:
 *
 *   dV[k][d] = sum_i P[i][k] dO[i][d]
 *   dP[i][k] = sum_d dO[i][d] V[k][d]
 *   D[i]     = sum_d dO[i][d] O[i][d]            (= sum_k P[i][k] dP[i][k])
 *   dS[i][k] = P[i][k] (dP[i][k] - D[i])
 *   dQ[i][d] = scale * sum_k dS[i][k] K[k][d]
 *   dK[k][d] = scale * sum_i dS[i][k] Q[i][d]
 *
 * Readings: tensors are [heads][T][D] row-major fp32 (a batch of B sequences of
 * H heads is BH = B H heads); `scale` is applied to the dot product; masked
 * scores take no part in the softmax (causal: key k > query i).
 *
 * Each output also gets a bound scale T, the sum of the magnitudes of the terms
 * of its last contraction with every earlier sum taken in magnitude:
 *   TO[i][d]  = sum_k P |V[k][d]|
 *   TdV[k][d] = sum_i P |dO[i][d]|
 *   TdQ[i][d] = scale sum_k P (|dP|[i][k] + |D|[i]) |K[k][d]|
 *   TdK[k][d] = scale sum_i P (|dP|[i][k] + |D|[i]) |Q[i][d]|
 * with |dP|[i][k] = sum_d |dO[i][d] V[k][d]| and |D|[i] = sum_d |dO[i][d] O[i][d]|,
 * so that cancellation inside dP - D does not shrink the scale below the size of
 * what was cancelled.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float *Q, *K, *V, *dO;
    int64_t h0, h1, T, D;
    int causal;
    double scale;
    double *O, *L, *TO;                 /* forward outputs (may be NULL in backward jobs) */
    double *dQ, *dK, *dV, *TdQ, *TdK, *TdV;
} attn_job;

/* P (T x T) of one head, from its scores; returns nothing, fills P and L. */
static void head_probs(const float *Q, const float *K, int64_t T, int64_t D, int causal, double scale,
                       double *P, double *L) {
    for (int64_t i = 0; i < T; ++i) {
        const int64_t kend = causal ? i + 1 : T;
        double m = -INFINITY;
        for (int64_t k = 0; k < kend; ++k) {
            double s = 0.0;
            for (int64_t d = 0; d < D; ++d) s += (double)Q[i * D + d] * (double)K[k * D + d];
            s *= scale;
            P[i * T + k] = s;
            if (s > m) m = s;
        }
        double l = 0.0;
        for (int64_t k = 0; k < kend; ++k) l += exp(P[i * T + k] - m);
        L[i] = m + log(l);
        for (int64_t k = 0; k < kend; ++k) P[i * T + k] = exp(P[i * T + k] - L[i]);
        for (int64_t k = kend; k < T; ++k) P[i * T + k] = 0.0;
    }
}

static void *fwd_thread(void *arg) {
    const attn_job *j = (const attn_job *)arg;
    const int64_t T = j->T, D = j->D;
    double *P = (double *)malloc((size_t)(T * T) * sizeof(double));
    for (int64_t h = j->h0; h < j->h1; ++h) {
        const float *Q = j->Q + h * T * D, *K = j->K + h * T * D, *V = j->V + h * T * D;
        head_probs(Q, K, T, D, j->causal, j->scale, P, j->L + h * T);
        for (int64_t i = 0; i < T; ++i)
            for (int64_t d = 0; d < D; ++d) {
                double o = 0.0, t = 0.0;
                for (int64_t k = 0; k < T; ++k) {
                    o += P[i * T + k] * (double)V[k * D + d];
                    t += P[i * T + k] * fabs((double)V[k * D + d]);
                }
                j->O[(h * T + i) * D + d] = o;
                j->TO[(h * T + i) * D + d] = t;
            }
    }
    free(P);
    return NULL;
}

static void *bwd_thread(void *arg) {
    const attn_job *j = (const attn_job *)arg;
    const int64_t T = j->T, D = j->D;
    double *P = (double *)malloc((size_t)(T * T) * sizeof(double));
    double *dS = (double *)malloc((size_t)(T * T) * sizeof(double));
    double *Ms = (double *)malloc((size_t)(T * T) * sizeof(double));  /* P (|dP| + |D|) */
    double *L = (double *)malloc((size_t)T * sizeof(double));
    double *O = (double *)malloc((size_t)(T * D) * sizeof(double));
    for (int64_t h = j->h0; h < j->h1; ++h) {
        const int64_t base = h * T * D;
        const float *Q = j->Q + base, *K = j->K + base, *V = j->V + base, *dO = j->dO + base;
        head_probs(Q, K, T, D, j->causal, j->scale, P, L);
        for (int64_t i = 0; i < T; ++i)
            for (int64_t d = 0; d < D; ++d) {
                double o = 0.0;
                for (int64_t k = 0; k < T; ++k) o += P[i * T + k] * (double)V[k * D + d];
                O[i * D + d] = o;
            }
        for (int64_t i = 0; i < T; ++i) {
            double Di = 0.0, Dabs = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                Di += (double)dO[i * D + d] * O[i * D + d];
                Dabs += fabs((double)dO[i * D + d] * O[i * D + d]);
            }
            for (int64_t k = 0; k < T; ++k) {
                double dp = 0.0, dpa = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    dp += (double)dO[i * D + d] * (double)V[k * D + d];
                    dpa += fabs((double)dO[i * D + d] * (double)V[k * D + d]);
                }
                dS[i * T + k] = P[i * T + k] * (dp - Di);
                Ms[i * T + k] = P[i * T + k] * (dpa + Dabs);
            }
        }
        for (int64_t k = 0; k < T; ++k)
            for (int64_t d = 0; d < D; ++d) {
                double v = 0.0, tv = 0.0, kk = 0.0, tk = 0.0;
                for (int64_t i = 0; i < T; ++i) {
                    v += P[i * T + k] * (double)dO[i * D + d];
                    tv += P[i * T + k] * fabs((double)dO[i * D + d]);
                    kk += dS[i * T + k] * (double)Q[i * D + d];
                    tk += Ms[i * T + k] * fabs((double)Q[i * D + d]);
                }
                j->dV[base + k * D + d] = v;
                j->TdV[base + k * D + d] = tv;
                j->dK[base + k * D + d] = j->scale * kk;
                j->TdK[base + k * D + d] = fabs(j->scale) * tk;
            }
        for (int64_t i = 0; i < T; ++i)
            for (int64_t d = 0; d < D; ++d) {
                double q = 0.0, tq = 0.0;
                for (int64_t k = 0; k < T; ++k) {
                    q += dS[i * T + k] * (double)K[k * D + d];
                    tq += Ms[i * T + k] * fabs((double)K[k * D + d]);
                }
                j->dQ[base + i * D + d] = j->scale * q;
                j->TdQ[base + i * D + d] = fabs(j->scale) * tq;
            }
    }
    free(P);
    free(dS);
    free(Ms);
    free(L);
    free(O);
    return NULL;
}

/* heads split over `threads` POSIX threads; each head is computed by one thread */
static void run_heads(attn_job *proto, int64_t BH, int threads, void *(*fn)(void *)) {
    if (threads < 1) threads = 1;
    if (threads > BH) threads = (int)BH;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    attn_job *jobs = (attn_job *)malloc(sizeof(attn_job) * (size_t)threads);
    for (int t = 0; t < threads; ++t) {
        jobs[t] = *proto;
        jobs[t].h0 = BH * t / threads;
        jobs[t].h1 = BH * (t + 1) / threads;
        pthread_create(&tid[t], NULL, fn, &jobs[t]);
    }
    for (int t = 0; t < threads; ++t) pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
}

void orc_attention_fwd(const float *Q, const float *K, const float *V, int64_t BH, int64_t T, int64_t D,
                       int causal, double scale, double *O, double *L, double *TO, int threads) {
    attn_job j;
    memset(&j, 0, sizeof(j));
    j.Q = Q;
    j.K = K;
    j.V = V;
    j.T = T;
    j.D = D;
    j.causal = causal;
    j.scale = scale;
    j.O = O;
    j.L = L;
    j.TO = TO;
    run_heads(&j, BH, threads, fwd_thread);
}

void orc_attention_bwd(const float *Q, const float *K, const float *V, const float *dO, int64_t BH, int64_t T,
                       int64_t D, int causal, double scale, double *dQ, double *dK, double *dV, double *TdQ,
                       double *TdK, double *TdV, int threads) {
    attn_job j;
    memset(&j, 0, sizeof(j));
    j.Q = Q;
    j.K = K;
    j.V = V;
    j.dO = dO;
    j.T = T;
    j.D = D;
    j.causal = causal;
    j.scale = scale;
    j.dQ = dQ;
    j.dK = dK;
    j.dV = dV;
    j.TdQ = TdQ;
    j.TdK = TdK;
    j.TdV = TdV;
    run_heads(&j, BH, threads, bwd_thread);
}
