/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule (test infrastructure).
 *
 * THIS IS TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * What it computes: the plain per-token definition of the gated delta rule,
 * one (sequence, value-head) unit at a time, in double precision.  The FlashQLA
 * pages ("Usage / High-level API" and "Low-level API" of the project README)
 * fix the tensor shapes and the forward/backward entry points; the recurrence
 * itself is the Gated DeltaNet rule those pages accelerate:
 *
 *   a_t   = exp(g_t)
 *   p_t   = a_t * S_{t-1}^T k_t                  (V-vector, prediction)
 *   d_t   = beta_t * (v_t - p_t)                 (V-vector, delta)
 *   S_t   = a_t * S_{t-1} + k_t d_t^T            (K x V state)
 *   o_t   = scale * S_t^T q_t
 *
 * Backward (reverse-mode of the same steps, written out by hand), with
 * dS = dL/dS_t flowing backwards from dht (or 0):
 *
 *   dS   += scale * q_t do_t^T
 *   dq_t  = scale * S_t do_t
 *   dk_t  = dS d_t ;   dd = dS^T k_t
 *   dbeta_t = dd . (v_t - p_t) ;  dv_t = beta_t dd ;  dp = -beta_t dd
 *   dS'   = dS + k_t dp^T        (gradient of the decayed state a_t S_{t-1})
 *   dk_t += a_t S_{t-1} dp
 *   dg_t  = a_t <dS', S_{t-1}>
 *   dS   <- a_t dS'              (now dL/dS_{t-1})
 *   dh0   = dS at the sequence start.
 *
 * The forward states needed in reverse are recomputed from checkpoints taken
 * every CKPT tokens (no blocking or reordering of the arithmetic itself).
 *
 * Grouped value heads: q and k have Hq heads, v/g/beta/state have Hv heads,
 * Hv % Hq == 0, and value head hv reads query/key head hv / (Hv / Hq).
 * dq and dk are the sums over the value heads of a group.
 *
 * Varlen: with cu_seqlens (then B == 1) sequence s covers tokens
 * [cu[s], cu[s+1]) and has its own initial / final state.
 *
 * Layouts (row-major, contiguous): q,k [B,T,Hq,K]; v,o,do,dv [B,T,Hv,V];
 * g,beta,dg,dbeta [B,T,Hv]; h0,ht,dht,dh0 [N,Hv,K,V].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

typedef struct {
    int64_t B, T, Hq, Hv, K, V;
    int64_t n_seqs;
    const int64_t *cu;   /* nullable */
} shape_t;

static void seq_range(const shape_t *s, int64_t seq, int64_t *b, int64_t *t0, int64_t *t1) {
    if (s->cu) { *b = 0; *t0 = s->cu[seq]; *t1 = s->cu[seq + 1]; }
    else { *b = seq; *t0 = 0; *t1 = s->T; }
}

/* index helpers: token t of batch b */
static inline int64_t ix_qk(const shape_t *s, int64_t b, int64_t t, int64_t hq) {
    return ((b * s->T + t) * s->Hq + hq) * s->K;
}
static inline int64_t ix_v(const shape_t *s, int64_t b, int64_t t, int64_t hv) {
    return ((b * s->T + t) * s->Hv + hv) * s->V;
}
static inline int64_t ix_g(const shape_t *s, int64_t b, int64_t t, int64_t hv) {
    return (b * s->T + t) * s->Hv + hv;
}

/* One forward step: S <- a S + k d^T, returns d (and p) in the given buffers. */
static void fwd_step(int64_t K, int64_t V, double *S, const double *k, const double *v,
                     double g, double beta, double *p, double *d) {
    double a = exp(g);
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < K; ++i) acc += S[i * V + j] * k[i];
        p[j] = a * acc;
        d[j] = beta * (v[j] - p[j]);
    }
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < V; ++j)
            S[i * V + j] = a * S[i * V + j] + k[i] * d[j];
}

int gdn_oracle_fwd(int64_t B, int64_t T, int64_t Hq, int64_t Hv, int64_t K, int64_t V,
                   int64_t n_seqs, const int64_t *cu_seqlens,
                   const double *q, const double *k, const double *v, const double *g,
                   const double *beta, double scale, const double *h0,
                   double *o, double *ht, int n_threads) {
    if (Hq <= 0 || Hv % Hq != 0) return 1;
    if (cu_seqlens && B != 1) return 2;
    shape_t s = {B, T, Hq, Hv, K, V, cu_seqlens ? n_seqs : B, cu_seqlens};
    int64_t G = Hv / Hq;
    int64_t units = s.n_seqs * Hv;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int64_t seq = u / Hv, hv = u % Hv, hq = hv / G, b, t0, t1;
        seq_range(&s, seq, &b, &t0, &t1);
        double *S = (double *)malloc(sizeof(double) * K * V);
        double *p = (double *)malloc(sizeof(double) * V);
        double *d = (double *)malloc(sizeof(double) * V);
        if (h0) memcpy(S, h0 + (seq * Hv + hv) * K * V, sizeof(double) * K * V);
        else memset(S, 0, sizeof(double) * K * V);
        for (int64_t t = t0; t < t1; ++t) {
            const double *kt = k + ix_qk(&s, b, t, hq), *qt = q + ix_qk(&s, b, t, hq);
            fwd_step(K, V, S, kt, v + ix_v(&s, b, t, hv), g[ix_g(&s, b, t, hv)],
                     beta[ix_g(&s, b, t, hv)], p, d);
            double *ot = o + ix_v(&s, b, t, hv);
            for (int64_t j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i) acc += S[i * V + j] * qt[i];
                ot[j] = scale * acc;
            }
        }
        if (ht) memcpy(ht + (seq * Hv + hv) * K * V, S, sizeof(double) * K * V);
        free(S); free(p); free(d);
    }
    return 0;
}

/*
 * Backward.  One work item is (sequence, query head); it walks the G value
 * heads of the group one after the other so that dq / dk need no atomics.
 */
int gdn_oracle_bwd(int64_t B, int64_t T, int64_t Hq, int64_t Hv, int64_t K, int64_t V,
                   int64_t n_seqs, const int64_t *cu_seqlens,
                   const double *q, const double *k, const double *v, const double *g,
                   const double *beta, double scale, const double *h0,
                   const double *d_o, const double *dht,
                   double *dq, double *dk, double *dv, double *dbeta, double *dg,
                   double *dh0, int n_threads) {
    if (Hq <= 0 || Hv % Hq != 0) return 1;
    if (cu_seqlens && B != 1) return 2;
    shape_t s = {B, T, Hq, Hv, K, V, cu_seqlens ? n_seqs : B, cu_seqlens};
    int64_t G = Hv / Hq;
    int64_t units = s.n_seqs * Hq;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int64_t seq = u / Hq, hq = u % Hq, b, t0, t1;
        seq_range(&s, seq, &b, &t0, &t1);
        int64_t len = t1 - t0;
        int64_t n_ck = (len + CKPT - 1) / CKPT;
        double *ck = (double *)malloc(sizeof(double) * (n_ck > 0 ? n_ck : 1) * K * V);
        double *Sbuf = (double *)malloc(sizeof(double) * (CKPT + 1) * K * V);
        double *dS = (double *)malloc(sizeof(double) * K * V);
        double *p = (double *)malloc(sizeof(double) * V);
        double *d = (double *)malloc(sizeof(double) * V);
        double *dd = (double *)malloc(sizeof(double) * V);
        double *dp = (double *)malloc(sizeof(double) * V);
        /* zero dq / dk of this (seq, hq) once; the G value heads accumulate */
        for (int64_t t = t0; t < t1; ++t) {
            memset(dq + ix_qk(&s, b, t, hq), 0, sizeof(double) * K);
            memset(dk + ix_qk(&s, b, t, hq), 0, sizeof(double) * K);
        }
        for (int64_t gi = 0; gi < G; ++gi) {
            int64_t hv = hq * G + gi;
            int64_t st = (seq * Hv + hv) * K * V;
            /* forward sweep: checkpoint S before each block of CKPT tokens */
            double *S = Sbuf;
            if (h0) memcpy(S, h0 + st, sizeof(double) * K * V);
            else memset(S, 0, sizeof(double) * K * V);
            for (int64_t t = t0; t < t1; ++t) {
                if ((t - t0) % CKPT == 0) memcpy(ck + ((t - t0) / CKPT) * K * V, S, sizeof(double) * K * V);
                fwd_step(K, V, S, k + ix_qk(&s, b, t, hq), v + ix_v(&s, b, t, hv),
                         g[ix_g(&s, b, t, hv)], beta[ix_g(&s, b, t, hv)], p, d);
            }
            if (dht) memcpy(dS, dht + st, sizeof(double) * K * V);
            else memset(dS, 0, sizeof(double) * K * V);
            /* reverse sweep, block by block */
            for (int64_t c = n_ck - 1; c >= 0; --c) {
                int64_t b0 = t0 + c * CKPT, b1 = b0 + CKPT < t1 ? b0 + CKPT : t1;
                /* Sbuf[j] = state after token b0 + j - 1, i.e. Sbuf[0] = S_{b0-1} */
                memcpy(Sbuf, ck + c * K * V, sizeof(double) * K * V);
                for (int64_t t = b0; t < b1; ++t) {
                    double *Sn = Sbuf + (t - b0 + 1) * K * V;
                    memcpy(Sn, Sbuf + (t - b0) * K * V, sizeof(double) * K * V);
                    fwd_step(K, V, Sn, k + ix_qk(&s, b, t, hq), v + ix_v(&s, b, t, hv),
                             g[ix_g(&s, b, t, hv)], beta[ix_g(&s, b, t, hv)], p, d);
                }
                for (int64_t t = b1 - 1; t >= b0; --t) {
                    const double *Sprev = Sbuf + (t - b0) * K * V;   /* S_{t-1} */
                    const double *Scur = Sbuf + (t - b0 + 1) * K * V; /* S_t */
                    const double *kt = k + ix_qk(&s, b, t, hq), *qt = q + ix_qk(&s, b, t, hq);
                    const double *vt = v + ix_v(&s, b, t, hv), *dot = d_o + ix_v(&s, b, t, hv);
                    double gt = g[ix_g(&s, b, t, hv)], bt = beta[ix_g(&s, b, t, hv)];
                    double a = exp(gt);
                    /* recompute p_t and d_t from S_{t-1} */
                    for (int64_t j = 0; j < V; ++j) {
                        double acc = 0.0;
                        for (int64_t i = 0; i < K; ++i) acc += Sprev[i * V + j] * kt[i];
                        p[j] = a * acc;
                        d[j] = bt * (vt[j] - p[j]);
                    }
                    /* output o_t = scale S_t^T q_t */
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t j = 0; j < V; ++j) dS[i * V + j] += scale * qt[i] * dot[j];
                    double *dqt = dq + ix_qk(&s, b, t, hq), *dkt = dk + ix_qk(&s, b, t, hq);
                    for (int64_t i = 0; i < K; ++i) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < V; ++j) acc += Scur[i * V + j] * dot[j];
                        dqt[i] += scale * acc;
                    }
                    /* S_t = S' + k d^T */
                    for (int64_t j = 0; j < V; ++j) {
                        double acc = 0.0;
                        for (int64_t i = 0; i < K; ++i) acc += dS[i * V + j] * kt[i];
                        dd[j] = acc;
                    }
                    for (int64_t i = 0; i < K; ++i) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < V; ++j) acc += dS[i * V + j] * d[j];
                        dkt[i] += acc;
                    }
                    /* d = beta (v - p) */
                    double db = 0.0;
                    double *dvt = dv + ix_v(&s, b, t, hv);
                    for (int64_t j = 0; j < V; ++j) {
                        db += dd[j] * (vt[j] - p[j]);
                        dvt[j] = bt * dd[j];
                        dp[j] = -bt * dd[j];
                    }
                    dbeta[ix_g(&s, b, t, hv)] = db;
                    /* p = S'^T k with S' = a S_{t-1} */
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t j = 0; j < V; ++j) dS[i * V + j] += kt[i] * dp[j];
                    for (int64_t i = 0; i < K; ++i) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < V; ++j) acc += Sprev[i * V + j] * dp[j];
                        dkt[i] += a * acc;
                    }
                    /* S' = a S_{t-1} */
                    double da = 0.0;
                    for (int64_t e = 0; e < K * V; ++e) da += dS[e] * Sprev[e];
                    dg[ix_g(&s, b, t, hv)] = a * da;
                    for (int64_t e = 0; e < K * V; ++e) dS[e] *= a;
                }
            }
            if (dh0) memcpy(dh0 + st, dS, sizeof(double) * K * V);
        }
        free(ck); free(Sbuf); free(dS); free(p); free(d); free(dd); free(dp);
    }
    return 0;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
