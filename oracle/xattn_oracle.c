/*
 * Reference oracle: causal scaled-dot-product attention with grouped KV heads,
 * forward and backward, in plain fp64 loops.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's library. The product path (libxattn and
 * its Python binding) never calls it and shares no code with it.
 *
 * What it computes, and where that is stated:
 *   - xtrain "演进总览" (docs/evolution.md), phase table row T14: attention is one
 *     fused op over causal scores; the forward keeps a per-row softmax statistic and
 *     the backward recomputes the scores and uses D_i = sum_d dO_id * O_id in place of
 *     the full softmax Jacobian.
 *   - same table, row T15: grouped KV heads. Query head h reads kv head h / group
 *     (the broadcast maps kv head kvh to query heads kvh*group + r, r < group), and
 *     the backward of that broadcast sums the group's gradients into the kv head.
 *   - xtrain "Known Issues & Perf Backlog" (docs/known-issues.md), KI-1 fix: the
 *     attention is a causal softmax over scaled scores (composed form).
 *   - xserv "Phase 21" page is not used.
 *
 * This file does not use the fused algorithm. It evaluates the plain definition:
 *
 *   s_ij  = scale * sum_d q[b,i,h,d] * k[b,j,kvh,d]        for j <= i
 *   LSE_i = log( sum_{j<=i} exp(s_ij) )                      (natural log)
 *   P_ij  = exp(s_ij - LSE_i)
 *   O_i   = sum_{j<=i} P_ij v[b,j,kvh,:]
 *   dP_ij = dO_i . v_j ,  D_i = dO_i . O_i ,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_{j<=i} dS_ij k_j
 *   dK_j  = scale * sum_{r<group} sum_{i>=j} dS^(h=kvh*group+r)_ij q_i
 *   dV_j  =         sum_{r<group} sum_{i>=j} P^(h)_ij dO^(h)_i
 *
 * LSE uses the row maximum as a shift only to avoid overflow of exp; that does not
 * change the value. All tensors are row-major [B, S, heads, hd] (lse: [B, S, nh]).
 *
 * Decode (xtrain "演进总览", post-training milestones M2a-M2c: one new query per
 * sequence against that sequence's cached keys and values, equal to the last row of
 * full causal attention, batch-agnostic over the sequences), xo_decode:
 *
 *   s_j = scale * sum_d q[b,h,d] * k[b,j,kvh,d]      for every cached j < T
 *   LSE = log( sum_j exp(s_j) ) ,  O = sum_j exp(s_j - LSE) v[b,j,kvh,:]
 *
 * with q, o [B, nh, hd], k, v [B, T, nkv, hd], lse [B, nh]. The query sits at the
 * newest position, so all T cached keys, its own included, are visible.
 *
 * ORACLE_MUTATION (compile-time, tests only): a nonzero value plants one known
 * mistake, so the test suite can show that its pins catch it. The default build
 * has ORACLE_MUTATION == 0 and contains none of them.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

#define IDX4(b, s, h, d, S, H, HD) ((((size_t)(b) * (S) + (s)) * (H) + (h)) * (HD) + (d))

static double dot(const double *x, const double *y, int n) {
    double acc = 0.0;
    for (int d = 0; d < n; ++d) acc += x[d] * y[d];
    return acc;
}

/* kv head read by query head h. */
static int kv_head_of(int h, int nh, int nkv) {
#if ORACLE_MUTATION == 2
    (void)nh;
    return h % nkv;               /* planted: interleaved instead of contiguous groups */
#else
    return h / (nh / nkv);
#endif
}

/* Is key j visible from query i? Causal, diagonal included. */
static int visible(int i, int j) {
#if ORACLE_MUTATION == 1
    return j >= i;                /* planted: mask flipped to the future */
#else
    return j <= i;
#endif
}

/* Score s_ij for one (b, h). */
static double score(const double *q, const double *k, int b, int i, int j, int h, int kvh,
                    int S, int nh, int nkv, int hd, double scale) {
    double s = dot(&q[IDX4(b, i, h, 0, S, nh, hd)], &k[IDX4(b, j, kvh, 0, S, nkv, hd)], hd);
#if ORACLE_MUTATION == 9
    return scale * scale * s;     /* planted: scale applied twice */
#else
    return scale * s;
#endif
}

/* Row i of (b, h): log-sum-exp of the visible scores. */
static double row_lse(const double *q, const double *k, int b, int i, int h, int kvh,
                      int S, int nh, int nkv, int hd, double scale) {
    double mx = -INFINITY;
    for (int j = 0; j < S; ++j)
        if (visible(i, j)) {
            double s = score(q, k, b, i, j, h, kvh, S, nh, nkv, hd, scale);
            if (s > mx) mx = s;
        }
    double sum = 0.0;
    for (int j = 0; j < S; ++j)
        if (visible(i, j)) sum += exp(score(q, k, b, i, j, h, kvh, S, nh, nkv, hd, scale) - mx);
#if ORACLE_MUTATION == 6
    return mx + log2(sum);        /* planted: base-2 log */
#else
    return mx + log(sum);
#endif
}

/*
 * Forward: o [B,S,nh,hd], lse [B,S,nh].
 */
void xo_fwd(const double *q, const double *k, const double *v, int B, int S, int nh, int nkv,
            int hd, double scale, double *o, double *lse) {
    long total = (long)B * nh * S;
#pragma omp parallel for schedule(dynamic, 8)
    for (long t = 0; t < total; ++t) {
        int i = (int)(t % S);
        int h = (int)((t / S) % nh);
        int b = (int)(t / ((long)S * nh));
        int kvh = kv_head_of(h, nh, nkv);
        double L = row_lse(q, k, b, i, h, kvh, S, nh, nkv, hd, scale);
        lse[((size_t)b * S + i) * nh + h] = L;
        double *oi = &o[IDX4(b, i, h, 0, S, nh, hd)];
        for (int d = 0; d < hd; ++d) oi[d] = 0.0;
        for (int j = 0; j < S; ++j) {
            if (!visible(i, j)) continue;
            double p = exp(score(q, k, b, i, j, h, kvh, S, nh, nkv, hd, scale) - L);
            const double *vj = &v[IDX4(b, j, kvh, 0, S, nkv, hd)];
            for (int d = 0; d < hd; ++d) oi[d] += p * vj[d];
        }
    }
}

/* D_i = dO_i . O_i for one row (O taken from this oracle's own forward). */
static double row_D(const double *dO, const double *o, int b, int i, int h, int S, int nh, int hd) {
#if ORACLE_MUTATION == 4
    (void)o;
    double acc = 0.0;             /* planted: the O factor dropped */
    for (int d = 0; d < hd; ++d) acc += dO[IDX4(b, i, h, d, S, nh, hd)];
    return acc;
#else
    return dot(&dO[IDX4(b, i, h, 0, S, nh, hd)], &o[IDX4(b, i, h, 0, S, nh, hd)], hd);
#endif
}

/*
 * Backward: given dO [B,S,nh,hd], writes dq [B,S,nh,hd], dk and dv [B,S,nkv,hd].
 * The forward (O and LSE) is recomputed here from the definition.
 */
void xo_bwd(const double *q, const double *k, const double *v, const double *dO, int B, int S,
            int nh, int nkv, int hd, double scale, double *dq, double *dk, double *dv) {
    int group = nh / nkv;
    size_t n_q = (size_t)B * S * nh * hd;
    double *o = (double *)malloc(n_q * sizeof(double));
    double *lse = (double *)malloc((size_t)B * S * nh * sizeof(double));
    double *D = (double *)malloc((size_t)B * S * nh * sizeof(double));
    xo_fwd(q, k, v, B, S, nh, nkv, hd, scale, o, lse);

    long total_rows = (long)B * nh * S;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < total_rows; ++t) {
        int i = (int)(t % S);
        int h = (int)((t / S) % nh);
        int b = (int)(t / ((long)S * nh));
        D[((size_t)b * S + i) * nh + h] = row_D(dO, o, b, i, h, S, nh, hd);
    }

    /* dQ: one query row at a time. */
#pragma omp parallel for schedule(dynamic, 8)
    for (long t = 0; t < total_rows; ++t) {
        int i = (int)(t % S);
        int h = (int)((t / S) % nh);
        int b = (int)(t / ((long)S * nh));
        int kvh = kv_head_of(h, nh, nkv);
        double L = lse[((size_t)b * S + i) * nh + h];
        double Di = D[((size_t)b * S + i) * nh + h];
        const double *dOi = &dO[IDX4(b, i, h, 0, S, nh, hd)];
        double *dqi = &dq[IDX4(b, i, h, 0, S, nh, hd)];
        for (int d = 0; d < hd; ++d) dqi[d] = 0.0;
        for (int j = 0; j < S; ++j) {
            if (!visible(i, j)) continue;
            double p = exp(score(q, k, b, i, j, h, kvh, S, nh, nkv, hd, scale) - L);
            double dp = dot(dOi, &v[IDX4(b, j, kvh, 0, S, nkv, hd)], hd);
            double ds = p * (dp - Di);
#if ORACLE_MUTATION == 7
            const double *kj = &k[IDX4(b, i, kvh, 0, S, nkv, hd)];   /* planted: row index for column */
#else
            const double *kj = &k[IDX4(b, j, kvh, 0, S, nkv, hd)];
#endif
            for (int d = 0; d < hd; ++d) dqi[d] += scale * ds * kj[d];
        }
    }

    /* dK, dV: one key row of one kv head at a time, summing its query group in order r = 0.. */
    long total_cols = (long)B * nkv * S;
#pragma omp parallel for schedule(dynamic, 8)
    for (long t = 0; t < total_cols; ++t) {
        int j = (int)(t % S);
        int kvh = (int)((t / S) % nkv);
        int b = (int)(t / ((long)S * nkv));
        double *dkj = &dk[IDX4(b, j, kvh, 0, S, nkv, hd)];
        double *dvj = &dv[IDX4(b, j, kvh, 0, S, nkv, hd)];
        for (int d = 0; d < hd; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
        for (int h = 0; h < nh; ++h) {
            if (kv_head_of(h, nh, nkv) != kvh) continue;
#if ORACLE_MUTATION == 5
            if (h % group != group - 1) continue;   /* planted: only one head of the group */
#else
            (void)group;
#endif
            for (int i = 0; i < S; ++i) {
                if (!visible(i, j)) continue;
                double L = lse[((size_t)b * S + i) * nh + h];
                double Di = D[((size_t)b * S + i) * nh + h];
                const double *dOi = &dO[IDX4(b, i, h, 0, S, nh, hd)];
                const double *qi = &q[IDX4(b, i, h, 0, S, nh, hd)];
                double p = exp(score(q, k, b, i, j, h, kvh, S, nh, nkv, hd, scale) - L);
                double dp = dot(dOi, &v[IDX4(b, j, kvh, 0, S, nkv, hd)], hd);
                double ds = p * (dp - Di);
#if ORACLE_MUTATION == 3
                double sk = 1.0;          /* planted: scale missing from dK */
#else
                double sk = scale;
#endif
                for (int d = 0; d < hd; ++d) {
                    dkj[d] += sk * ds * qi[d];
                    dvj[d] += p * dOi[d];
                }
            }
        }
    }
    free(o);
    free(lse);
    free(D);
}

/* Build identification for the test suite (which mutation, if any, was compiled in). */
/*
 * Decode: q [B,nh,hd], k/v [B,T,nkv,hd] -> o [B,nh,hd], lse [B,nh].
 */
void xo_decode(const double *q, const double *k, const double *v, int B, int T, int nh, int nkv,
               int hd, double scale, double *o, double *lse) {
#if ORACLE_MUTATION == 10
    const int n_keys = T - 1;     /* planted: the newest cached key left out */
#else
    const int n_keys = T;
#endif
    long total = (long)B * nh;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < total; ++t) {
        int h = (int)(t % nh);
        int b = (int)(t / nh);
        int kvh = kv_head_of(h, nh, nkv);
        const double *qh = &q[((size_t)b * nh + h) * hd];
        double mx = -INFINITY;
        for (int j = 0; j < n_keys; ++j) {
            double s = scale * dot(qh, &k[IDX4(b, j, kvh, 0, T, nkv, hd)], hd);
            if (s > mx) mx = s;
        }
        double sum = 0.0;
        for (int j = 0; j < n_keys; ++j)
            sum += exp(scale * dot(qh, &k[IDX4(b, j, kvh, 0, T, nkv, hd)], hd) - mx);
        double L = mx + log(sum);
        lse[(size_t)b * nh + h] = L;
        double *oh = &o[((size_t)b * nh + h) * hd];
        for (int d = 0; d < hd; ++d) oh[d] = 0.0;
        for (int j = 0; j < n_keys; ++j) {
            double p = exp(scale * dot(qh, &k[IDX4(b, j, kvh, 0, T, nkv, hd)], hd) - L);
            const double *vj = &v[IDX4(b, j, kvh, 0, T, nkv, hd)];
            for (int d = 0; d < hd; ++d) oh[d] += p * vj[d];
        }
    }
}

int xo_mutation(void) { return ORACLE_MUTATION; }
