/*
 * dspark_oracle.c -- plain, slow, single-threaded CPU oracle (fp64).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no code
 * with the CUDA library.  Every function follows one passage of the pages,
 * cited in its comment, in the pages' order and notation:
 *   [D] "DSpark: confidence-scheduled speculative decoding" (ai-papers-daily digest)
 *   [E] "DSpark explained" (interactive explainer)
 * Pins: tests/test_oracle_*.py.
 */
#include "dspark_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element access: bf16 is the top half of an IEEE binary32                 */
/* ------------------------------------------------------------------------ */
static double load_elem(const void *base, size_t i, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Philox-4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64      */
/* multiplies with the published multipliers and Weyl key increments.      */
/* ------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* u = ((w >> 9) + 1/2) 2^-23: 2^23 equally spaced points inside (0, 1). */
double oracle_uniform(uint32_t word) {
    return ((double)(word >> 9) + 0.5) * (1.0 / 8388608.0);
}

uint32_t oracle_philox_word(uint64_t seed, uint32_t w0, uint32_t w1, uint32_t req,
                            uint64_t cycle, uint32_t stream, uint32_t lane) {
    uint32_t ctr[4] = {w0, w1, req, (uint32_t)((cycle << 2) | (uint64_t)stream)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[lane];
}

/* ------------------------------------------------------------------------ */
/* [D] eq. (4): p_k(v) = exp(U_k(v) + B_k(v)) / sum_u exp(U_k(u) + B_k(u)).  */
/* The pages fix the distribution, not how it is sampled; x_k is drawn in   */
/* two levels, which together pick v with probability exactly p_k(v):       */
/*   blocks: the vocabulary in blocks of DRAFT_BLOCK consecutive entries    */
/*     (the last one may be shorter); block b has mass                      */
/*     S_b = sum_{v in b} exp(z_v - m) for a fixed m (here the max of z);   */
/*   level 1: the block by the Gumbel-max rule over the blocks' masses,     */
/*     b* = argmax_b ln S_b + g_b, g_b = -log(-log u_b), ties to the lowest */
/*     b -- block b wins with probability S_b / sum_b S_b;                  */
/*   level 2: the entry of b* by inverse CDF: the first v of the block whose */
/*     running sum of exp(z - m), in index order from the block's start,    */
/*     exceeds u'_{b*} S_{b*} -- v with probability exp(z_v - m) / S_{b*}.  */
/* Random words (stream 0): block b uses the Philox counter                 */
/* (floor(b / 2), k, request, cycle << 2 | 0), word 2 (b mod 2) for u_b and */
/* word 2 (b mod 2) + 1 for u'_b.                                           */
/* ------------------------------------------------------------------------ */
#define DRAFT_BLOCK 16

static void block_words(uint64_t seed, uint32_t step, uint32_t req, uint64_t cycle, int b,
                        double *u_race, double *u_entry) {
    uint32_t ctr[4] = {(uint32_t)(b / 2), step, req, (uint32_t)(cycle << 2)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    *u_race = oracle_uniform(out[2 * (b % 2)]);
    *u_entry = oracle_uniform(out[2 * (b % 2) + 1]);
}

/* Level 2 inside block b: the entry; optionally the target's distances to  */
/* the lower and upper ends of that entry's interval (fractions of S_b) and */
/* the entries of the block across them (-1: none).                         */
static int block_entry(const double *z, int V, double m, int b, double u_entry,
                       double margin[2], int across[2]) {
    int v0 = b * DRAFT_BLOCK, v1 = v0 + DRAFT_BLOCK < V ? v0 + DRAFT_BLOCK : V;
    double S = 0.0;
    for (int v = v0; v < v1; ++v) S += exp(z[v] - m);
    double target = u_entry * S, cum = 0.0;
    int pick = -1;
    double lo = 0.0, hi = 0.0;
    for (int v = v0; v < v1; ++v) {
        double e = exp(z[v] - m);
        if (cum + e > target) {
            pick = v;
            lo = target - cum;
            hi = cum + e - target;
            break;
        }
        cum += e;
    }
    if (pick < 0) { /* rounding put the target at the total: the last entry of positive mass */
        for (int v = v1 - 1; v >= v0 && pick < 0; --v)
            if (exp(z[v] - m) > 0.0) pick = v;
    }
    if (margin) {
        margin[0] = lo / S;
        margin[1] = hi / S;
    }
    if (across) {
        across[0] = pick - 1 >= v0 ? pick - 1 : -1;
        across[1] = pick + 1 < v1 && exp(z[pick + 1] - m) > 0.0 ? pick + 1 : -1;
    }
    return pick;
}

/* Writes lse, the sampled index x, log q of it and the near-tie records:  */
/* gap / runner -- the difference between the two best block scores and    */
/* the token the runner-up block gives at level 2; cdf_gap[2] /             */
/* cdf_runner[2] -- the level-2 target's distances to the lower and upper   */
/* ends of x's interval (fractions of S_{b*}) and the entries across them.  */
static void sample_step(const double *z, int V, uint64_t seed, uint32_t step, uint32_t req,
                        uint64_t cycle, int32_t *x_out, double *logq_out, double *lse_out,
                        double *gap_out, int32_t *runner_out, double *cdf_gap_out,
                        int32_t *cdf_runner_out) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (z[v] > m) m = z[v];
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += exp(z[v] - m);
    double lse = m + log(S);

    int nb = (V + DRAFT_BLOCK - 1) / DRAFT_BLOCK;
    double best = -INFINITY, second = -INFINITY;
    int arg = -1, arg2 = -1;
    double u_race, u_entry;
    for (int b = 0; b < nb; ++b) {
        int v0 = b * DRAFT_BLOCK, v1 = v0 + DRAFT_BLOCK < V ? v0 + DRAFT_BLOCK : V;
        double Sb = 0.0;
        for (int v = v0; v < v1; ++v) Sb += exp(z[v] - m);
        if (!(Sb > 0.0)) continue;
        block_words(seed, step, req, cycle, b, &u_race, &u_entry);
        double score = log(Sb) - log(-log(u_race));
        if (score > best) {
            second = best;
            arg2 = arg;
            best = score;
            arg = b;
        } else if (score > second) {
            second = score;
            arg2 = b;
        }
    }
    double margin[2];
    int across[2];
    block_words(seed, step, req, cycle, arg, &u_race, &u_entry);
    int v = block_entry(z, V, m, arg, u_entry, margin, across);
    *x_out = v;
    *logq_out = z[v] - lse;
    *lse_out = lse;
    if (gap_out) *gap_out = best - second;
    if (runner_out) {
        int other = -1;
        if (arg2 >= 0) {
            block_words(seed, step, req, cycle, arg2, &u_race, &u_entry);
            other = block_entry(z, V, m, arg2, u_entry, NULL, NULL);
        }
        *runner_out = other;
    }
    if (cdf_gap_out) {
        cdf_gap_out[0] = margin[0];
        cdf_gap_out[1] = margin[1];
    }
    if (cdf_runner_out) {
        cdf_runner_out[0] = across[0];
        cdf_runner_out[1] = across[1];
    }
}

/* [D] eq. (7): c_k = sigma(w^T [h_k ; W_1[x_{k-1}]]); the optional per-step
 * temperature T_k is the sequential temperature scaling of Module D applied
 * to the logit (T_k = 1 when not given). */
static double confidence(const float *w, const void *h_k, int d, const double *e, int r,
                         int dtype, double T_k, double *logit) {
    double dot = 0.0;
    for (int j = 0; j < d; ++j) dot += (double)w[j] * load_elem(h_k, (size_t)j, dtype);
    for (int i = 0; i < r; ++i) dot += (double)w[d + i] * e[i];
    if (logit) *logit = dot;
    return 1.0 / (1.0 + exp(-dot / T_k));
}

/* ------------------------------------------------------------------------ */
/* Markov head: [D] eq. (5) B(x_{k-1}, .) = W_1[x_{k-1}] W_2, used in eq. (4) */
/* for k = 1..gamma with x_0 the anchor; confidence by eq. (7).             */
/* ------------------------------------------------------------------------ */
int oracle_draft_markov(int R, int gamma, int V, int r, int d, int dtype,
                        const void *U, const void *h, const void *W1, const void *W2t,
                        const float *w, const float *sts_T, const int32_t *anchor,
                        uint64_t seed, uint64_t cycle, const int32_t *reqs, int n_reqs,
                        int32_t *x, double *logq, double *lse, double *c, double *gap,
                        int32_t *runner, double *cdf_gap, int32_t *cdf_runner, double *z_out,
                        double *logit) {
    int n = reqs ? n_reqs : R;
    double *e = (double *)malloc(sizeof(double) * (size_t)r);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    if (!e || !z) { free(e); free(z); return -1; }
    int status = 0;
    for (int t = 0; t < n && status == 0; ++t) {
        int rq = reqs ? reqs[t] : t;
        if (rq < 0 || rq >= R || anchor[rq] < 0 || anchor[rq] >= V) { status = -1; break; }
        int32_t x_prev = anchor[rq];
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)t * gamma + (size_t)(k - 1);
            /* E_k = W_1[x_{k-1}] */
            for (int i = 0; i < r; ++i) e[i] = load_elem(W1, (size_t)x_prev * r + i, dtype);
            /* z = U_k + E_k W_2 */
            size_t urow = ((size_t)rq * gamma + (size_t)(k - 1)) * (size_t)V;
            for (int v = 0; v < V; ++v) {
                double b = 0.0;
                for (int i = 0; i < r; ++i) b += e[i] * load_elem(W2t, (size_t)v * r + i, dtype);
                z[v] = load_elem(U, urow + (size_t)v, dtype) + b;
            }
            if (z_out) memcpy(z_out + o * (size_t)V, z, sizeof(double) * (size_t)V);
            sample_step(z, V, seed, (uint32_t)k, (uint32_t)rq, cycle, &x[o], &logq[o], &lse[o],
                        gap ? &gap[o] : NULL, runner ? &runner[o] : NULL,
                        cdf_gap ? &cdf_gap[2 * o] : NULL, cdf_runner ? &cdf_runner[2 * o] : NULL);
            const void *h_k = dtype == ORACLE_F32
                                  ? (const void *)((const float *)h + ((size_t)rq * gamma + (k - 1)) * (size_t)d)
                                  : (const void *)((const uint16_t *)h + ((size_t)rq * gamma + (k - 1)) * (size_t)d);
            c[o] = confidence(w, h_k, d, e, r, dtype, sts_T ? (double)sts_T[k - 1] : 1.0,
                              logit ? &logit[o] : NULL);
            x_prev = x[o];
        }
    }
    free(e);
    free(z);
    return status;
}

static double sigmoid(double t) { return 1.0 / (1.0 + exp(-t)); }

/* ------------------------------------------------------------------------ */
/* RNN head, [D] eq. (6):                                                    */
/*   z_k = [s_{k-1}; W_1[x_{k-1}]; h_k]                                      */
/*   s_k = sigma(W_g z_k) * s_{k-1} + (1 - sigma(W_g z_k)) * tanh(W_c z_k)   */
/*   B_k = W_2^T tanh(W_o z_k),  s_0 = 0                                     */
/* with W_g, W_c, W_o the three row blocks of one projection W [3r, 2r+d].   */
/* ------------------------------------------------------------------------ */
int oracle_draft_rnn(int R, int gamma, int V, int r, int d, int dtype,
                     const void *U, const void *h, const void *W1, const void *W2t,
                     const void *W, const float *s0, const float *w, const float *sts_T,
                     const int32_t *anchor, uint64_t seed, uint64_t cycle,
                     const int32_t *reqs, int n_reqs, int32_t *x, double *logq,
                     double *lse, double *c, double *gap, int32_t *runner, double *cdf_gap,
                     int32_t *cdf_runner, double *z_out, double *A_out, double *logit) {
    int n = reqs ? n_reqs : R;
    int zlen = 2 * r + d;
    double *s = (double *)malloc(sizeof(double) * (size_t)r);
    double *s_next = (double *)malloc(sizeof(double) * (size_t)r);
    double *zk = (double *)malloc(sizeof(double) * (size_t)zlen);
    double *G = (double *)malloc(sizeof(double) * (size_t)(3 * r));
    double *A = (double *)malloc(sizeof(double) * (size_t)r);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    int status = (s && s_next && zk && G && A && z) ? 0 : -1;
    for (int t = 0; t < n && status == 0; ++t) {
        int rq = reqs ? reqs[t] : t;
        if (rq < 0 || rq >= R || anchor[rq] < 0 || anchor[rq] >= V) { status = -1; break; }
        for (int i = 0; i < r; ++i) s[i] = s0 ? (double)s0[(size_t)rq * r + i] : 0.0;
        int32_t x_prev = anchor[rq];
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)t * gamma + (size_t)(k - 1);
            /* z_k = [s_{k-1}; W_1[x_{k-1}]; h_k] */
            for (int i = 0; i < r; ++i) zk[i] = s[i];
            for (int i = 0; i < r; ++i) zk[r + i] = load_elem(W1, (size_t)x_prev * r + i, dtype);
            size_t hrow = ((size_t)rq * gamma + (size_t)(k - 1)) * (size_t)d;
            for (int j = 0; j < d; ++j) zk[2 * r + j] = load_elem(h, hrow + (size_t)j, dtype);
            /* G = W z_k */
            for (int oi = 0; oi < 3 * r; ++oi) {
                double acc = 0.0;
                for (int j = 0; j < zlen; ++j)
                    acc += load_elem(W, (size_t)oi * zlen + (size_t)j, dtype) * zk[j];
                G[oi] = acc;
            }
            for (int i = 0; i < r; ++i) {
                double gate = sigmoid(G[i]);
                double cand = tanh(G[r + i]);
                A[i] = tanh(G[2 * r + i]);
                s_next[i] = gate * s[i] + (1.0 - gate) * cand;
            }
            if (A_out) memcpy(A_out + o * (size_t)r, A, sizeof(double) * (size_t)r);
            /* z = U_k + W_2^T A_k */
            size_t urow = ((size_t)rq * gamma + (size_t)(k - 1)) * (size_t)V;
            for (int v = 0; v < V; ++v) {
                double b = 0.0;
                for (int i = 0; i < r; ++i) b += A[i] * load_elem(W2t, (size_t)v * r + i, dtype);
                z[v] = load_elem(U, urow + (size_t)v, dtype) + b;
            }
            if (z_out) memcpy(z_out + o * (size_t)V, z, sizeof(double) * (size_t)V);
            sample_step(z, V, seed, (uint32_t)k, (uint32_t)rq, cycle, &x[o], &logq[o], &lse[o],
                        gap ? &gap[o] : NULL, runner ? &runner[o] : NULL,
                        cdf_gap ? &cdf_gap[2 * o] : NULL, cdf_runner ? &cdf_runner[2 * o] : NULL);
            /* eq. (7) reads the embedding W_1[x_{k-1}], i.e. the middle block of z_k */
            const void *h_k = dtype == ORACLE_F32 ? (const void *)((const float *)h + hrow)
                                                  : (const void *)((const uint16_t *)h + hrow);
            c[o] = confidence(w, h_k, d, zk + r, r, dtype, sts_T ? (double)sts_T[k - 1] : 1.0,
                              logit ? &logit[o] : NULL);
            memcpy(s, s_next, sizeof(double) * (size_t)r);
            x_prev = x[o];
        }
    }
    free(s); free(s_next); free(zk); free(G); free(A); free(z);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Hardware-aware prefix scheduler, [D] Module E and Algorithm 1.           */
/*   a_{r,j} = prod_{i<=j} c_{r,i}; E = {(r,j): a_{r,j} > 0} sorted by a desc */
/*   B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a_{r,j}),            */
/*   Theta = tau * SPS(B).                                                   */
/* Number formats (the pages fix none): a as an fp32 running product in j    */
/* order; tau as an integer count of 2^-32 units, each a rounded to nearest  */
/* (ties to even) on that grid, so every summation order gives the same tau; */
/* Theta = (tau_units * 2^-32) * SPS(B) in fp64.                             */
/* ------------------------------------------------------------------------ */
typedef struct {
    float a;
    int32_t flat; /* r * gamma + (j - 1) */
} pool_entry;

/* descending a, then ascending flat index (request, then position) */
static int pool_cmp(const void *pa, const void *pb) {
    const pool_entry *x = (const pool_entry *)pa, *y = (const pool_entry *)pb;
    if (x->a > y->a) return -1;
    if (x->a < y->a) return 1;
    return (x->flat > y->flat) - (x->flat < y->flat);
}

static double theta_of(int64_t tau_units, const double *sps, int B_min, int B) {
    double tau = (double)tau_units * (1.0 / 4294967296.0);
    return tau * sps[B - B_min];
}

int oracle_schedule(int R, int gamma, const float *c, const double *sps, int B_min,
                    int B_count, int mode, int K_in, int32_t *ell, int32_t *K_out,
                    double *theta_best_out, float *a_out) {
    if (R < 1 || gamma < 1) return -1;
    if (B_min > R || (int64_t)R * (gamma + 1) > (int64_t)B_min + B_count - 1) return -1;
    size_t n = (size_t)R * gamma;
    for (size_t i = 0; i < n; ++i)
        if (!(c[i] >= 0.0f && c[i] <= 1.0f)) return -2;

    /* Algorithm 1, line 1: prefix survival probabilities */
    float *a = (float *)malloc(sizeof(float) * n);
    pool_entry *pool = (pool_entry *)malloc(sizeof(pool_entry) * n);
    int64_t *units = (int64_t *)malloc(sizeof(int64_t) * (n + 1));
    int32_t *ell_cur = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    if (!a || !pool || !units || !ell_cur) {
        free(a); free(pool); free(units); free(ell_cur);
        return -1;
    }
    for (int rq = 0; rq < R; ++rq) {
        float prod = 1.0f;
        for (int j = 0; j < gamma; ++j) {
            prod = prod * c[(size_t)rq * gamma + j];
            a[(size_t)rq * gamma + j] = prod;
        }
    }
    if (a_out) memcpy(a_out, a, sizeof(float) * n);

    /* line 2: candidate pool, sorted by a descending */
    size_t m = 0;
    for (size_t i = 0; i < n; ++i)
        if (a[i] > 0.0f) {
            pool[m].a = a[i];
            pool[m].flat = (int32_t)i;
            ++m;
        }
    qsort(pool, m, sizeof(pool_entry), pool_cmp);

    /* tau after admitting the first t entries, in 2^-32 units */
    units[0] = (int64_t)R << 32;
    for (size_t t = 0; t < m; ++t)
        units[t + 1] = units[t] + (int64_t)llrintf(pool[t].a * 4294967296.0f);

    /* capacity for the asynchronous variant: best count without the break */
    int32_t K_best = 0;
    double theta_K = theta_of(units[0], sps, B_min, R);
    for (size_t t = 1; t <= m; ++t) {
        double th = theta_of(units[t], sps, B_min, R + (int)t);
        if (th > theta_K) { theta_K = th; K_best = (int32_t)t; }
    }
    *K_out = K_best;

    for (int rq = 0; rq < R; ++rq) ell[rq] = 0;
    if (mode == ORACLE_SCHED_SYNC || (mode == ORACLE_SCHED_ASYNC && K_in < 0)) {
        /* lines 3-9 */
        for (int rq = 0; rq < R; ++rq) ell_cur[rq] = 0;
        int B = R;
        int64_t tau = units[0];
        double theta_best = theta_of(tau, sps, B_min, B);
        for (size_t t = 0; t < m; ++t) {
            int rq = pool[t].flat / gamma, j = pool[t].flat % gamma + 1;
            ell_cur[rq] = j;                                           /* line 5 */
            B += 1;
            tau += (int64_t)llrintf(pool[t].a * 4294967296.0f);
            double theta = theta_of(tau, sps, B_min, B);              /* line 6 */
            if (theta > theta_best) {                                  /* line 7 */
                theta_best = theta;
                memcpy(ell, ell_cur, sizeof(int32_t) * (size_t)R);
            } else {
                break;                                                 /* line 8 */
            }
        }
        *theta_best_out = theta_best;
    } else {
        /* production variant: top-K of the current order, no break; the
         * test-only backtracking mode takes K from the current pool itself */
        size_t count = mode == ORACLE_SCHED_NOBREAK ? (size_t)K_best
                                                    : ((size_t)K_in < m ? (size_t)K_in : m);
        for (size_t t = 0; t < count; ++t) {
            int rq = pool[t].flat / gamma, j = pool[t].flat % gamma + 1;
            ell[rq] = j;
        }
        *theta_best_out = theta_of(units[count], sps, B_min, R + (int)count);
    }
    free(a); free(pool); free(units); free(ell_cur);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Verification: [E] section 06 single-token rule, applied along the        */
/* prefix ([D] overview step 3): accept x_{j+1} with probability            */
/* min(1, p_j(x)/q_{j+1}(x)); at the first rejection sample from            */
/* norm(max(0, p_j - q_{j+1})); if all scheduled tokens pass, sample the     */
/* bonus token from p_{l_r}.  Row (r, j) of T holds the target logits for   */
/* x_{j+1} given x_0..x_j.  The pages fix no sampler for the correction;    */
/* it is drawn by inverse CDF with one uniform (any exact draw from the      */
/* normalised residual keeps the method lossless).                           */
/* ------------------------------------------------------------------------ */
static double row_logsumexp(const void *T, size_t row, int V, int dtype) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double t = load_elem(T, row * (size_t)V + v, dtype);
        if (t > m) m = t;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += exp(load_elem(T, row * (size_t)V + v, dtype) - m);
    return m + log(S);
}

int oracle_verify(int R, int gamma, int V, int r, int dtype, int N, const void *T,
                  const int32_t *tags, const int32_t *anchor, const int32_t *x,
                  const float *logq, const float *lse, const void *U, const void *W1,
                  const void *W2t, const float *A, uint64_t seed, uint64_t cycle,
                  const int32_t *reqs, int n_reqs, int32_t *n_accept, int32_t *out_tokens,
                  int32_t *next_anchor, double *lse_p, double *logp, double *margin,
                  double *gap, int32_t *runner) {
    /* rows of each request: first row index and count */
    int32_t *first = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *count = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *b = (double *)malloc(sizeof(double) * (size_t)r);
    if (!first || !count || !w || !b) {
        free(first); free(count); free(w); free(b);
        return -1;
    }
    int status = 0;
    for (int rq = 0; rq < R; ++rq) { first[rq] = -1; count[rq] = 0; }
    for (int i = 0; i < N && status == 0; ++i) {
        int rq = tags[2 * i], pos = tags[2 * i + 1];
        if (rq < 0 || rq >= R || pos < 0 || pos > gamma) { status = -1; break; }
        if (pos == 0) {
            if (first[rq] != -1) { status = -1; break; }
            first[rq] = i;
        } else if (i == 0 || tags[2 * (i - 1)] != rq || tags[2 * (i - 1) + 1] != pos - 1) {
            status = -1;
            break;
        }
        count[rq] += 1;
    }
    for (int rq = 0; rq < R && status == 0; ++rq)
        if (first[rq] < 0) status = -1;

    int n = reqs ? n_reqs : R;
    for (int t = 0; t < n && status == 0; ++t) {
        int rq = reqs ? reqs[t] : t;
        if (rq < 0 || rq >= R) { status = -1; break; }
        int ell = count[rq] - 1;
        int n_r = -1;
        /* phase 1: every scheduled row */
        for (int j = 0; j <= ell; ++j) {
            size_t row = (size_t)first[rq] + (size_t)j;
            double lp = row_logsumexp(T, row, V, dtype);
            if (lse_p) lse_p[row] = lp;
            if (j < ell) {
                int32_t tok = x[(size_t)rq * gamma + j];
                if (tok < 0 || tok >= V) { status = -1; break; }
                double log_p = load_elem(T, row * (size_t)V + (size_t)tok, dtype) - lp;
                double log_q = (double)logq[(size_t)rq * gamma + j];
                double u = oracle_uniform(oracle_philox_word(seed, 0, (uint32_t)j, (uint32_t)rq,
                                                             cycle, 1, 0));
                double mg = (log_p - log_q) - log(u);
                if (logp) logp[row] = log_p;
                if (margin) margin[row] = mg;
                int accept = log(u) < log_p - log_q;
                if (!accept && n_r < 0) n_r = j;
            } else {
                if (logp) logp[row] = NAN;
                if (margin) margin[row] = NAN;
            }
        }
        if (status) break;
        if (n_r < 0) n_r = ell;

        /* phase 2: residual at the first rejection, else the bonus token */
        size_t row = (size_t)first[rq] + (size_t)n_r;
        double lp = row_logsumexp(T, row, V, dtype);
        for (int v = 0; v < V; ++v) w[v] = exp(load_elem(T, row * (size_t)V + v, dtype) - lp);
        if (n_r < ell) {
            if (A) {
                for (int i = 0; i < r; ++i) b[i] = (double)A[((size_t)rq * gamma + n_r) * (size_t)r + i];
            } else {
                int32_t xn = n_r == 0 ? anchor[rq] : x[(size_t)rq * gamma + (n_r - 1)];
                for (int i = 0; i < r; ++i) b[i] = load_elem(W1, (size_t)xn * r + i, dtype);
            }
            double lq = (double)lse[(size_t)rq * gamma + n_r];
            size_t urow = ((size_t)rq * gamma + (size_t)n_r) * (size_t)V;
            int any = 0;
            for (int v = 0; v < V; ++v) {
                double bias = 0.0;
                for (int i = 0; i < r; ++i) bias += b[i] * load_elem(W2t, (size_t)v * r + i, dtype);
                double q = exp(load_elem(U, urow + v, dtype) + bias - lq);
                double res = w[v] - q;
                w[v] = res > 0.0 ? res : 0.0;
                any |= w[v] > 0.0;
            }
            if (!any) /* degenerate p == q: fall back to p itself */
                for (int v = 0; v < V; ++v) w[v] = exp(load_elem(T, row * (size_t)V + v, dtype) - lp);
        }
        /* inverse-CDF draw from norm(w): one uniform u (stream 2, counter
         * (0, n_r, request, cycle), word 0), the target u * sum(w), and the first
         * v whose cumulative weight exceeds it */
        double total = 0.0;
        for (int v = 0; v < V; ++v) total += w[v];
        double u2 = oracle_uniform(oracle_philox_word(seed, 0, (uint32_t)n_r, (uint32_t)rq, cycle, 2, 0));
        double target = u2 * total;
        double cum = 0.0, below = 0.0;
        int y = -1;
        for (int v = 0; v < V; ++v) {
            if (!(w[v] > 0.0)) continue;
            below = cum;
            cum += w[v];
            y = v; /* the last positive-weight index, if the target is never passed */
            if (cum > target) break;
        }
        /* the distances of the target to the two ends of y's interval, relative
         * to the total, and the positive-weight indices across them (the draws a
         * slightly lower or higher target would give) */
        int y_lo = -1, y_hi = -1;
        double d_lo = INFINITY, d_hi = INFINITY;
        if (y >= 0 && total > 0.0) {
            d_lo = (target - below) / total;
            d_hi = (cum - target) / total;
            for (int v = y - 1; v >= 0 && y_lo < 0; --v)
                if (w[v] > 0.0) y_lo = v;
            for (int v = y + 1; v < V && y_hi < 0; ++v)
                if (w[v] > 0.0) y_hi = v;
        }
        n_accept[rq] = n_r;
        for (int j = 0; j <= gamma; ++j) {
            int32_t tok = -1;
            if (j < n_r) tok = x[(size_t)rq * gamma + j];
            else if (j == n_r) tok = y;
            out_tokens[(size_t)rq * (gamma + 1) + j] = tok;
        }
        next_anchor[rq] = y;
        if (gap) {
            gap[2 * (size_t)rq] = d_lo;
            gap[2 * (size_t)rq + 1] = d_hi;
        }
        if (runner) {
            runner[2 * (size_t)rq] = y_lo;
            runner[2 * (size_t)rq + 1] = y_hi;
        }
    }
    free(first); free(count); free(w); free(b);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Sequential temperature scaling, [D] Module D.                             */
/* c_i is the probability that position i is accepted given that every      */
/* earlier position was, so by the chain rule the probability that the      */
/* first k drafted tokens are all accepted is P_k = prod_{i<=k} c_i with     */
/* c_i = sigma(s_i / T_i).  Left to right, T_k is the grid point whose       */
/* P_k has the smallest expected calibration error against the held-out     */
/* outcome y_k = 1[n >= k] (n = accepted prefix length of the sample), with  */
/* T_1..T_{k-1} held at the values already chosen.                          */
/* ECE (the pages fix no binning; the usual equal-width reading): n_bins     */
/* bins of [0, 1], bin(P) = min(floor(P n_bins), n_bins - 1), and           */
/*   ECE = sum_b (|b| / M) |mean_b P - mean_b y| = (1/M) sum_b |sum_b (P - y)|. */
/* Ties between grid points go to the lowest index.                         */
/* ------------------------------------------------------------------------ */
int oracle_sts_fit(int M, int gamma, const float *logit, const int32_t *n_accept, int G,
                   const float *grid, int n_bins, const float *T_prefix, float *T_out,
                   double *ece_out, double *curve, double edge_eps, int32_t *near_edge) {
    if (M < 1 || gamma < 1 || G < 1 || n_bins < 1) return -1;
    for (int g = 0; g < G; ++g)
        if (!(grid[g] > 0.0f) || !isfinite(grid[g])) return -1;
    for (int m = 0; m < M; ++m) {
        if (n_accept[m] < 0 || n_accept[m] > gamma) return -1;
        for (int k = 0; k < gamma; ++k)
            if (isnan(logit[(size_t)m * gamma + k])) return -1;
    }
    double *prefix = (double *)malloc(sizeof(double) * (size_t)M);   /* P_{k-1} per sample */
    double *bin_sum = (double *)malloc(sizeof(double) * (size_t)n_bins);
    if (!prefix || !bin_sum) { free(prefix); free(bin_sum); return -1; }
    for (int m = 0; m < M; ++m) prefix[m] = 1.0;
    if (near_edge) memset(near_edge, 0, sizeof(int32_t) * (size_t)gamma * (size_t)G);
    for (int k = 1; k <= gamma; ++k) {
        int best = 0;
        double best_ece = 0.0;
        for (int g = 0; g < G; ++g) {
            double T = (double)grid[g];
            for (int b = 0; b < n_bins; ++b) bin_sum[b] = 0.0;
            for (int m = 0; m < M; ++m) {
                double s = (double)logit[(size_t)m * gamma + (k - 1)];
                double P = prefix[m] * (1.0 / (1.0 + exp(-s / T)));
                int b = (int)floor(P * n_bins);
                if (b > n_bins - 1) b = n_bins - 1;
                double y = n_accept[m] >= k ? 1.0 : 0.0;
                bin_sum[b] += P - y;
                if (near_edge) {
                    /* samples within edge_eps of an interior bin edge j / n_bins */
                    int j = (int)floor(P * n_bins + 0.5);
                    if (j >= 1 && j <= n_bins - 1 && fabs(P - (double)j / n_bins) < edge_eps)
                        ++near_edge[(size_t)(k - 1) * G + g];
                }
            }
            double ece = 0.0;
            for (int b = 0; b < n_bins; ++b) ece += fabs(bin_sum[b]);
            ece /= (double)M;
            if (curve) curve[(size_t)(k - 1) * G + g] = ece;
            if (g == 0 || ece < best_ece) { best = g; best_ece = ece; }
        }
        T_out[k - 1] = grid[best];
        ece_out[k - 1] = best_ece;
        /* hold T_k for the later positions (a caller may impose its own) */
        double T_k = T_prefix ? (double)T_prefix[k - 1] : (double)grid[best];
        for (int m = 0; m < M; ++m) {
            double s = (double)logit[(size_t)m * gamma + (k - 1)];
            prefix[m] *= 1.0 / (1.0 + exp(-s / T_k));
        }
    }
    free(prefix);
    free(bin_sum);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [D] analysis 1: per-position conditional acceptance, counted over the     */
/* instances whose first k - 1 positions were accepted; the acceptance       */
/* length tau = n + 1 (the target's own token included).                      */
/* ------------------------------------------------------------------------ */
int oracle_accept_stats(int R, int gamma, const int32_t *n_accept, const int32_t *ell, uint64_t *reached,
                        uint64_t *accepted, uint64_t *tau_hist, uint64_t *ell_hist) {
    for (int r = 0; r < R; ++r) {
        const int l = ell ? ell[r] : gamma;
        if (l < 0) continue;
        const int n = n_accept[r];
        if (n < 0 || n > l || n > gamma || l > gamma) return -1;
    }
    for (int r = 0; r < R; ++r) {
        const int l = ell ? ell[r] : gamma;
        if (l < 0) continue;
        const int n = n_accept[r];
        for (int k = 1; k <= gamma; ++k) {
            if (l >= k && n >= k - 1) reached[k - 1] += 1; /* position k was tested */
            if (n >= k) accepted[k - 1] += 1;              /* and passed            */
        }
        tau_hist[n] += 1;
        if (ell_hist) ell_hist[l] += 1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [D] Module F, eqs. (8)-(12): position-weighted cross-entropy, total        */
/* variation and confidence BCE; the gradient with respect to the draft     */
/* logits for the first two (the label c* of the third held fixed).          */
/* ------------------------------------------------------------------------ */
static double softplus(double t) { return t > 0.0 ? t + log1p(exp(-t)) : log1p(exp(t)); }

int oracle_train_losses(int B, int gamma, int V, int dtype, const void *zd, const void *zt,
                        const int32_t *xs, const float *s, double a_ce, double a_tv, double a_conf,
                        double *row, double *loss, double *grad_z, double *grad_s) {
    const int N = B * gamma;
    for (int i = 0; i < N; ++i)
        if (xs[i] < 0 || xs[i] >= V) return -1;
    double L_ce = 0.0, L_tv = 0.0, L_conf = 0.0;
    double *pd = (double *)malloc(sizeof(double) * (size_t)V);
    double *pt = (double *)malloc(sizeof(double) * (size_t)V);
    for (int i = 0; i < N; ++i) {
        const int k = i % gamma + 1;
        const double wk = exp(-(double)(k - 1) / (double)gamma);
        /* the two softmaxes (max-shifted) */
        double md = -INFINITY, mt = -INFINITY;
        for (int v = 0; v < V; ++v) {
            const double a = load_elem(zd, (size_t)i * V + v, dtype), b = load_elem(zt, (size_t)i * V + v, dtype);
            if (a > md) md = a;
            if (b > mt) mt = b;
        }
        double Sd = 0.0, St = 0.0;
        for (int v = 0; v < V; ++v) {
            pd[v] = exp(load_elem(zd, (size_t)i * V + v, dtype) - md);
            pt[v] = exp(load_elem(zt, (size_t)i * V + v, dtype) - mt);
            Sd += pd[v];
            St += pt[v];
        }
        const double lse_d = md + log(Sd), lse_t = mt + log(St);
        double tv = 0.0;
        for (int v = 0; v < V; ++v) {
            pd[v] /= Sd;
            pt[v] /= St;
            tv += fabs(pd[v] - pt[v]);
        }
        const double ce = lse_d - load_elem(zd, (size_t)i * V + xs[i], dtype);
        const double cstar = 1.0 - 0.5 * tv;
        const double si = (double)s[i];
        const double bce = softplus(si) - cstar * si;
        double *ro = row + (size_t)i * 6;
        ro[0] = lse_d; ro[1] = lse_t; ro[2] = ce; ro[3] = tv; ro[4] = cstar; ro[5] = bce;
        L_ce += wk * ce;
        L_tv += wk * tv;
        L_conf += wk * bce;
        if (grad_z) {
            double mean_sgn = 0.0; /* sum_u p^d_u sgn(p^d_u - p^t_u) */
            for (int v = 0; v < V; ++v) {
                const double dlt = pd[v] - pt[v];
                mean_sgn += pd[v] * (dlt > 0.0 ? 1.0 : dlt < 0.0 ? -1.0 : 0.0);
            }
            for (int v = 0; v < V; ++v) {
                const double dlt = pd[v] - pt[v];
                const double sg = dlt > 0.0 ? 1.0 : dlt < 0.0 ? -1.0 : 0.0;
                const double g_ce = pd[v] - (v == xs[i] ? 1.0 : 0.0);
                const double g_tv = pd[v] * (sg - mean_sgn);
                grad_z[(size_t)i * V + v] = wk / B * (a_ce * g_ce + a_tv * g_tv);
            }
        }
        if (grad_s) grad_s[i] = a_conf * wk / B * (1.0 / (1.0 + exp(-si)) - cstar);
    }
    free(pd);
    free(pt);
    loss[0] = L_ce / B;
    loss[1] = L_tv / B;
    loss[2] = L_conf / B;
    loss[3] = a_ce * loss[0] + a_tv * loss[1] + a_conf * loss[2];
    return 0;
}
