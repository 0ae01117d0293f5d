/*
 * dspark_oracle.h -- plain CPU oracle for the DSpark per-cycle hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA library.
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load it; the product path never does.
 *
 * Single-threaded, fp64 arithmetic, written to be read against the pages:
 *   [D] "DSpark: confidence-scheduled speculative decoding" (ai-papers-daily
 *       digest): eq. (4) causal block distribution, eq. (5) Markov head,
 *       eq. (6) RNN head, eq. (7) confidence head, Module E + Algorithm 1
 *       (hardware-aware prefix scheduler), Appendix A (non-anticipation),
 *       production section (asynchronous top-K scheduler, flattened batch),
 *       Module D (sequential temperature scaling of the confidences).
 *   [E] "DSpark explained" (interactive explainer), section 06: single-token
 *       rule accept with min(1, p/q), else resample from norm(max(0, p-q)).
 *
 * Random numbers: Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11), implemented here from its
 * published definition.  Counter layout (a reading; the pages name no RNG):
 *   key     = (seed low 32 bits, seed high 32 bits)
 *   counter = (word0, word1, request, (cycle << 2) | stream)
 *   stream 0: draft draw              word0 = b / 2 for vocabulary block b (16
 *                                     entries), word1 = step k (1..gamma); words
 *                                     2 (b % 2) and 2 (b % 2) + 1 are block b's
 *                                     race and entry uniforms
 *   stream 1: acceptance uniforms     word0 = 0, word1 = row position j, word 0
 *   stream 2: residual / bonus draw   word0 = 0, word1 = row position, word 0
 *   stream 3: reserved for synthetic-input noise
 * Word to uniform: u = ((w >> 9) + 0.5) * 2^-23, strictly inside (0, 1).
 *
 * Parity pins for every function are in tests/test_oracle_*.py.
 */
#ifndef DSPARK_ORACLE_H
#define DSPARK_ORACLE_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of the tensor inputs */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* scheduler modes */
#define ORACLE_SCHED_SYNC 0     /* Algorithm 1 with the early-stop break     */
#define ORACLE_SCHED_ASYNC 1    /* top-K of the current order, K from t-2    */
#define ORACLE_SCHED_NOBREAK 2  /* backtracking global search (lossy; tests) */

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
double oracle_uniform(uint32_t word);
uint32_t oracle_philox_word(uint64_t seed, uint32_t w0, uint32_t w1, uint32_t req,
                            uint64_t cycle, uint32_t stream, uint32_t lane);

/* Markov-head draft (eqs. 4, 5, 7).  All requests independent; `reqs` lists
 * the requests to compute (NULL = all R, in order), outputs are indexed by
 * position in that list.  Optional outputs may be NULL.
 *   U [R, gamma, V], h [R, gamma, d], W1 [V, r], W2t [V, r] (row v = column v
 *   of W_2), w [d + r] f32, sts_T [gamma] f32 or NULL, anchor [R].
 * x_k is drawn in two levels (16-entry vocabulary blocks by the Gumbel-max
 * rule over their masses, then the entry of the winning block by inverse CDF).
 * Outputs: x [n, gamma], logq, lse, c [n, gamma]; the near-tie records
 * gap [n, gamma] = difference between the two best block scores, runner
 * [n, gamma] = the token the runner-up block gives, cdf_gap [n, gamma, 2] =
 * distances of the entry draw's target to the lower and upper ends of x's
 * interval (fractions of the block's mass), cdf_runner [n, gamma, 2] = the
 * entries across those ends (-1: none); z [n, gamma, V] logits,
 * logit [n, gamma] = w^T [h_k ; W_1[x_{k-1}]] (the confidence logit). */
int oracle_draft_markov(int R, int gamma, int V, int r, int d, int dtype,
                        const void *U, const void *h, const void *W1, const void *W2t,
                        const float *w, const float *sts_T, const int32_t *anchor,
                        uint64_t seed, uint64_t cycle, const int32_t *reqs, int n_reqs,
                        int32_t *x, double *logq, double *lse, double *c, double *gap,
                        int32_t *runner, double *cdf_gap, int32_t *cdf_runner, double *z,
                        double *logit);

/* RNN-head draft (eq. 6).  W [3r, 2r + d]: rows [0, r) gate, [r, 2r) candidate,
 * [2r, 3r) output.  s0 [R, r] f32 or NULL (zero).  Extra output: A [n, gamma, r],
 * the vector tanh(W_o z_k) whose product with W_2 is the bias B_k. */
int oracle_draft_rnn(int R, int gamma, int V, int r, int d, int dtype,
                     const void *U, const void *h, const void *W1, const void *W2t,
                     const void *W, const float *s0, const float *w, const float *sts_T,
                     const int32_t *anchor, uint64_t seed, uint64_t cycle,
                     const int32_t *reqs, int n_reqs, int32_t *x, double *logq,
                     double *lse, double *c, double *gap, int32_t *runner, double *cdf_gap,
                     int32_t *cdf_runner, double *z, double *A, double *logit);

/* Hardware-aware prefix scheduler (Module E, Algorithm 1; production async
 * variant).  c [R, gamma] f32; sps[i] = SPS(B_min + i) for i < B_count.
 * Outputs: ell [R], K_out (argmax of Theta over the sorted pool, no break),
 * theta_best, a [R, gamma] f32 (may be NULL).  Returns 0, or -1 if the table
 * does not cover B in [R, R(gamma + 1)]. */
int oracle_schedule(int R, int gamma, const float *c, const double *sps, int B_min,
                    int B_count, int mode, int K_in, int32_t *ell, int32_t *K_out,
                    double *theta_best, float *a);

/* Lossless verification ([E] section 06; [D] overview step 3).
 *   T [N, V] target logits of the flattened batch, tags [N][2] = (request,
 *   position), grouped by request with positions 0..ell_r ascending.
 *   x [R, gamma] drafted tokens, logq / lse [R, gamma] f32 from the draft.
 *   Residual bias: A [R, gamma, r] f32 if non-NULL (RNN head), else W1[x_n].
 * Requests listed in `reqs` (NULL = all) are verified; outputs are full-size
 * [R] / [R, gamma + 1] / [N] arrays, written only for those requests.
 *   n_accept [R], out_tokens [R, gamma + 1] (-1 padded), next_anchor [R],
 *   lse_p [N], logp [N] (NaN on rows without a test), margin [N] =
 *   (log p - log q) - log u.  The correction / bonus token y is drawn by
 *   inverse CDF: u from Philox stream 2 (counter (0, n, request, cycle), word
 *   0), y = the first v whose cumulative weight exceeds u * sum(w).
 *   gap [R, 2] = the distances of u * sum(w) to the lower and upper ends of
 *   y's interval, relative to sum(w); runner [R, 2] = the positive-weight
 *   indices across those ends (-1 if none).
 * Returns 0, or -1 on malformed tags. */
int oracle_verify(int R, int gamma, int V, int r, int dtype, int N, const void *T,
                  const int32_t *tags, const int32_t *anchor, const int32_t *x,
                  const float *logq, const float *lse, const void *U, const void *W1,
                  const void *W2t, const float *A, uint64_t seed, uint64_t cycle,
                  const int32_t *reqs, int n_reqs, int32_t *n_accept, int32_t *out_tokens,
                  int32_t *next_anchor, double *lse_p, double *logp, double *margin,
                  double *gap, int32_t *runner);

/* Sequential temperature scaling ([D] Module D).  logit [M, gamma] f32
 * confidence logits s_k of M held-out draft blocks, n_accept [M] their
 * accepted prefix lengths (0..gamma), grid [G] candidate temperatures (> 0),
 * n_bins equal-width ECE bins.  For k = 1..gamma in order, T_out[k-1] is the
 * grid point minimising the ECE of prod_{i<=k} sigma(s_i / T_i) against
 * 1[n >= k]; ece_out[k-1] is that minimum and curve [gamma, G] (may be NULL)
 * the ECE of every grid point.  T_prefix [gamma] (may be NULL) replaces the
 * chosen T_i in the products of the later positions.  near_edge [gamma, G]
 * (may be NULL) counts the samples whose P lies within edge_eps of an interior
 * bin edge: the only ones a perturbation of P below edge_eps can move to
 * another bin (tests derive their tolerances from it).  Returns 0, or -1 on a
 * bad argument (n_accept outside 0..gamma, a NaN logit, a grid point <= 0). */
int oracle_sts_fit(int M, int gamma, const float *logit, const int32_t *n_accept, int G,
                   const float *grid, int n_bins, const float *T_prefix, float *T_out,
                   double *ece_out, double *curve, double edge_eps, int32_t *near_edge);

/* Per-position acceptance diagnostics ([D] analysis 1: the per-position
 * conditional acceptance rate, whose denominator counts only the instances
 * whose positions 1..k-1 were all accepted; [D] offline results: the
 * acceptance length tau).  For R requests of one cycle, n_accept [R] accepted
 * drafted tokens and ell [R] verified drafted tokens (NULL = gamma for all;
 * ell < 0 = request not verified this cycle, counted nowhere).  ADDS into
 *   reached [gamma]: position k (index k-1) verified with 1..k-1 accepted,
 *                    i.e. ell >= k and n >= k - 1;
 *   accepted [gamma]: position k accepted, i.e. n >= k;
 *   tau_hist [gamma + 1]: index n = tau - 1 (tau = n + 1 tokens per cycle);
 *   ell_hist [gamma + 1] (may be NULL): index ell.
 * Returns 0, or -1 if some n lies outside 0..min(ell, gamma) (nothing added). */
int oracle_accept_stats(int R, int gamma, const int32_t *n_accept, const int32_t *ell, uint64_t *reached,
                        uint64_t *accepted, uint64_t *tau_hist, uint64_t *ell_hist);

/* Training losses of the drafter ([D] Module F, eqs. 8-12), for B blocks of
 * gamma positions (row i = b gamma + k - 1), in fp64:
 *   w_k = exp(-(k - 1) / gamma);
 *   p^d_i = softmax(zd_i), p^t_i = softmax(zt_i) over V (zd draft logits,
 *   zt target logits, dtype f32 or bf16);
 *   ce_i = -log p^d_i(xs_i) (xs the target's token);
 *   tv_i = || p^d_i - p^t_i ||_1;  cstar_i = 1 - tv_i / 2 (eq. 8);
 *   c_i = sigma(s_i) (s the confidence logit);
 *   bce_i = -[cstar_i log c_i + (1 - cstar_i) log(1 - c_i)], in the stable form
 *           softplus(s_i) - cstar_i s_i;
 *   L_ce = (1/B) sum_i w_k ce_i, L_tv = (1/B) sum_i w_k tv_i,
 *   L_conf = (1/B) sum_i w_k bce_i  (eqs. 9-11, averaged over the blocks);
 *   L = a_ce L_ce + a_tv L_tv + a_conf L_conf  (eq. 12).
 * Outputs: row [N, 6] = (lse_d, lse_t, ce, tv, cstar, bce) per row and
 * loss [4] = (L_ce, L_tv, L_conf, L).  If grad_z [N, V] is non-NULL it gets
 * dL/dzd with cstar held fixed (a label): w_k / B times
 *   a_ce (p^d - onehot(xs)) + a_tv p^d (sgn(p^d - p^t) - sum_u p^d_u sgn_u),
 * sgn(0) = 0; grad_s [N] (may be NULL) gets dL/ds = a_conf w_k / B (c - cstar).
 * Returns 0, or -1 on a token outside 0..V-1. */
int oracle_train_losses(int B, int gamma, int V, int dtype, const void *zd, const void *zt,
                        const int32_t *xs, const float *s, double a_ce, double a_tv, double a_conf,
                        double *row, double *loss, double *grad_z, double *grad_s);

#ifdef __cplusplus
}
#endif
#endif
