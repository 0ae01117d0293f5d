/*
 * dspark.h -- C ABI of the DSpark per-cycle hot path on one GB300 (sm_103a).
 *
 * The method is DSpark's semi-autoregressive draft + confidence-scheduled
 * verification, as described in
 *   [D] "DSpark: confidence-scheduled speculative decoding" (ai-papers-daily
 *       digest): eq. (4) causal block distribution, eq. (5) Markov head,
 *       eq. (6) RNN head, eq. (7) confidence head, Module D (sequential
 *       temperature scaling), Module E + Algorithm 1 (prefix scheduler),
 *       Appendix A, production section (async top-K, flattened batch);
 *   [E] "DSpark explained" (interactive explainer), section 06 (single-token
 *       rejection rule).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; row-major,
 *   contiguous, with the shapes given per field.  The library allocates no
 *   device memory: scratch comes from the caller through `ws`, whose size the
 *   matching *_workspace_size() function returns (256-byte aligned pointer).
 * - Every call only enqueues work on `stream` (a cudaStream_t) and returns
 *   without synchronising.  Calls on one stream run in order.
 * - dtype: DSPARK_F32 or DSPARK_BF16 applies to U, h, W1, W2t, W and T.
 *   Logits accumulate in fp32 whatever the storage type.
 * - Return value: DSPARK_OK, or an error code for a problem the host can see
 *   (bad shape, NULL pointer, unsupported size, CUDA launch failure); the
 *   message is in dspark_last_error() (thread-local).  Problems only the
 *   device can see (a token id >= V, malformed tags, a confidence outside
 *   [0, 1], non-finite logits) are written as the first non-zero error code
 *   into `*err` (a device int32 the caller zeroes; may be NULL to ignore) and
 *   the outputs of the affected rows are then unspecified.
 * - Sampling is deterministic given (seed, cycle): Philox-4x32-10 with
 *   key = (seed lo, seed hi) and counter = (w0, w1, request, cycle << 2 | stream);
 *   stream 0 the draft draw (w0 = b / 2 for vocabulary block b of 16 entries,
 *   w1 = step k; words 2 (b % 2) and 2 (b % 2) + 1 are block b's uniforms u_b
 *   and u'_b): the block is argmax_b ln S_b - ln(-ln u_b) (S_b the block's sum
 *   of exp(z), ties to the lowest b), the token the first entry of that block
 *   whose running sum of exp(z) exceeds u'_b S_b,
 *   stream 1 acceptance uniforms (w0 = 0, w1 = position j, word 0),
 *   stream 2 the residual / bonus draw (w0 = 0, w1 = position, word 0): one
 *   uniform u per request, the token the first v whose cumulative weight
 *   (fp32, vocabulary order) exceeds u times the total weight.
 *   A word w maps to u = ((w >> 9) + 1/2) 2^-23.  Only the low 30 bits of
 *   `cycle` enter the counter.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

typedef struct CUstream_st *dspark_stream_t; /* same type as cudaStream_t */

enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVAL = 1,       /* bad argument: NULL pointer, shape, mode     */
    DSPARK_ERR_RANGE = 2,       /* token id >= V, B outside the SPS table,     */
                                /* confidence outside [0, 1]                   */
    DSPARK_ERR_NONFINITE = 3,   /* NaN / Inf logits left no sample             */
    DSPARK_ERR_CUDA = 4,        /* a CUDA runtime call failed                  */
    DSPARK_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up          */
    DSPARK_ERR_UNSUPPORTED = 6  /* size beyond what this build handles         */
};

enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 };
enum { DSPARK_SCHED_SYNC = 0, DSPARK_SCHED_ASYNC = 1 };

/* ------------------------------------------------------------------------ */
/* Draft, Markov head.  [D] eq. (5) B(x_{k-1}, .) = W_1[x_{k-1}] W_2 added to  */
/* the base logits U_k in eq. (4), sampled left to right for k = 1..gamma     */
/* from the anchor x_0; confidence c_k = sigma(w^T [h_k ; W_1[x_{k-1}]] / T_k) */
/* by eq. (7) with the Module D temperature T_k (1 when sts_T is NULL).       */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t R;            /* requests                                           */
    int32_t gamma;        /* block length                                       */
    int32_t V;            /* vocabulary                                         */
    int32_t r;            /* rank of W_1 W_2                                    */
    int32_t d;            /* hidden size of h                                   */
    int32_t dtype;        /* DSPARK_F32 | DSPARK_BF16                           */
    const void *U;        /* [R, gamma, V] base logits U_k                      */
    const void *h;        /* [R, gamma, d] backbone hidden states h_k           */
    const void *W1;       /* [V, r] embedding table W_1                         */
    const void *W2t;      /* [V, r] W_2 transposed: row v is column v of W_2    */
    const float *w;       /* [d + r] confidence weights (hidden part first)     */
    const float *sts_T;   /* [gamma] temperatures T_k, or NULL for 1            */
    const int32_t *anchor;/* [R] anchor tokens x_0                              */
    uint64_t seed;        /* Philox key                                         */
    uint64_t cycle;       /* decoding-cycle counter (Philox counter word 3)     */
    int32_t *x;           /* out [R, gamma] drafted tokens x_1..x_gamma         */
    float *logq;          /* out [R, gamma] log q_k(x_k)                        */
    float *lse;           /* out [R, gamma] log sum_v exp(U_k(v) + B_k(v))      */
    float *c;             /* out [R, gamma] confidences c_k                     */
    int32_t *err;         /* device error word (see conventions), or NULL       */
    float *conf_logit;    /* out [R, gamma] w^T [h_k ; W_1[x_{k-1}]], the logit  */
                          /* before 1/T_k (the input of dspark_sts_fit), or NULL */
} dspark_draft_args;

DSPARK_API size_t dspark_draft_markov_workspace_size(const dspark_draft_args *a);
DSPARK_API int dspark_draft_markov(const dspark_draft_args *a, void *ws, dspark_stream_t stream);
/* Step k (1..gamma) of the same loop alone: reads x_{k-1} (the anchor for
 * k = 1, else column k-2 of a->x) and writes column k-1 of x, logq, lse, c.
 * dspark_draft_markov equals calls for k = 1..gamma in order on one stream
 * with one workspace; the split lets an engine interleave other work between
 * steps.  Step 1 (re)starts the per-draft step counters kept in the
 * workspace, so a step k > 1 must follow steps 1..k-1 of the same draft.
 * (dspark_draft_markov itself runs all gamma steps in one launch on the
 * tensor-core path.) */
DSPARK_API int dspark_draft_markov_step(const dspark_draft_args *a, int32_t k, void *ws,
                                        dspark_stream_t stream);

/* Markov-head draft that allocates nothing and takes no workspace.
 *
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory: a plugin living inside another runtime whose
 * caching allocator already owns the device's memory, a plain C host with no
 * allocator of its own, or a code path that must not call cudaMalloc because
 * that call can synchronise the device.  Such callers still pass every input
 * and output tensor; only the scratch (the per-slice partial results the
 * steps exchange) comes from a fixed array inside the library, which every
 * GPU that loads the library holds until the process exits.
 *
 * - Limit: the scratch is what dspark_draft_markov_workspace_size() returns
 *   for the same arguments -- 32 bytes per (request, vocabulary range), once
 *   per step on the tensor-core path, plus 8 bytes per (request, step) and
 *   256, each part rounded up to 256 bytes; the ranges are one per SM on the
 *   tensor-core path (bf16, r a multiple of 64 up to 256, V a multiple of 8:
 *   all the standard workloads, under 11 MiB) and ceil(V / 64) on the
 *   CUDA-core path --
 *   and the array holds
 *   DSPARK_NOALLOC_SCRATCH_BYTES (16 MiB).  Larger needs return
 *   DSPARK_ERR_UNSUPPORTED (message in dspark_last_error()) and launch nothing.
 * - The first call on each device looks up the array's device address (with
 *   that device current) and caches it with the id of the device's current
 *   context; a call in another context of the device (after cudaDeviceReset,
 *   for instance, which unloads the module) looks it up again.  Make the first
 *   call in each context before any stream capture on the device.
 * - Every call on a device shares the one array.  Each call first clears the
 *   part that must start at zero (completion counters, with an asynchronous
 *   memset on the stream) and every step overwrites the rest before reading
 *   it, but calls that overlap on the GPU (different streams, or different
 *   host threads) race: serialise them, e.g. by issuing them on one stream.
 * Results equal dspark_draft_markov's for the same arguments. */
#define DSPARK_NOALLOC_SCRATCH_BYTES (16u << 20)
DSPARK_API int dspark_draft_markov_noalloc(const dspark_draft_args *a, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Draft, RNN head.  [D] eq. (6): z_k = [s_{k-1}; W_1[x_{k-1}]; h_k],          */
/* s_k = sigma(W_g z_k) s_{k-1} + (1 - sigma(W_g z_k)) tanh(W_c z_k),          */
/* B_k = W_2^T tanh(W_o z_k); otherwise as the Markov head.                    */
/* ------------------------------------------------------------------------ */
typedef struct {
    dspark_draft_args base; /* fields as for the Markov head                    */
    const void *W;          /* [3r, 2r + d]: rows [0,r) W_g, [r,2r) W_c, [2r,3r) W_o */
    const float *s0;        /* [R, r] initial state, or NULL for s_0 = 0        */
    float *A;               /* out [R, gamma, r] A_k = tanh(W_o z_k), the vector */
                            /* whose product with W_2 is B_k (verify needs it)  */
    float *s_out;           /* out [R, r] final state s_gamma, or NULL          */
} dspark_rnn_args;

/* The h_k columns of W do not depend on the recurrence: W[:, 2r:] h_k is
 * formed for all (request, k) first, one bf16 GEMM on the tensor cores
 * (tcgen05; fp32, or shapes it does not take -- d or 2r + d not a multiple of
 * 8 -- go to a CUDA-core kernel).  The workspace holds the draft scratch, two
 * [R, r] state buffers, the [R gamma, 3r] fp32 projection and 128 KiB per
 * 128 requests for the bf16 operands the tensor-core steps prepare. */
DSPARK_API size_t dspark_draft_rnn_workspace_size(const dspark_rnn_args *a);
DSPARK_API int dspark_draft_rnn(const dspark_rnn_args *a, void *ws, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Hardware-aware prefix scheduler.  [D] Module E, Algorithm 1:               */
/* a_{r,j} = prod_{i<=j} c_{r,i}; pool E = {(r,j): a_{r,j} > 0} sorted by a    */
/* descending (ties: request, then position, ascending); scan with            */
/* B = R + #admitted, tau = R + sum admitted a, Theta = tau * SPS(B).         */
/*  - DSPARK_SCHED_SYNC: Algorithm 1 with the early-stop break.                */
/*  - DSPARK_SCHED_ASYNC (production section): admit the top min(K, |E|)      */
/*    entries of the current order, no break, with K read from *K_in (the     */
/*    capacity computed two cycles earlier); *K_in < 0 or K_in == NULL falls  */
/*    back to SYNC.  Both modes write *K_out = argmax_m Theta(m) over the     */
/*    current pool without break (smallest m on ties), for use at cycle t+2.  */
/* Number formats: a is an fp32 running product; tau is summed exactly as     */
/* integers in units of 2^-32 (each a rounded to nearest-even on that grid);  */
/* Theta = (tau units * 2^-32) * SPS(B) in fp64.  Results are bit-exact.      */
/* Limits: R * gamma <= 8192.  The table must cover B in [R, R (gamma + 1)]   */
/* (checked on the host: DSPARK_ERR_RANGE).                                   */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t R, gamma;
    const float *c;        /* [R, gamma] confidences, each in [0, 1]            */
    const double *sps;     /* [B_count] SPS(B_min + i), steps per second         */
    int32_t B_min, B_count;
    int32_t mode;          /* DSPARK_SCHED_SYNC | DSPARK_SCHED_ASYNC             */
    const int32_t *K_in;   /* device scalar: async capacity, or NULL             */
    int32_t *ell;          /* out [R] verify lengths l_r in 0..gamma             */
    int32_t *K_out;        /* out device scalar: capacity for cycle t + 2        */
    double *theta_best;    /* out device scalar: Theta at the admitted point     */
    float *a;              /* out [R, gamma] survival products, or NULL          */
    int32_t *err;
} dspark_sched_args;

DSPARK_API size_t dspark_schedule_workspace_size(const dspark_sched_args *a);
DSPARK_API int dspark_schedule(const dspark_sched_args *a, void *ws, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Flattened batch layout ([D] production section, marker tensor): from     */
/* ell [R] write tags [N, 2] = (request, position) for positions 0..l_r of   */
/* each request in request order, and N = sum_r (1 + l_r) to *N_out (device).*/
/* tags must hold R (gamma + 1) rows.                                         */
/* ------------------------------------------------------------------------ */
DSPARK_API int dspark_build_tags(int32_t R, int32_t gamma, const int32_t *ell, int32_t *tags,
                                 int32_t *N_out, int32_t *err, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Lossless verification.  [E] section 06: accept x_{j+1} with probability    */
/* min(1, p_j(x_{j+1}) / q_{j+1}(x_{j+1})), test: log u < log p - log q with */
/* u from Philox stream 1; at the first rejection j* sample y from           */
/* norm(max(0, p_{j*} - q_{j*+1})) (q recomputed from U, the bias operand and */
/* W_2; p itself if the residual is empty); if all l_r tokens pass sample     */
/* the bonus y from p_{l_r}, both by inverse CDF (one stream-2 uniform per   */
/* request; the pages fix no sampler, any exact draw keeps the method        */
/* lossless).  Row i of T is the target's logits for position                */
/* tags[i] = (r, j), i.e. the distribution of x_{j+1} given x_0..x_j; rows    */
/* are grouped by request with positions 0..l_r ascending, every request      */
/* present (violations: DSPARK_ERR_INVAL in *err).                            */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t R, gamma, V, r, dtype;
    int32_t N;              /* rows of T (the capacity when N_dev is given)     */
    const int32_t *N_dev;   /* device scalar: rows in use, or NULL for N        */
    const void *T;          /* [N, V] target logits, flattened                  */
    const int32_t *tags;    /* [N, 2] (request, position)                       */
    const int32_t *anchor;  /* [R] x_0                                          */
    const int32_t *x;       /* [R, gamma] drafted tokens                        */
    const float *logq;      /* [R, gamma] from the draft                        */
    const float *lse;       /* [R, gamma] from the draft                        */
    const void *U;          /* [R, gamma, V] base logits (residual recompute)   */
    const void *W1;         /* [V, r] (Markov bias operand W_1[x_j])            */
    const void *W2t;        /* [V, r]                                           */
    const float *A;         /* [R, gamma, r] RNN bias operands, or NULL (Markov)*/
    uint64_t seed, cycle;
    int32_t *n_accept;      /* out [R] accepted draft tokens n_r                */
    int32_t *out_tokens;    /* out [R, gamma + 1] x_1..x_{n_r}, y, then -1      */
    int32_t *next_anchor;   /* out [R] y, the next cycle's anchor               */
    float *lse_p;           /* out [N] log sum exp of each row, or NULL         */
    float *logp;            /* out [N] log p_j(x_{j+1}) (NaN on last rows), or NULL */
    int32_t *err;
} dspark_verify_args;

DSPARK_API size_t dspark_verify_workspace_size(const dspark_verify_args *a);
DSPARK_API int dspark_verify(const dspark_verify_args *a, void *ws, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Sequential temperature scaling.  [D] Module D: c_i is the probability     */
/* that position i passes given that the positions before it passed, so the  */
/* prefix of length k is accepted with probability                           */
/* P_k = prod_{i<=k} sigma(s_i / T_i).  For k = 1..gamma in order, T_k is    */
/* the grid temperature that minimises the expected calibration error of P_k */
/* against the held-out outcome 1[n >= k], with T_1..T_{k-1} held fixed.     */
/* ECE: n_bins equal-width bins of [0, 1], bin(P) = min(floor(P n_bins),      */
/* n_bins - 1), ECE = (1/M) sum_b |sum_{m in b} (P_m - y_m)|.  The bin sums  */
/* are exact integers (P rounded to units of 2^-16 / n_bins), so results    */
/* depend on the order of the additions; the rounding can move a P within  */
/* 2^-17 / n_bins below a bin edge into the next bin.  Ties go to the lowest */
/* grid index.                                                               */
/* The fitted T is the draft's sts_T.  Device-side errors: a grid point that */
/* is not a positive finite number is skipped (DSPARK_ERR_INVAL), a NaN logit */
/* counts as 0 (DSPARK_ERR_NONFINITE), n outside 0..gamma is clamped          */
/* (DSPARK_ERR_RANGE).                                                        */
/* ------------------------------------------------------------------------ */
#define DSPARK_STS_MAX_GAMMA 64
#define DSPARK_STS_MAX_BINS 64
typedef struct {
    int32_t M;               /* held-out draft blocks                            */
    int32_t gamma;           /* positions per block (<= DSPARK_STS_MAX_GAMMA)    */
    int32_t G;               /* grid points                                      */
    int32_t n_bins;          /* ECE bins (1..DSPARK_STS_MAX_BINS)                */
    const float *logit;      /* [M, gamma] confidence logits s_k (conf_logit of  */
                             /* the draft, taken with T = 1)                     */
    const int32_t *n_accept; /* [M] accepted prefix length of each block, with   */
                             /* all gamma positions verified                     */
    const float *grid;       /* [G] candidate temperatures                       */
    float *T;                /* out [gamma] fitted temperatures T_k              */
    double *ece;             /* out [gamma] ECE of P_k at the fitted T_k         */
    double *curve;           /* out [gamma, G] ECE at every grid point, or NULL  */
    int32_t *err;            /* device error word, or NULL                       */
} dspark_sts_args;

/* Scratch: the [gamma, G, n_bins] bin sums (8 bytes each), gamma counters and
 * two [M] fp32 prefix-product buffers.  One launch per position on the given
 * stream, after one memset. */
DSPARK_API size_t dspark_sts_fit_workspace_size(const dspark_sts_args *a);
DSPARK_API int dspark_sts_fit(const dspark_sts_args *a, void *ws, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Acceptance diagnostics ([D] analysis 1: the per-position conditional      */
/* acceptance rate, whose denominator counts only the instances whose       */
/* positions 1..k-1 were all accepted; [D] offline results: the acceptance  */
/* length tau = accepted drafted tokens + the target's own token).           */
/* For the R requests of one cycle -- n_accept from dspark_verify, ell the    */
/* verified lengths (the scheduler's ell; NULL means gamma for all; ell < 0:  */
/* not in this cycle's batch, counted nowhere) -- the call ADDS into caller-  */
/* owned device counters, so consecutive cycles accumulate:                   */
/*   reached [gamma]   position k (index k-1) verified with 1..k-1 accepted   */
/*                     (ell >= k and n >= k - 1);                             */
/*   accepted [gamma]  position k accepted (n >= k);                          */
/*   tau_hist [gamma + 1]  requests by n (= tau - 1);                          */
/*   ell_hist [gamma + 1]  requests by ell (may be NULL).                      */
/* The conditional acceptance at position k is accepted / reached.  A request */
/* with n outside 0..min(ell, gamma) is skipped and DSPARK_ERR_RANGE written  */
/* to *err.  gamma <= DSPARK_DIAG_MAX_GAMMA.  No workspace; one launch.        */
/* ------------------------------------------------------------------------ */
#define DSPARK_DIAG_MAX_GAMMA 1024
typedef struct {
    int32_t R, gamma;
    const int32_t *n_accept;      /* [R]                                      */
    const int32_t *ell;           /* [R] or NULL                              */
    unsigned long long *reached;  /* [gamma]      accumulated                 */
    unsigned long long *accepted; /* [gamma]      accumulated                 */
    unsigned long long *tau_hist; /* [gamma + 1]  accumulated                 */
    unsigned long long *ell_hist; /* [gamma + 1]  accumulated, or NULL        */
    int32_t *err;                 /* device error word, or NULL               */
} dspark_accept_stats_args;

DSPARK_API int dspark_accept_stats(const dspark_accept_stats_args *a, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Drafter training losses ([D] Module F, eqs. 8-12) over B blocks of gamma   */
/* positions, row i = b gamma + k - 1, with w_k = exp(-(k - 1) / gamma):      */
/*   p_d = softmax(zd_i), p_t = softmax(zt_i) over V;                          */
/*   ce_i = -log p_d(xs_i); tv_i = ||p_d - p_t||_1; c*_i = 1 - tv_i / 2 (eq. 8);*/
/*   bce_i = -[c* log c + (1 - c*) log(1 - c)], c = sigma(s_i), evaluated as   */
/*           softplus(s_i) - c*_i s_i;                                         */
/*   L_ce, L_tv, L_conf = (1/B) sum_i w_k (ce_i, tv_i, bce_i)  (eqs. 9-11);    */
/*   L = a_ce L_ce + a_tv L_tv + a_conf L_conf  (eq. 12; the pages' defaults   */
/*       are 0.1, 0.9, 1.0).                                                   */
/* Outputs: row [N, 6] f32 = (lse_d, lse_t, ce, tv, c*, bce) per row (may be  */
/* NULL); loss [4] f64 = (L_ce, L_tv, L_conf, L), overwritten; grad_z [N, V]  */
/* f32 = dL/dzd with c* held fixed as a label (may be NULL: forward only):    */
/* w_k / B [a_ce (p_d - onehot(xs)) + a_tv p_d (sgn(p_d - p_t) - sum_u p_d,u   */
/* sgn_u)], sgn(0) = 0; grad_s [N] f32 = dL/ds = a_conf w_k / B (c - c*) (may */
/* be NULL).  zd, zt: dtype f32 or bf16, 16-byte aligned rows (V a multiple  */
/* of 8 for bf16, of 4 for f32).  Row sums run in fp32, the loss totals in   */
/* fp64 (added in an unspecified order).  A token outside 0..V-1 writes       */
/* DSPARK_ERR_RANGE to *err and that row's terms are skipped.  No workspace.  */
/* One launch.  Each row is swept three times (twice without grad_z).  For  */
/* V <= ~226K (bf16) or ~113K (f32) a cluster of 8 CTAs holds the row pair   */
/* in shared memory, 1/8 each, and HBM sees it once; for larger V the second */
/* and third sweeps read the row back from L2.                               */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t B, gamma, V, dtype;
    const void *zd;          /* [N, V] draft logits, N = B gamma                 */
    const void *zt;          /* [N, V] target logits                             */
    const int32_t *xs;       /* [N] target tokens                                */
    const float *s;          /* [N] confidence logits                            */
    float a_ce, a_tv, a_conf;
    float *row;              /* out [N, 6] or NULL                               */
    double *loss;            /* out [4]                                          */
    float *grad_z;           /* out [N, V] or NULL                               */
    float *grad_s;           /* out [N] or NULL                                  */
    int32_t *err;            /* device error word, or NULL                       */
} dspark_train_loss_args;

DSPARK_API int dspark_train_losses(const dspark_train_loss_args *a, dspark_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Helpers                                                                    */
/* ------------------------------------------------------------------------ */
/* Message of the last failing call on this host thread ("" if none). */
DSPARK_API const char *dspark_last_error(void);
/* Library version as major * 10000 + minor * 100 + patch. */
DSPARK_API int dspark_version(void);
/* Self-check of the device-side failure detection (no counterpart in the
 * pages).  Every spin-wait in the tensor-core kernels -- a CTA waiting for the
 * other CTAs of its M-tile, a role waiting on an mbarrier -- gives up after a
 * wall-clock limit, writes DSPARK_ERR_TIMEOUT into the error word and returns.
 * This call runs the same two waits on a condition that nothing satisfies
 * unless the caller set it: mode 0 waits for *flag >= target (a device int32);
 * mode 1 waits on a fresh mbarrier that completes only when target <= 0.
 * limit_ns in (0, 2e9].  After the stream reaches it, *err holds
 * DSPARK_ERR_TIMEOUT if the wait ran out, else it is unchanged. */
DSPARK_API int dspark_wait_selfcheck(const int32_t *flag, int32_t target, int32_t mode, uint64_t limit_ns,
                                     int32_t *err, dspark_stream_t stream);

/* Philox-4x32-10 on the device: out[i][0..3] for counters ctr[i][0..3] and
 * key (seed lo, seed hi), i < n.  Exposes the sampler's generator for checks. */
DSPARK_API int dspark_philox(const uint32_t *ctr, uint64_t seed, int32_t n, uint32_t *out,
                             dspark_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
