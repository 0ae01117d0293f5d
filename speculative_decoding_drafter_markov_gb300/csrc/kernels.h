// kernels.h -- host-side launchers of the DSpark kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dspark {

// ----- draft step (eqs. 4, 5): vocabulary-sliced partials of one step k ---------
// The bias operand of row i is either W1[x_prev[i * x_stride]] (Markov head) or
// the fp32 vector A_op + i * a_stride (RNN head).
struct RnnStep {
    int R, V, r, d, gamma, k, dtype;
    const void *W;                   // [3r, 2r + d]
    const void *W1;
    const int32_t *x_prev;           // x_{k-1} of request i at x_prev[i * x_stride], unless
    int x_stride;
    const unsigned long long *x_win; // set: x_{k-1} = the packed race winner x_win[i] of step k-1
    const float *Hpre;               // [R * gamma, 3r]
    const float *s_in;               // [R, r] state s_{k-1}
    float *s_out;                    // [R, r] state s_k (a different buffer)
    float *A;                        // [R, gamma, r]
    int32_t *err;
};

struct DraftStep {
    int R, V, r, gamma, k;          // k = 1..gamma
    int dtype;
    const void *U;                   // [R, gamma, V]
    const void *W1;                  // [V, r]
    const void *W2t;                 // [V, r]
    const int32_t *x_prev;           // Markov: token of row i at x_prev[i * x_stride]
    int x_stride;
    const float *A_op;               // RNN: operand of row i at A_op[i * a_stride]
    int a_stride;
    uint64_t seed, cycle;
    DraftPartial *part;              // [R, nparts] (tensor-core step: [2, R, nparts])
    int nparts;
    int32_t *err;
    // used by the tensor-core step, which also merges the partials and computes
    // the confidence itself
    const void *h;                   // [R, gamma, d]
    int d;
    const float *w, *sts_T;
    int32_t *x_out;
    float *logq, *lse, *c;
    float *conf_logit;               // [R, gamma] or null
    int *counters;                   // [number of M-tiles], zero at the start of the call
    unsigned long long *winners;     // [gamma, R] packed race winners, zero at the start of the call
    int step_index;                  // 1 for the first step launched since the counters were zeroed
    int nsteps;                      // tensor-core step: steps k .. k + nsteps - 1 in one launch
    int phase0;                      // tensor-core step: cross-CTA synchronisation points that
                                     // earlier launches of the same draft already passed
    // tensor-core RNN head (A_op set): the operand of step k' of the launch is
    // A_op + (k' - k) r; before it, the launch runs the state update of step k'
    // from `rnn` (s_in: the buffer holding s_{k-1}; the buffers alternate)
    RnnStep rnn;
    unsigned char *a_stage;          // RNN: [n_mtiles][kRnnStageBytes] operands prepared for the
                                     // bulk copy (rows beyond R zero)
};
// the RNN operand of one M-tile (128 rows x 256 K x hi/lo bf16) as the
// tensor-core step lays it out in shared memory
constexpr size_t kRnnStageBytes = 131072;
int draft_step_nparts(int V);  // CUDA-core path: one partial per 64-entry slice
cudaError_t launch_draft_step(const DraftStep &p, cudaStream_t s);
// tensor-core path (bf16, r in {64, 128, 192, 256}, V % 8 == 0)
bool draft_step_tc_supported(const DraftStep &p);
void draft_step_tc_shape(int R, int V, bool rnn, int *nparts, int *n_mtiles);
cudaError_t launch_draft_step_tc(const DraftStep &p, cudaStream_t s);
cudaError_t launch_wait_selfcheck(const int *flag, int target, int mode, uint64_t limit_ns, int32_t *err,
                                  cudaStream_t s);
// shared tensor-core helpers
int sm_count();
bool tc_available();
bool tc_kernels_enabled();
bool encode_w2t_map(CUtensorMap *m, const void *W2t, int V, int r, int BN);
bool encode_kmajor_map(CUtensorMap *m, const void *base, int rows, int K, int ld, int box_rows);
bool encode_u_map(CUtensorMap *m, const void *U, int R, int gamma, int V, int MV);
void tc_grid_shape(int R, int V, int MV, int BN, int *nparts, int *n_mtiles);

// ----- reduce partials of step k, write x, logq, lse; confidence (eq. 7) -------
struct DraftReduce {
    int R, V, r, d, gamma, k, dtype;
    const DraftPartial *part;
    int nparts;
    const void *h;                   // [R, gamma, d]
    const void *W1;                  // [V, r]
    const int32_t *x_prev;           // token x_{k-1} of row i at x_prev[i * x_stride]
    int x_stride;
    const float *w;                  // [d + r]
    const float *sts_T;              // [gamma] or null
    int32_t *x;
    float *logq, *lse, *c;           // [R, gamma]
    float *conf_logit;               // [R, gamma] or null
    int32_t *err;
};
cudaError_t launch_draft_reduce(const DraftReduce &p, cudaStream_t s);

// ----- RNN head (eq. 6) --------------------------------------------------------
// Hpre[m, o] = sum_j h[m, j] W[o, 2r + j] for every (request, step) row m.
cudaError_t launch_rnn_hproj(int M, int d, int r, int dtype, const void *h, const void *W,
                             float *Hpre, cudaStream_t s);
// One recurrent step: gates from [s; W1[x_{k-1}]] and Hpre; updates state in
// place, writes A[:, k-1, :] = tanh(W_o z_k).
cudaError_t launch_rnn_step(const RnnStep &p, cudaStream_t s);
// Hpre [M, 3r] = h [M, d] W[:, 2r:]^T on the tensor cores (bf16, tcgen05, gemm_tc.cu)
bool hproj_tc_supported(int M, int d, int r, int dtype, const void *h, const void *W, const float *Hpre);
cudaError_t launch_hproj_tc(int M, int d, int r, const void *h, const void *W, float *Hpre, int32_t *err,
                            cudaStream_t s);

// ----- scheduler (Module E, Algorithm 1; async variant) ---------------------
cudaError_t launch_schedule(const dspark_sched_args &a, cudaStream_t s);
size_t schedule_smem_bytes(int R, int gamma);

// ----- flattened batch tags ---------------------------------------------------
cudaError_t launch_build_tags(int R, int gamma, const int32_t *ell, int32_t *tags, int32_t *N_out,
                              int32_t *err, cudaStream_t s);

// ----- verification -------------------------------------------------------------
struct VerifyWs {
    float *lse_p;          // [N]
    int32_t *first_rej;    // [R]
    int32_t *ell;          // [R]
    int32_t *row_of;       // [R, gamma + 1]
    VerifyPartial *part;   // [R, nparts] slice sums (CUDA-core phase 2)
    int *done;             // [kVerifyMaxMTiles] CTAs of an M-tile that published (tensor-core phase 2)
    int *tctr;             // [kVerifyMaxMTiles] vocabulary tiles taken per M-tile (tensor-core phase 2)
    float *csum;           // [ceil(V / 16), R] sums of 16 consecutive weights (tensor-core phase 2)
    unsigned long long *ttot;  // [tiles + ceil(tiles / 32), R] sums over each vocabulary tile, then over each
                               // run of 32 tiles, fixed point 2^-47 (tensor-core phase 2; tiles <= ceil(V / 64))
    int nparts;
};
constexpr int kVerifyMaxMTiles = 64;
size_t verify_ws_bytes(int R, int gamma, int V, int N);
VerifyWs verify_ws_carve(void *ws, int R, int gamma, int V, int N);
cudaError_t launch_verify(const dspark_verify_args &a, const VerifyWs &w, cudaStream_t s);
bool verify_tc_supported(const dspark_verify_args &a);
int verify_tc_tiles(const dspark_verify_args &a);  // vocabulary tiles of the tensor-core phase 2
cudaError_t launch_verify_phase2_tc(const dspark_verify_args &a, VerifyWs &w, cudaStream_t s);

// ----- acceptance diagnostics and training losses ------------------------------------
cudaError_t launch_accept_stats(const dspark_accept_stats_args &a, cudaStream_t s);
cudaError_t launch_train_losses(const dspark_train_loss_args &a, cudaStream_t s);

// ----- philox check ------------------------------------------------------------------
cudaError_t launch_philox(const uint32_t *ctr, uint64_t seed, int n, uint32_t *out, cudaStream_t s);

// ----- sequential temperature scaling (Module D) --------------------------------
constexpr int kStsMaxGamma = DSPARK_STS_MAX_GAMMA;
constexpr int kStsMaxBins = DSPARK_STS_MAX_BINS;
struct StsFit {
    int M, gamma, G, n_bins;
    const float *logit;        // [M, gamma]
    const int32_t *n_accept;   // [M]
    const float *grid;         // [G]
    float *T;                  // [gamma]
    double *ece;               // [gamma]
    double *curve;             // [gamma, G] or null
    int32_t *err;
};
size_t sts_ws_bytes(int M, int gamma, int G, int n_bins);
cudaError_t launch_sts_fit(const StsFit &f, void *ws, cudaStream_t s);

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace dspark
