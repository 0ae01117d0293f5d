// abi.cu -- the C ABI declared in include/dspark.h: argument checks, workspace
// carving and kernel launches.  Nothing here synchronises or allocates.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cuda.h>

#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *where) {
    return fail(DSPARK_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

int ok() {
    g_last_error.clear();
    return DSPARK_OK;
}

constexpr int kMaxRank = 512;  // shared-memory bound of the CUDA-core draft kernels

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_draft(const dspark_draft_args *a) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->R < 1 || a->gamma < 1 || a->V < 1 || a->r < 1 || a->d < 0)
        return fail(DSPARK_ERR_INVAL, "bad shape R=%d gamma=%d V=%d r=%d d=%d", a->R, a->gamma, a->V,
                    a->r, a->d);
    if (a->dtype != DSPARK_F32 && a->dtype != DSPARK_BF16)
        return fail(DSPARK_ERR_INVAL, "bad dtype %d", a->dtype);
    if (a->r > kMaxRank) return fail(DSPARK_ERR_UNSUPPORTED, "rank r=%d above %d", a->r, kMaxRank);
    if (!a->U || !a->W1 || !a->W2t || !a->w || !a->anchor || !a->x || !a->logq || !a->lse || !a->c ||
        (a->d > 0 && !a->h))
        return fail(DSPARK_ERR_INVAL, "null tensor pointer");
    return DSPARK_OK;
}

// The step kernels' scratch: one partial per (request, vocabulary range) --
// ceil(V / 64) ranges on the CUDA-core path; one per CTA on the tensor-core
// path, for each of the gamma steps -- then the tensor-core step's
// per-M-tile completion counters and its [gamma, R] packed race winners, the
// part cleared at the start of a call.
constexpr size_t kCounterBytes = 256;

dspark::DraftStep step_template(const dspark_draft_args *a, const float *A_rnn) {
    dspark::DraftStep st{};
    st.R = a->R; st.V = a->V; st.r = a->r; st.gamma = a->gamma; st.dtype = a->dtype;
    st.U = a->U; st.W1 = a->W1; st.W2t = a->W2t;
    st.seed = a->seed; st.cycle = a->cycle;
    st.err = a->err;
    st.A_op = A_rnn;
    st.a_stride = a->gamma * a->r;
    st.h = a->h; st.d = a->d; st.w = a->w; st.sts_T = a->sts_T;
    st.x_out = a->x; st.logq = a->logq; st.lse = a->lse; st.c = a->c;
    st.conf_logit = a->conf_logit;
    return st;
}

bool use_tc_path(const dspark::DraftStep &st) {
    if (!dspark::draft_step_tc_supported(st)) return false;
    int np = 0, mt = 0;
    dspark::draft_step_tc_shape(st.R, st.V, st.A_op != nullptr, &np, &mt);
    return (size_t)mt * sizeof(int) <= kCounterBytes;  // one counter per M-tile
}

int step_nparts(const dspark::DraftStep &st, bool tc) {
    if (!tc) return dspark::draft_step_nparts(st.V);
    int np = 0, mt = 0;
    dspark::draft_step_tc_shape(st.R, st.V, st.A_op != nullptr, &np, &mt);
    return np;
}

size_t winners_bytes(const dspark_draft_args *a) {
    return dspark::align256(sizeof(unsigned long long) * (size_t)a->R * a->gamma);
}

size_t partials_bytes(const dspark_draft_args *a, const float *A_rnn) {
    const dspark::DraftStep st = step_template(a, A_rnn);
    const bool tc = use_tc_path(st);
    const int np = step_nparts(st, tc);
    return dspark::align256(sizeof(dspark::DraftPartial) * (size_t)a->R * np * (tc ? a->gamma : 1));
}

size_t draft_ws_bytes(const dspark_draft_args *a, const float *A_rnn) {
    return partials_bytes(a, A_rnn) + kCounterBytes + winners_bytes(a);
}

// the gamma sequential steps shared by both heads
int run_draft_loop(const dspark_draft_args *a, const float *A_rnn, void *part_ws, cudaStream_t s,
                   const dspark::RnnStep *rnn, int k_first, int k_last, unsigned char *a_stage = nullptr) {
    using namespace dspark;
    DraftStep st = step_template(a, rnn ? A_rnn : nullptr);
    st.part = static_cast<DraftPartial *>(part_ws);
    const bool use_tc = use_tc_path(st);
    st.nparts = step_nparts(st, use_tc);
    char *cleared = static_cast<char *>(part_ws) + partials_bytes(a, st.A_op);
    const size_t cleared_bytes = kCounterBytes + winners_bytes(a);
    st.counters = reinterpret_cast<int *>(cleared);
    st.winners = reinterpret_cast<unsigned long long *>(cleared + kCounterBytes);
    DraftReduce rd{};
    rd.R = a->R; rd.V = a->V; rd.r = a->r; rd.d = a->d; rd.gamma = a->gamma; rd.dtype = a->dtype;
    rd.part = st.part; rd.nparts = st.nparts;
    rd.h = a->h; rd.W1 = a->W1; rd.w = a->w; rd.sts_T = a->sts_T;
    rd.x = a->x; rd.logq = a->logq; rd.lse = a->lse; rd.c = a->c; rd.err = a->err;
    rd.conf_logit = a->conf_logit;
    if (use_tc && k_first == 1) {  // step 1 starts the step counters; later steps continue them
        cudaError_t e = cudaMemsetAsync(cleared, 0, cleared_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft counters");
    }
    if (use_tc) {
        // on the tensor cores all the steps run in one launch (the RNN head's
        // state updates between them, the first one included)
        st.k = k_first;
        st.step_index = k_first;
        st.phase0 = k_first - 1;  // Markov: one synchronisation point per step
        st.nsteps = k_last - k_first + 1;
        st.x_prev = k_first == 1 ? a->anchor : a->x + (k_first - 2);
        st.x_stride = k_first == 1 ? 1 : a->gamma;
        if (rnn) {
            if (k_first != 1 || !a_stage) return fail(DSPARK_ERR_INVAL, "RNN draft runs from step 1");
            st.rnn = *rnn;
            st.phase0 = 0;
            st.a_stage = a_stage;
        }
        cudaError_t e = launch_draft_step_tc(st, s);
        return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "draft steps (tensor cores)");
    }
    // the RNN state update of step k: s_{k-1} in buffer (k - 1) % 2, s_k into buffer k % 2
    auto rnn_update = [&](int k) {
        RnnStep rs = *rnn;
        if ((k & 1) == 0) {
            rs.s_in = rnn->s_out;
            rs.s_out = const_cast<float *>(rnn->s_in);
        }
        rs.k = k;
        rs.x_prev = k == 1 ? a->anchor : a->x + (k - 2);
        rs.x_stride = k == 1 ? 1 : a->gamma;
        rs.x_win = nullptr;
        return rs;
    };
    // CUDA cores: one step (and, RNN head, one state update) per launch
    for (int k = k_first; k <= k_last; ++k) {
        const int32_t *xp = k == 1 ? a->anchor : a->x + (k - 2);
        const int xs = k == 1 ? 1 : a->gamma;
        if (rnn) {
            cudaError_t e = launch_rnn_step(rnn_update(k), s);
            if (e != cudaSuccess) return cuda_fail(e, "rnn step");
            st.A_op = A_rnn + (size_t)(k - 1) * a->r;
        }
        st.k = k;
        st.step_index = k;
        st.nsteps = 1;
        st.x_prev = xp;
        st.x_stride = xs;
        cudaError_t e = launch_draft_step(st, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft step");
        rd.k = k;
        rd.x_prev = xp;
        rd.x_stride = xs;
        e = launch_draft_reduce(rd, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft reduce");
    }
    return DSPARK_OK;
}

}  // namespace

extern "C" {

DSPARK_API const char *dspark_last_error(void) { return g_last_error.c_str(); }

DSPARK_API int dspark_version(void) { return 100; }

DSPARK_API size_t dspark_draft_markov_workspace_size(const dspark_draft_args *a) {
    if (check_draft(a) != DSPARK_OK) return 0;
    return draft_ws_bytes(a, nullptr);
}

DSPARK_API int dspark_draft_markov(const dspark_draft_args *a, void *ws, dspark_stream_t stream) {
    int rc = check_draft(a);
    if (rc != DSPARK_OK) return rc;
    if (!ws) return fail(DSPARK_ERR_INVAL, "null workspace");
    rc = run_draft_loop(a, nullptr, ws, reinterpret_cast<cudaStream_t>(stream), nullptr, 1, a->gamma);
    return rc == DSPARK_OK ? ok() : rc;
}

DSPARK_API int dspark_draft_markov_step(const dspark_draft_args *a, int32_t k, void *ws,
                                        dspark_stream_t stream) {
    int rc = check_draft(a);
    if (rc != DSPARK_OK) return rc;
    if (k < 1 || k > a->gamma) return fail(DSPARK_ERR_INVAL, "step k=%d outside 1..%d", k, a->gamma);
    if (!ws) return fail(DSPARK_ERR_INVAL, "null workspace");
    rc = run_draft_loop(a, nullptr, ws, reinterpret_cast<cudaStream_t>(stream), nullptr, k, k);
    return rc == DSPARK_OK ? ok() : rc;
}

// Scratch of dspark_draft_markov_noalloc: a fixed device array, so that call
// never allocates.  Host code may only use its address as looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSPARK_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
// device address of the array per device, and the id of the context it was
// looked up in: a new context (e.g. after cudaDeviceReset) loads the module
// again, so the address is looked up again there
void *g_noalloc_ptr[kMaxDevices];
unsigned long long g_noalloc_ctx[kMaxDevices];

// driver entry points for the current context and its process-unique id
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
void *driver_fn(const char *name) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return ptr;
}

// id of the calling thread's current context (0: none yet, or unknown)
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
    static CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(DSPARK_ERR_UNSUPPORTED, "noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const unsigned long long ctx = current_ctx_id();
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current if needed
        if (e != cudaSuccess) return cuda_fail(e, "noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = current_ctx_id();
    }
    *out = g_noalloc_ptr[dev];
    return DSPARK_OK;
}
}  // namespace

DSPARK_API int dspark_draft_markov_noalloc(const dspark_draft_args *a, dspark_stream_t stream) {
    int rc = check_draft(a);
    if (rc != DSPARK_OK) return rc;
    const size_t need = draft_ws_bytes(a, nullptr);
    if (need > (size_t)DSPARK_NOALLOC_SCRATCH_BYTES)
        return fail(DSPARK_ERR_UNSUPPORTED,
                    "noalloc draft needs %zu bytes of scratch for R=%d V=%d; the fixed array holds %u",
                    need, a->R, a->V, (unsigned)DSPARK_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != DSPARK_OK) return rc;
    rc = run_draft_loop(a, nullptr, scratch, reinterpret_cast<cudaStream_t>(stream), nullptr, 1,
                        a->gamma);
    return rc == DSPARK_OK ? ok() : rc;
}

namespace {
// prepared operands of the tensor-core RNN step, one region per M-tile of 128 requests
size_t rnn_stage_bytes(const dspark_draft_args &b) { return (size_t)((b.R + 127) / 128) * dspark::kRnnStageBytes; }

size_t rnn_ws_bytes(const dspark_rnn_args *a) {
    const dspark_draft_args &b = a->base;
    return draft_ws_bytes(&b, a->A) + 2 * dspark::align256(sizeof(float) * (size_t)b.R * b.r) +
           dspark::align256(sizeof(float) * (size_t)b.R * b.gamma * 3 * b.r) + rnn_stage_bytes(b);
}
}  // namespace

DSPARK_API size_t dspark_draft_rnn_workspace_size(const dspark_rnn_args *a) {
    if (!a || check_draft(&a->base) != DSPARK_OK) return 0;
    return rnn_ws_bytes(a);
}

DSPARK_API int dspark_draft_rnn(const dspark_rnn_args *a, void *ws, dspark_stream_t stream) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    int rc = check_draft(&a->base);
    if (rc != DSPARK_OK) return rc;
    if (!a->W || !a->A) return fail(DSPARK_ERR_INVAL, "null RNN tensor pointer");
    if (!ws) return fail(DSPARK_ERR_INVAL, "null workspace");
    const dspark_draft_args &b = a->base;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t state_bytes = sizeof(float) * (size_t)b.R * b.r;
    char *p = static_cast<char *>(ws);
    void *part = p;
    p += draft_ws_bytes(&b, a->A);
    float *state0 = reinterpret_cast<float *>(p);
    p += dspark::align256(state_bytes);
    float *state1 = reinterpret_cast<float *>(p);
    p += dspark::align256(state_bytes);
    float *Hpre = reinterpret_cast<float *>(p);
    p += dspark::align256(sizeof(float) * (size_t)b.R * b.gamma * 3 * b.r);
    unsigned char *stage = reinterpret_cast<unsigned char *>(p);  // rows beyond R stay zero
    cudaError_t e = cudaMemsetAsync(stage, 0, rnn_stage_bytes(b), s);
    if (e != cudaSuccess) return cuda_fail(e, "rnn operand staging");
    e = a->s0 ? cudaMemcpyAsync(state0, a->s0, state_bytes, cudaMemcpyDeviceToDevice, s)
                          : cudaMemsetAsync(state0, 0, state_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "rnn state init");
    if (b.d > 0) {
        if (dspark::hproj_tc_supported(b.R * b.gamma, b.d, b.r, b.dtype, b.h, a->W, Hpre))
            e = dspark::launch_hproj_tc(b.R * b.gamma, b.d, b.r, b.h, a->W, Hpre, b.err, s);
        else
            e = dspark::launch_rnn_hproj(b.R * b.gamma, b.d, b.r, b.dtype, b.h, a->W, Hpre, s);
    } else {
        e = cudaMemsetAsync(Hpre, 0, sizeof(float) * (size_t)b.R * b.gamma * 3 * b.r, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "rnn h projection");
    dspark::RnnStep rs{};
    rs.R = b.R; rs.V = b.V; rs.r = b.r; rs.d = b.d; rs.gamma = b.gamma; rs.dtype = b.dtype;
    rs.W = a->W; rs.W1 = b.W1; rs.Hpre = Hpre; rs.A = a->A; rs.err = b.err;
    rs.s_in = state0;
    rs.s_out = state1;
    rc = run_draft_loop(&b, a->A, part, s, &rs, 1, b.gamma, stage);
    if (rc != DSPARK_OK) return rc;
    if (a->s_out) {
        const float *last = (b.gamma & 1) ? state1 : state0;
        e = cudaMemcpyAsync(a->s_out, last, state_bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "rnn state out");
    }
    return ok();
}

DSPARK_API size_t dspark_schedule_workspace_size(const dspark_sched_args *a) {
    (void)a;
    return 0;
}

DSPARK_API int dspark_schedule(const dspark_sched_args *a, void *ws, dspark_stream_t stream) {
    (void)ws;
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->R < 1 || a->gamma < 1) return fail(DSPARK_ERR_INVAL, "bad shape R=%d gamma=%d", a->R, a->gamma);
    if ((long long)a->R * a->gamma > 8192)
        return fail(DSPARK_ERR_UNSUPPORTED, "pool R*gamma=%lld above 8192", (long long)a->R * a->gamma);
    if (a->mode != DSPARK_SCHED_SYNC && a->mode != DSPARK_SCHED_ASYNC)
        return fail(DSPARK_ERR_INVAL, "bad mode %d", a->mode);
    if (!a->c || !a->sps || !a->ell || !a->K_out || !a->theta_best)
        return fail(DSPARK_ERR_INVAL, "null tensor pointer");
    if (a->B_count < 1 || a->B_min > a->R ||
        (long long)a->R * (a->gamma + 1) > (long long)a->B_min + a->B_count - 1)
        return fail(DSPARK_ERR_RANGE, "SPS table [%d, %d] does not cover B in [%d, %lld]", a->B_min,
                    a->B_min + a->B_count - 1, a->R, (long long)a->R * (a->gamma + 1));
    cudaError_t e = dspark::launch_schedule(*a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "schedule");
    return ok();
}

DSPARK_API int dspark_build_tags(int32_t R, int32_t gamma, const int32_t *ell, int32_t *tags,
                                 int32_t *N_out, int32_t *err, dspark_stream_t stream) {
    if (R < 1 || gamma < 0) return fail(DSPARK_ERR_INVAL, "bad shape R=%d gamma=%d", R, gamma);
    if (!ell || !tags || !N_out) return fail(DSPARK_ERR_INVAL, "null tensor pointer");
    cudaError_t e = dspark::launch_build_tags(R, gamma, ell, tags, N_out, err,
                                              reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "build tags");
    return ok();
}

static int check_verify(const dspark_verify_args *a) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->R < 1 || a->gamma < 1 || a->V < 1 || a->r < 1 || a->N < a->R ||
        (long long)a->N > (long long)a->R * (a->gamma + 1))
        return fail(DSPARK_ERR_INVAL, "bad shape R=%d gamma=%d V=%d r=%d N=%d", a->R, a->gamma, a->V,
                    a->r, a->N);
    if (a->dtype != DSPARK_F32 && a->dtype != DSPARK_BF16)
        return fail(DSPARK_ERR_INVAL, "bad dtype %d", a->dtype);
    if (a->r > kMaxRank) return fail(DSPARK_ERR_UNSUPPORTED, "rank r=%d above %d", a->r, kMaxRank);
    if (!a->T || !a->tags || !a->anchor || !a->x || !a->logq || !a->lse || !a->U || !a->W1 ||
        !a->W2t || !a->n_accept || !a->out_tokens || !a->next_anchor)
        return fail(DSPARK_ERR_INVAL, "null tensor pointer");
    if (!aligned16(a->T)) return fail(DSPARK_ERR_INVAL, "T must be 16-byte aligned");
    return DSPARK_OK;
}

DSPARK_API size_t dspark_verify_workspace_size(const dspark_verify_args *a) {
    if (check_verify(a) != DSPARK_OK) return 0;
    return dspark::verify_ws_bytes(a->R, a->gamma, a->V, a->N);
}

DSPARK_API int dspark_verify(const dspark_verify_args *a, void *ws, dspark_stream_t stream) {
    int rc = check_verify(a);
    if (rc != DSPARK_OK) return rc;
    if (!ws) return fail(DSPARK_ERR_INVAL, "null workspace");
    const dspark::VerifyWs w = dspark::verify_ws_carve(ws, a->R, a->gamma, a->V, a->N);
    cudaError_t e = dspark::launch_verify(*a, w, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "verify");
    return ok();
}

DSPARK_API size_t dspark_sts_fit_workspace_size(const dspark_sts_args *a) {
    if (!a || a->M < 1 || a->gamma < 1 || a->G < 1 || a->n_bins < 1) return 0;
    return dspark::sts_ws_bytes(a->M, a->gamma, a->G, a->n_bins);
}

DSPARK_API int dspark_sts_fit(const dspark_sts_args *a, void *ws, dspark_stream_t stream) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->M < 1 || a->gamma < 1 || a->G < 1 || a->n_bins < 1)
        return fail(DSPARK_ERR_INVAL, "bad shape M=%d gamma=%d G=%d n_bins=%d", a->M, a->gamma, a->G,
                    a->n_bins);
    if (a->gamma > dspark::kStsMaxGamma || a->n_bins > dspark::kStsMaxBins)
        return fail(DSPARK_ERR_UNSUPPORTED, "gamma=%d or n_bins=%d above %d", a->gamma, a->n_bins,
                    dspark::kStsMaxGamma);
    if (!a->logit || !a->n_accept || !a->grid || !a->T || !a->ece || !ws)
        return fail(DSPARK_ERR_INVAL, "null pointer");
    dspark::StsFit f{};
    f.M = a->M; f.gamma = a->gamma; f.G = a->G; f.n_bins = a->n_bins;
    f.logit = a->logit; f.n_accept = a->n_accept; f.grid = a->grid;
    f.T = a->T; f.ece = a->ece; f.curve = a->curve; f.err = a->err;
    cudaError_t e = dspark::launch_sts_fit(f, ws, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "sts fit");
}

DSPARK_API int dspark_accept_stats(const dspark_accept_stats_args *a, dspark_stream_t stream) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->R < 0 || a->gamma < 1) return fail(DSPARK_ERR_INVAL, "bad shape R=%d gamma=%d", a->R, a->gamma);
    if (a->gamma > DSPARK_DIAG_MAX_GAMMA)
        return fail(DSPARK_ERR_UNSUPPORTED, "gamma=%d above %d", a->gamma, DSPARK_DIAG_MAX_GAMMA);
    if ((a->R > 0 && !a->n_accept) || !a->reached || !a->accepted || !a->tau_hist)
        return fail(DSPARK_ERR_INVAL, "null pointer");
    if (a->R == 0) return ok();
    cudaError_t e = dspark::launch_accept_stats(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "accept stats");
}

DSPARK_API int dspark_train_losses(const dspark_train_loss_args *a, dspark_stream_t stream) {
    if (!a) return fail(DSPARK_ERR_INVAL, "null argument struct");
    if (a->B < 1 || a->gamma < 1 || a->V < 1)
        return fail(DSPARK_ERR_INVAL, "bad shape B=%d gamma=%d V=%d", a->B, a->gamma, a->V);
    if (a->dtype != DSPARK_F32 && a->dtype != DSPARK_BF16) return fail(DSPARK_ERR_INVAL, "bad dtype %d", a->dtype);
    if ((long long)a->B * a->gamma > 0x7fffffffll) return fail(DSPARK_ERR_UNSUPPORTED, "too many rows");
    const int vec = a->dtype == DSPARK_BF16 ? 8 : 4;
    if (a->V % vec) return fail(DSPARK_ERR_UNSUPPORTED, "V=%d not a multiple of %d", a->V, vec);
    if (!a->zd || !a->zt || !a->xs || !a->s || !a->loss) return fail(DSPARK_ERR_INVAL, "null pointer");
    if ((reinterpret_cast<uintptr_t>(a->zd) | reinterpret_cast<uintptr_t>(a->zt) |
         reinterpret_cast<uintptr_t>(a->grad_z)) & 15u)
        return fail(DSPARK_ERR_INVAL, "logit and gradient rows must be 16-byte aligned");
    cudaError_t e = dspark::launch_train_losses(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "train losses");
}

DSPARK_API int dspark_wait_selfcheck(const int32_t *flag, int32_t target, int32_t mode, uint64_t limit_ns,
                                     int32_t *err, dspark_stream_t stream) {
    if (!flag || !err) return fail(DSPARK_ERR_INVAL, "null pointer");
    if (mode != 0 && mode != 1) return fail(DSPARK_ERR_INVAL, "bad mode %d", mode);
    if (limit_ns == 0 || limit_ns > 2000000000ull) return fail(DSPARK_ERR_INVAL, "limit outside (0, 2 s]");
    cudaError_t e = dspark::launch_wait_selfcheck(flag, target, mode, limit_ns, err,
                                                  reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait self-check");
    return ok();
}

DSPARK_API int dspark_philox(const uint32_t *ctr, uint64_t seed, int32_t n, uint32_t *out,
                             dspark_stream_t stream) {
    if (n < 0 || (n > 0 && (!ctr || !out))) return fail(DSPARK_ERR_INVAL, "bad philox arguments");
    if (n == 0) return ok();
    cudaError_t e = dspark::launch_philox(ctr, seed, n, out, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "philox");
    return ok();
}

}  // extern "C"

namespace dspark {

namespace {
__global__ void philox_kernel(const uint32_t *ctr, uint64_t seed, int n, uint32_t *out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint4 w = philox4x32_10(make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]),
                                  philox_key(seed));
    out[4 * i] = w.x;
    out[4 * i + 1] = w.y;
    out[4 * i + 2] = w.z;
    out[4 * i + 3] = w.w;
}
}  // namespace

cudaError_t launch_philox(const uint32_t *ctr, uint64_t seed, int n, uint32_t *out, cudaStream_t s) {
    philox_kernel<<<(n + 255) / 256, 256, 0, s>>>(ctr, seed, n, out);
    return cudaGetLastError();
}

}  // namespace dspark
