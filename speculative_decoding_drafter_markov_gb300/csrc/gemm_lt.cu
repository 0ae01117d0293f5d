// gemm_lt.cu -- the RNN head's hidden-state projection, a plain dense GEMM,
// on the tensor cores through cuBLASLt.
//
// DSpark digest eq. (6): z_k = [s_{k-1}; W_1[x_{k-1}]; h_k] and W z_k with
// W = [W_g; W_c; W_o] of shape [3r, 2r + d].  The h_k columns of W do not
// depend on the recurrence, so W[:, 2r:] h_k is computed for every (request, k)
// up front: Hpre[R gamma, 3r] = h[R gamma, d] W[:, 2r:]^T, bf16 operands, fp32
// accumulation and output.  cuBLASLt is loaded at run time; without it the call
// returns cudaErrorNotSupported, which the C ABI reports.
#include <cublasLt.h>
#include <dlfcn.h>

#include <mutex>

#include "kernels.h"

namespace dspark {

namespace {

struct LtApi {
    decltype(&cublasLtCreate) create = nullptr;
    decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
    decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
    decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
    decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
    decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
    decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
    decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
    decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
    decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
    decltype(&cublasLtMatmul) matmul = nullptr;
    bool ok = false;
};

template <class F>
bool resolve(void *lib, const char *name, F &fn) {
    fn = reinterpret_cast<F>(dlsym(lib, name));
    return fn != nullptr;
}

const LtApi &lt_api() {
    static LtApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        void *lib = dlopen("libcublasLt.so.13", RTLD_NOW | RTLD_LOCAL);
        if (!lib) lib = dlopen("libcublasLt.so", RTLD_NOW | RTLD_LOCAL);
        if (!lib) return;
        api.ok = resolve(lib, "cublasLtCreate", api.create) &&
                 resolve(lib, "cublasLtMatmulDescCreate", api.desc_create) &&
                 resolve(lib, "cublasLtMatmulDescSetAttribute", api.desc_set) &&
                 resolve(lib, "cublasLtMatmulDescDestroy", api.desc_destroy) &&
                 resolve(lib, "cublasLtMatrixLayoutCreate", api.layout_create) &&
                 resolve(lib, "cublasLtMatrixLayoutDestroy", api.layout_destroy) &&
                 resolve(lib, "cublasLtMatmulPreferenceCreate", api.pref_create) &&
                 resolve(lib, "cublasLtMatmulPreferenceSetAttribute", api.pref_set) &&
                 resolve(lib, "cublasLtMatmulPreferenceDestroy", api.pref_destroy) &&
                 resolve(lib, "cublasLtMatmulAlgoGetHeuristic", api.heuristic) &&
                 resolve(lib, "cublasLtMatmul", api.matmul);
    });
    return api;
}

constexpr int kMaxDevices = 64;

// one handle per device, created on first use
cublasLtHandle_t lt_handle(const LtApi &api) {
    static std::mutex mu;
    static cublasLtHandle_t handles[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!handles[dev] && api.create(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
    return handles[dev];
}

}  // namespace

bool hproj_lt_available() { return lt_api().ok; }

// Hpre [M, 3r] (row-major) = h [M, d] W[:, 2r : 2r + d]^T, with W [3r, 2r + d]
// row-major.  In cuBLASLt's column-major terms: C (3r x M, ld 3r) =
// op(A) B with A the d x 3r view of W's h columns (ld 2r + d, transposed) and
// B the d x M view of h (ld d).
cudaError_t launch_hproj_lt(int M, int d, int r, const void *h, const void *W, float *Hpre, void *lt_ws,
                            size_t lt_ws_bytes, cudaStream_t s) {
    const LtApi &api = lt_api();
    if (!api.ok) return cudaErrorNotSupported;
    cublasLtHandle_t handle = lt_handle(api);
    if (!handle) return cudaErrorNotSupported;
    const int N = 3 * r, ldw = 2 * r + d;
    const void *A = static_cast<const __nv_bfloat16 *>(W) + 2 * r;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    cudaError_t result = cudaErrorNotSupported;
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    const uint64_t ws_bytes = lt_ws ? lt_ws_bytes : 0;
    cublasLtMatmulHeuristicResult_t heur;
    int found = 0;
    if (api.desc_create(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) goto done;
    if (api.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta) != CUBLAS_STATUS_SUCCESS ||
        api.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb) != CUBLAS_STATUS_SUCCESS)
        goto done;
    if (api.layout_create(&la, CUDA_R_16BF, (uint64_t)d, (uint64_t)N, ldw) != CUBLAS_STATUS_SUCCESS ||
        api.layout_create(&lb, CUDA_R_16BF, (uint64_t)d, (uint64_t)M, d) != CUBLAS_STATUS_SUCCESS ||
        api.layout_create(&lc, CUDA_R_32F, (uint64_t)N, (uint64_t)M, N) != CUBLAS_STATUS_SUCCESS)
        goto done;
    if (api.pref_create(&pref) != CUBLAS_STATUS_SUCCESS ||
        api.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof ws_bytes) !=
            CUBLAS_STATUS_SUCCESS)
        goto done;
    if (api.heuristic(handle, op, la, lb, lc, lc, pref, 1, &heur, &found) != CUBLAS_STATUS_SUCCESS || found < 1)
        goto done;
    {
        const float one = 1.0f, zero = 0.0f;
        result = api.matmul(handle, op, &one, A, la, h, lb, &zero, Hpre, lc, Hpre, lc, &heur.algo, lt_ws, ws_bytes,
                            s) == CUBLAS_STATUS_SUCCESS
                     ? cudaSuccess
                     : cudaErrorLaunchFailure;
    }
done:
    if (pref) api.pref_destroy(pref);
    if (lc) api.layout_destroy(lc);
    if (lb) api.layout_destroy(lb);
    if (la) api.layout_destroy(la);
    if (op) api.desc_destroy(op);
    return result;
}

}  // namespace dspark
