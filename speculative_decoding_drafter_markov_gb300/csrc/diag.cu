// diag.cu -- acceptance diagnostics of the verification outcomes.
//
// DSpark digest, analysis 1: the per-position conditional acceptance rate
// counts, at position k, only the instances whose positions 1..k-1 were all
// accepted; the offline results report the acceptance length tau = n + 1 (the
// accepted drafted tokens and the target's own token).  One small launch adds a
// cycle's counts into the caller's device counters: per-block histograms in
// shared memory, then one global atomic per non-zero bin.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

__global__ void __launch_bounds__(256) accept_stats_kernel(const dspark_accept_stats_args a) {
    extern __shared__ unsigned long long sh[];
    const int g = a.gamma;
    unsigned long long *reached = sh, *accepted = sh + g, *tau = sh + 2 * g, *ellh = sh + 3 * g + 1;
    const int nbins = 4 * g + 2;
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) sh[i] = 0ull;
    __syncthreads();
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < a.R; r += gridDim.x * blockDim.x) {
        const int l = a.ell ? a.ell[r] : g;
        if (l < 0) continue;  // not verified this cycle
        const int n = a.n_accept[r];
        if (n < 0 || n > l || l > g) {
            set_err(a.err, DSPARK_ERR_RANGE);
            continue;
        }
        // position k was tested with its prefix accepted for k <= min(l, n + 1),
        // and passed for k <= n
        const int kr = min(l, n + 1);
        for (int k = 0; k < kr; ++k) atomicAdd(&reached[k], 1ull);
        for (int k = 0; k < n; ++k) atomicAdd(&accepted[k], 1ull);
        atomicAdd(&tau[n], 1ull);
        atomicAdd(&ellh[l], 1ull);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) {
        const unsigned long long c = sh[i];
        if (c == 0ull) continue;
        if (i < g) atomicAdd(a.reached + i, c);
        else if (i < 2 * g) atomicAdd(a.accepted + (i - g), c);
        else if (i < 3 * g + 1) atomicAdd(a.tau_hist + (i - 2 * g), c);
        else if (a.ell_hist) atomicAdd(a.ell_hist + (i - 3 * g - 1), c);
    }
}

}  // namespace

cudaError_t launch_accept_stats(const dspark_accept_stats_args &a, cudaStream_t s) {
    const int threads = 256;
    int blocks = (a.R + threads - 1) / threads;
    if (blocks > 16) blocks = 16;  // a handful of blocks: few global atomics per bin
    const size_t smem = sizeof(unsigned long long) * (size_t)(4 * a.gamma + 2);
    accept_stats_kernel<<<blocks, threads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
