// sts.cu -- sequential temperature scaling of the confidences (DSpark digest,
// Module D).  c_i is the probability that position i is accepted given that the
// positions before it were, so the probability that the first k drafted tokens
// are all accepted is P_k = prod_{i<=k} sigma(s_i / T_i).  For k = 1..gamma in
// order, T_k is the grid temperature whose P_k has the smallest expected
// calibration error against the held-out outcome y_k = 1[n >= k], with
// T_1..T_{k-1} already fixed:
//   ECE = sum_b (|b| / M) |mean_b P - mean_b y| = (1/M) sum_b |sum_{m in b} (P_m - y_m)|,
// bins b = min(floor(P n_bins), n_bins - 1) of width 1/n_bins.
//
// One launch per position k.  Block (x, y) owns grid points y*256 .. y*256+255,
// one per thread, and the sample tiles x, x + gridDim.x, ...  A tile of 256
// samples is staged in shared memory as (P_{k-1}, s_k, y_k).  Every thread then
// scores the whole tile at its own temperature and adds P - y to its own row
// of per-bin sums in shared memory.  The sums are fixed point (units of 2^-31)
// with exact integer additions, so the result does not depend on the order of
// the additions.  At the end the block adds its rows to the position's global
// [G, n_bins] table with 64-bit atomics.  The last block to finish (a ticket
// counter, no waiting) reduces sum_b |D_b| per grid point, takes the smallest
// (lowest grid index on ties) and writes T_k, its ECE and the ECE curve.  The
// next launch reads T_1..T_k from device memory.
#include <float.h>
#include <limits.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kStsThreads = 256;  // grid points per block
constexpr int kStsTile = 256;     // samples staged per pass
constexpr float kFixScale = 2147483648.0f;  // 2^31 fixed-point units per 1.0
constexpr long long kFixOne = 1ll << 31;

struct StsParams {
    int M, gamma, G, n_bins, k;
    const float *logit;       // [M, gamma]
    const int32_t *n_acc;     // [M]
    const float *grid;        // [G]
    float *T;                 // [gamma]; T[0 .. k-2] fitted by the earlier launches
    double *ece;              // [gamma]
    double *curve;            // [gamma, G] or null
    long long *D;             // [gamma, G, n_bins] fixed-point sums of P - y
    unsigned int *tickets;    // [gamma] blocks finished per position
    int32_t *err;
};

// 1 / (1 + e^{-x}): e^{-x} through MUFU ex2, the reciprocal through the fast
// divide; saturates to exactly 0 and 1 for |x| large (no NaN for x = +-inf).
__device__ __forceinline__ float sigmoid_fast(float x) {
    return __fdividef(1.0f, 1.0f + ex2(-x * kLog2e));
}

// 1/T, capped so that a subnormal T gives a huge finite factor (0 * 1/T stays 0)
__device__ __forceinline__ float inv_temperature(float T) { return fminf(1.0f / T, FLT_MAX); }

__device__ __forceinline__ bool valid_temperature(float T) { return T > 0.0f && T <= FLT_MAX; }

__global__ void __launch_bounds__(kStsThreads) sts_position_kernel(const StsParams p) {
    extern __shared__ __align__(16) unsigned char sts_smem[];
    long long *hist = reinterpret_cast<long long *>(sts_smem);  // [n_bins][kStsThreads]
    float4 *tile = reinterpret_cast<float4 *>(hist + (size_t)p.n_bins * kStsThreads);
    __shared__ float s_inv_prev[kStsMaxGamma];  // 1 / T_i of the fitted positions i < k
    __shared__ bool s_last;

    const int tid = threadIdx.x;
    const int g = blockIdx.y * kStsThreads + tid;
    const int k = p.k;
    for (int i = tid; i < k - 1; i += kStsThreads) s_inv_prev[i] = inv_temperature(p.T[i]);
    for (int b = 0; b < p.n_bins; ++b) hist[b * kStsThreads + tid] = 0;

    bool live = g < p.G;
    float inv_T = 1.0f;
    if (live) {
        const float T = p.grid[g];
        if (!valid_temperature(T)) {
            set_err(p.err, DSPARK_ERR_INVAL);
            live = false;
        } else {
            inv_T = inv_temperature(T);
        }
    }
    const float nb_f = (float)p.n_bins;
    const int nb_max = p.n_bins - 1;
    __syncthreads();

    for (long long t0 = (long long)blockIdx.x * kStsTile; t0 < p.M; t0 += (long long)gridDim.x * kStsTile) {
        // stage (P_{k-1}, s_k, y_k) of the tile's samples
        const long long m = t0 + tid;
        if (m < p.M) {
            const float *row = p.logit + m * p.gamma;
            float prefix = 1.0f;
            for (int i = 0; i < k - 1; ++i) {
                float s = row[i];
                if (s != s) s = 0.0f;  // reported when position i + 1 was fitted
                prefix *= sigmoid_fast(s * s_inv_prev[i]);
            }
            float s = row[k - 1];
            if (s != s) {
                set_err(p.err, DSPARK_ERR_NONFINITE);
                s = 0.0f;
            }
            int n = p.n_acc[m];
            if (n < 0 || n > p.gamma) {
                set_err(p.err, DSPARK_ERR_RANGE);
                n = n < 0 ? 0 : p.gamma;
            }
            tile[tid] = make_float4(prefix, s, n >= k ? 1.0f : 0.0f, 0.0f);
        }
        __syncthreads();
        const int cnt = (int)min((long long)kStsTile, p.M - t0);
        if (live) {
            for (int j = 0; j < cnt; ++j) {
                const float4 e = tile[j];  // the same address for every lane: a broadcast
                const float P = e.x * sigmoid_fast(e.y * inv_T);
                const int b = min((int)(P * nb_f), nb_max);
                const long long d = (long long)__float2uint_rn(P * kFixScale) - (e.z != 0.0f ? kFixOne : 0ll);
                hist[b * kStsThreads + tid] += d;
            }
        }
        __syncthreads();
    }

    // this block's sums into the position's table
    long long *Dk = p.D + (size_t)(k - 1) * p.G * p.n_bins;
    if (live) {
        for (int b = 0; b < p.n_bins; ++b) {
            const long long v = hist[b * kStsThreads + tid];
            if (v != 0)
                atomicAdd(reinterpret_cast<unsigned long long *>(Dk + (size_t)g * p.n_bins + b),
                          static_cast<unsigned long long>(v));
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(p.tickets + (k - 1), 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // last block: ECE of every grid point, then the smallest (lowest index on ties)
    const double ece_units = (double)kFixScale * (double)p.M;  // ECE = sum / (2^31 M)
    unsigned long long best_v = ULLONG_MAX;
    int best_g = INT_MAX;
    for (int gg = tid; gg < p.G; gg += kStsThreads) {
        unsigned long long tot = ULLONG_MAX;
        if (valid_temperature(p.grid[gg])) {
            tot = 0;
            for (int b = 0; b < p.n_bins; ++b) {
                const long long v = __ldcg(Dk + (size_t)gg * p.n_bins + b);
                tot += (unsigned long long)(v < 0 ? -v : v);
            }
        }
        if (p.curve)
            p.curve[(size_t)(k - 1) * p.G + gg] =
                tot == ULLONG_MAX ? __longlong_as_double(0x7ff8000000000000ll) : (double)tot / ece_units;
        if (tot < best_v) {  // gg rises within a thread, so ties keep the lowest index
            best_v = tot;
            best_g = gg;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long ov = __shfl_xor_sync(0xffffffffu, best_v, off);
        const int og = __shfl_xor_sync(0xffffffffu, best_g, off);
        if (ov < best_v || (ov == best_v && og < best_g)) {
            best_v = ov;
            best_g = og;
        }
    }
    __shared__ unsigned long long s_v[kStsThreads / 32];
    __shared__ int s_g[kStsThreads / 32];
    if ((tid & 31) == 0) {
        s_v[tid >> 5] = best_v;
        s_g[tid >> 5] = best_g;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kStsThreads / 32; ++w)
            if (s_v[w] < best_v || (s_v[w] == best_v && s_g[w] < best_g)) {
                best_v = s_v[w];
                best_g = s_g[w];
            }
        if (best_g == INT_MAX) {  // no valid grid point
            set_err(p.err, DSPARK_ERR_INVAL);
            p.T[k - 1] = 1.0f;
            p.ece[k - 1] = __longlong_as_double(0x7ff8000000000000ll);
        } else {
            p.T[k - 1] = p.grid[best_g];
            p.ece[k - 1] = (double)best_v / ece_units;
        }
    }
}

size_t sts_smem_bytes(int n_bins) {
    return (size_t)n_bins * kStsThreads * sizeof(long long) + kStsTile * sizeof(float4);
}

}  // namespace

size_t sts_ws_bytes(int gamma, int G, int n_bins) {
    return align256(sizeof(long long) * (size_t)gamma * G * n_bins) + align256(sizeof(unsigned) * gamma);
}

cudaError_t launch_sts_fit(const StsFit &f, void *ws, cudaStream_t s) {
    char *base = static_cast<char *>(ws);
    const size_t d_bytes = align256(sizeof(long long) * (size_t)f.gamma * f.G * f.n_bins);
    cudaError_t e = cudaMemsetAsync(base, 0, sts_ws_bytes(f.gamma, f.G, f.n_bins), s);
    if (e != cudaSuccess) return e;
    const size_t smem = sts_smem_bytes(f.n_bins);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(sts_position_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sts_position_kernel, kStsThreads, smem);
    if (e != cudaSuccess) return e;
    const int gy = (f.G + kStsThreads - 1) / kStsThreads;
    const long long tiles = ((long long)f.M + kStsTile - 1) / kStsTile;
    const long long want = std::max(1, sm_count() * std::max(per_sm, 1) / gy);
    const int gx = (int)std::min(tiles, want);

    StsParams p{};
    p.M = f.M; p.gamma = f.gamma; p.G = f.G; p.n_bins = f.n_bins;
    p.logit = f.logit; p.n_acc = f.n_accept; p.grid = f.grid;
    p.T = f.T; p.ece = f.ece; p.curve = f.curve; p.err = f.err;
    p.D = reinterpret_cast<long long *>(base);
    p.tickets = reinterpret_cast<unsigned int *>(base + d_bytes);
    for (int k = 1; k <= f.gamma; ++k) {
        p.k = k;
        sts_position_kernel<<<dim3(gx, gy), kStsThreads, smem, s>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
