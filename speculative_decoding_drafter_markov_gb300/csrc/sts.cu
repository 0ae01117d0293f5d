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
// One cooperative launch runs all positions.  Block (x, y) owns 64 grid points
// (y) and the sample tiles x, x + gridDim.x, ... of 256 samples.  At position k
// a tile is staged in shared memory as (P_{k-1} n_bins, -s_k log2 e, y_k);
// P_{k-1} = P_{k-2} sigma(s_{k-1} / T_{k-1}) comes from a prefix buffer written
// at position k - 1 (ping-pong by parity).  Thread (q, j) scores slice q (64
// samples) of the tile at grid point j and adds P - y to its own row of per-bin
// sums.  One fused multiply-add forms 128 + P n_bins, whose bits hold
// u = round(P n_bins 2^16) (the binade [128, 256) has a spacing of 2^-16).  The
// bin is u >> 16.  The sums are integers in units of 2^-16 / n_bins of P, so
// the additions are exact and their order does not matter.  The rounding can
// move a P within 2^-17 / n_bins below a bin edge into the next bin.  P = 1
// lands in a spare row n_bins, folded into bin n_bins - 1.  After each tile the
// four slices are summed into the block's 64-bit totals, which go into the
// position's global [n_bins, G] table with 64-bit atomics.  A grid barrier
// follows, a counter with a bounded wait (the launch is cooperative, so all
// blocks are resident).  Then every block reads the table, which is cached in
// L1 and so read from L2 about once per SM, and takes the same smallest
// sum_b |D_b| (lowest grid index on ties) as T_k.  Block (0, 0) writes T_k, its
// ECE and the curve.
#include <float.h>
#include <limits.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kStsThreads = 256;
constexpr int kStsPoints = 64;                          // grid points per block
constexpr int kStsSlices = kStsThreads / kStsPoints;    // sample slices per grid point
constexpr int kStsTile = 256;                           // samples per tile
constexpr int kStsSlice = kStsTile / kStsSlices;        // samples per slice
constexpr int kFixBits = 16;          // P n_bins in units of 2^-16
constexpr float kMagic = 128.0f;       // 128 + P n_bins (n_bins <= 64) keeps the 2^-16 spacing
constexpr int kMagicBits = 0x43000000; // bits of 128.0f (low 16 bits zero)

struct StsParams {
    int M, gamma, G, n_bins;
    const float *logit;       // [M, gamma]
    const int32_t *n_acc;     // [M]
    const float *grid;        // [G]
    float *T;                 // [gamma]
    double *ece;              // [gamma]
    double *curve;            // [gamma, G] or null
    long long *D;             // [gamma, n_bins, G] sums of P - y, units of 2^-16 / n_bins
    unsigned int *barrier;    // [gamma] blocks arrived after position k
    float *pre[2];            // [M] prefix products, ping-pong by position parity
    int32_t *err;
};

// 1 / (1 + e^{-x}): e^{-x} through MUFU ex2, the reciprocal through the fast
// divide; saturates to exactly 0 and 1 for |x| large (no NaN for x = +-inf).
__device__ __forceinline__ float sigmoid_fast(float x) {
    return __fdividef(1.0f, 1.0f + ex2(-x * kLog2e));
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/T, capped so that a subnormal T gives a huge finite factor (0 * 1/T stays 0)
__device__ __forceinline__ float inv_temperature(float T) { return fminf(1.0f / T, FLT_MAX); }

__device__ __forceinline__ bool valid_temperature(float T) { return T > 0.0f && T <= FLT_MAX; }

// ECE = sum / (2^16 n_bins M)
__device__ __forceinline__ double ece_units(const StsParams &p) {
    return (double)(1 << kFixBits) * (double)p.n_bins * (double)p.M;
}

// grid barrier: every block arrives once per position; bounded wait, false on timeout
__device__ __forceinline__ bool grid_arrive_wait(unsigned int *ctr, unsigned int nblocks, int32_t *err) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t t0 = tc::globaltimer_ns();
    for (;;) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= nblocks) break;
        if (tc::globaltimer_ns() - t0 > tc::kWaitLimitNs) {
            set_err(err, DSPARK_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
    __threadfence();
    return true;
}

__global__ void __launch_bounds__(kStsThreads, 6) sts_fit_kernel(const StsParams p) {
    extern __shared__ __align__(16) unsigned char sts_smem[];
    float4 *tile = reinterpret_cast<float4 *>(sts_smem);                            // [kStsTile]
    long long *acc = reinterpret_cast<long long *>(tile + kStsTile);                // [n_bins][kStsPoints]
    int *hist = reinterpret_cast<int *>(acc + (size_t)p.n_bins * kStsPoints);       // [n_bins + 1][kStsThreads]
    __shared__ unsigned long long s_v[kStsThreads / 32];
    __shared__ int s_g[kStsThreads / 32];
    __shared__ int s_best;
    __shared__ bool s_ok;

    const int tid = threadIdx.x;
    const int q = tid / kStsPoints;
    const int g = blockIdx.y * kStsPoints + tid % kStsPoints;
    const int nb = p.n_bins;
    const unsigned int nblocks = gridDim.x * gridDim.y;
    const bool lead = blockIdx.x == 0 && blockIdx.y == 0;
    const bool write_prefix = blockIdx.y == 0;
    for (int b = 0; b <= nb; ++b) hist[b * kStsThreads + tid] = 0;

    bool live = g < p.G;
    float inv_T = 1.0f;
    if (live) {
        const float T = p.grid[g];
        live = valid_temperature(T);
        if (!live) {
            if (q == 0 && blockIdx.x == 0) set_err(p.err, DSPARK_ERR_INVAL);
        } else {
            inv_T = inv_temperature(T);
        }
    }
    float inv_T_prev = 1.0f;  // 1 / T_{k-1}

    for (int k = 1; k <= p.gamma; ++k) {
        for (int i = tid; i < nb * kStsPoints; i += kStsThreads) acc[i] = 0;
        const float *pre_in = (k & 1) ? p.pre[1] : p.pre[0];   // P_{k-2}, written at position k - 1
        float *pre_out = (k & 1) ? p.pre[0] : p.pre[1];        // P_{k-1}
        // M < 2^31, so tile starts and sample indices stay below 2^32
        for (unsigned t0 = blockIdx.x * kStsTile; t0 < (unsigned)p.M; t0 += gridDim.x * kStsTile) {
            // stage (P_{k-1} n_bins, -s_k log2 e, bits of 128 + y_k n_bins) of the tile's samples
            const unsigned m = t0 + tid;
            if (m < (unsigned)p.M) {
                const float *row = p.logit + (size_t)m * p.gamma;
                float prefix = 1.0f;
                if (k >= 2) {
                    float sp = row[k - 2];
                    if (sp != sp) sp = 0.0f;  // reported at position k - 1
                    prefix = pre_in[m] * sigmoid_fast(sp * inv_T_prev);
                }
                if (write_prefix) pre_out[m] = prefix;
                float s = row[k - 1];
                if (s != s) {
                    if (blockIdx.y == 0) set_err(p.err, DSPARK_ERR_NONFINITE);
                    s = 0.0f;
                }
                int n = p.n_acc[m];
                if (n < 0 || n > p.gamma) {
                    if (blockIdx.y == 0) set_err(p.err, DSPARK_ERR_RANGE);
                    n = n < 0 ? 0 : p.gamma;
                }
                const int y_bits = kMagicBits + (n >= k ? nb << kFixBits : 0);
                tile[tid] = make_float4(prefix * (float)nb, -s * kLog2e, __int_as_float(y_bits), 0.0f);
            }
            __syncthreads();
            if (live) {
                const int j0 = q * kStsSlice;
                const int j1 = min(j0 + kStsSlice, (int)((unsigned)p.M - t0));
#pragma unroll 4
                for (int j = j0; j < j1; ++j) {
                    const float4 e = tile[j];  // the same address for the whole warp: a broadcast
                    // bits of 128 + P n_bins, P = P_{k-1} sigma(s_k / T) in [0, 1]: the row
                    // (u >> 16) - 0x4300 lies in 0..n_bins
                    const int u = __float_as_int(fmaf(e.x, rcp_approx(1.0f + ex2(e.y * inv_T)), kMagic));
                    hist[((u >> kFixBits) - (kMagicBits >> kFixBits)) * kStsThreads + tid] += u - __float_as_int(e.z);
                }
            }
            __syncthreads();
            // fold the four slices (and the spare row of P = 1 into the last bin) into
            // the block's totals; one sample adds at most 2^22 + 1 in magnitude and a
            // thread sees 64 samples per tile, so a fold of four threads' rows stays
            // below 2^31
            for (int i = tid; i < nb * kStsPoints; i += kStsThreads) {
                const int b = i / kStsPoints, j = i % kStsPoints;
                int *hb = hist + b * kStsThreads + j;
                int sum = 0;
#pragma unroll
                for (int sl = 0; sl < kStsSlices; ++sl) {
                    sum += hb[sl * kStsPoints];
                    hb[sl * kStsPoints] = 0;
                }
                if (b == nb - 1) {
#pragma unroll
                    for (int sl = 0; sl < kStsSlices; ++sl) {
                        sum += hb[kStsThreads + sl * kStsPoints];
                        hb[kStsThreads + sl * kStsPoints] = 0;
                    }
                }
                acc[i] += sum;
            }
            __syncthreads();
        }

        // this block's totals into the position's table, then the grid barrier
        long long *Dk = p.D + (size_t)(k - 1) * nb * p.G;
        for (int i = tid; i < nb * kStsPoints; i += kStsThreads) {
            const int gg = blockIdx.y * kStsPoints + i % kStsPoints;
            const long long v = acc[i];
            if (gg < p.G && v != 0)
                atomicAdd(reinterpret_cast<unsigned long long *>(Dk + (size_t)(i / kStsPoints) * p.G + gg),
                          static_cast<unsigned long long>(v));
        }
        __syncthreads();
        if (tid == 0) s_ok = grid_arrive_wait(p.barrier + (k - 1), nblocks, p.err);
        __syncthreads();
        if (!s_ok) return;

        // every block: the ECE of every grid point and the smallest (lowest index on ties)
        unsigned long long best_v = ULLONG_MAX;
        int best_g = INT_MAX;
        for (int gg = tid; gg < p.G; gg += kStsThreads) {
            unsigned long long tot = ULLONG_MAX;
            if (valid_temperature(p.grid[gg])) {
                tot = 0;
                for (int b = 0; b < nb; ++b) {
                    const long long v = Dk[(size_t)b * p.G + gg];  // first read of this table on this SM
                    tot += (unsigned long long)(v < 0 ? -v : v);
                }
            }
            if (lead && p.curve)
                p.curve[(size_t)(k - 1) * p.G + gg] =
                    tot == ULLONG_MAX ? __longlong_as_double(0x7ff8000000000000ll) : (double)tot / ece_units(p);
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
            s_best = best_g;
            if (lead) {
                if (best_g == INT_MAX) {  // no valid grid point
                    set_err(p.err, DSPARK_ERR_INVAL);
                    p.T[k - 1] = 1.0f;
                    p.ece[k - 1] = __longlong_as_double(0x7ff8000000000000ll);
                } else {
                    p.T[k - 1] = p.grid[best_g];
                    p.ece[k - 1] = (double)best_v / ece_units(p);
                }
            }
        }
        __syncthreads();
        inv_T_prev = s_best == INT_MAX ? 1.0f : inv_temperature(p.grid[s_best]);
    }
}

size_t sts_smem_bytes(int n_bins) {
    return kStsTile * sizeof(float4) + (size_t)n_bins * kStsPoints * sizeof(long long) +
           (size_t)(n_bins + 1) * kStsThreads * sizeof(int);
}

size_t table_bytes(int gamma, int G, int n_bins) {
    return align256(sizeof(long long) * (size_t)gamma * G * n_bins);
}

size_t barrier_bytes(int gamma) { return align256(sizeof(unsigned) * (size_t)gamma); }

}  // namespace

size_t sts_ws_bytes(int M, int gamma, int G, int n_bins) {
    return table_bytes(gamma, G, n_bins) + barrier_bytes(gamma) + 2 * align256(sizeof(float) * (size_t)M);
}

bool sts_grid_shape(int M, int G, int n_bins, int *gx, int *gy) {
    const size_t smem = sts_smem_bytes(n_bins);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(sts_fit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sts_fit_kernel, kStsThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return false;
    const long long resident = (long long)sm_count() * per_sm;
    *gy = (G + kStsPoints - 1) / kStsPoints;
    if (*gy > resident) return false;
    // equal tiles per block: the fewest rounds over the columns that fit
    const long long tiles = ((long long)M + kStsTile - 1) / kStsTile;
    const long long cols = resident / *gy;
    const long long rounds = (tiles + cols - 1) / cols;
    *gx = (int)((tiles + rounds - 1) / rounds);
    return true;
}

cudaError_t launch_sts_fit(const StsFit &f, void *ws, cudaStream_t s) {
    char *base = static_cast<char *>(ws);
    const size_t d_bytes = table_bytes(f.gamma, f.G, f.n_bins);
    const size_t pre_bytes = align256(sizeof(float) * (size_t)f.M);
    // the bin sums and the barrier counters start at zero; the prefix buffers need no init
    cudaError_t e = cudaMemsetAsync(base, 0, d_bytes + barrier_bytes(f.gamma), s);
    if (e != cudaSuccess) return e;
    int gx = 0, gy = 0;
    if (!sts_grid_shape(f.M, f.G, f.n_bins, &gx, &gy)) return cudaErrorInvalidConfiguration;
    StsParams p{};
    p.M = f.M; p.gamma = f.gamma; p.G = f.G; p.n_bins = f.n_bins;
    p.logit = f.logit; p.n_acc = f.n_accept; p.grid = f.grid;
    p.T = f.T; p.ece = f.ece; p.curve = f.curve; p.err = f.err;
    p.D = reinterpret_cast<long long *>(base);
    p.barrier = reinterpret_cast<unsigned int *>(base + d_bytes);
    p.pre[0] = reinterpret_cast<float *>(base + d_bytes + barrier_bytes(f.gamma));
    p.pre[1] = reinterpret_cast<float *>(base + d_bytes + barrier_bytes(f.gamma) + pre_bytes);
    void *args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(sts_fit_kernel), dim3(gx, gy),
                                       dim3(kStsThreads), args, sts_smem_bytes(f.n_bins), s);
}

}  // namespace dspark
