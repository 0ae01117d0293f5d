// sched.cu -- hardware-aware prefix scheduler and flattened-batch tags.
//
// DSpark digest, Module E and Algorithm 1: a_{r,j} = prod_{i<=j} c_{r,i}; the
// pool E = {(r,j): a_{r,j} > 0} sorted by a descending; admit greedily while
// Theta = tau * SPS(B) improves (break at the first non-improvement).  The
// production section replaces the break by a top-K of the current order with K
// taken from the confidences of two cycles earlier.
//
// One CTA does the whole decision (the pool holds at most 8192 entries):
//   1. fp32 running products a (IEEE products, identical to any CPU);
//   2. 64-bit keys (~bits(a) << 32 | flat index): ascending key order is a
//      descending with ties broken by (request, position); bitonic sort in
//      shared memory;
//   3. tau as an exact integer prefix sum in 2^-32 units;
//   4. Theta(m) = (tau_m 2^-32) * SPS(R + m) for every prefix m in parallel;
//      the synchronous stop is the first m with Theta(m) <= Theta(m-1), the
//      capacity for cycle t+2 is argmax_m Theta(m) (smallest m on ties);
//   5. l_r = largest admitted position of request r.
#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kSchedThreads = 1024;
constexpr unsigned long long kOutKey = 0xFFFFFFFFull << 32;

__device__ __forceinline__ double theta_at(long long units, const double *sps, int B_min, int B) {
    return __dmul_rn((double)units * (1.0 / 4294967296.0), sps[B - B_min]);
}

// inclusive block scan of one long long per thread (1024 threads)
__device__ long long block_inclusive_scan(long long v, long long *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        long long t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long o = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += o;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const long long prefix = warp > 0 ? warp_tot[warp - 1] : 0;
    __syncthreads();
    return v + prefix;
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const dspark_sched_args a, int npad) {
    extern __shared__ unsigned long long sched_smem[];
    unsigned long long *keys = sched_smem;                         // [npad]
    long long *units = reinterpret_cast<long long *>(keys + npad);  // [npad + 1]
    int *ell_s = reinterpret_cast<int *>(units + npad + 1);         // [R]
    __shared__ long long warp_tot[32];
    __shared__ int s_bad, s_pool, s_first;
    __shared__ double s_th[32];
    __shared__ int s_arg[32];

    const int R = a.R, G = a.gamma, n = R * G, tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) {
        s_bad = 0;
        s_pool = n;
        s_first = 0x7fffffff;
    }
    __syncthreads();

    // 1. prefix survival products (Algorithm 1, line 1) and sort keys (line 2)
    for (int rq = tid; rq < R; rq += nt) {
        float prod = 1.0f;
        bool bad = false;
        for (int j = 0; j < G; ++j) {
            const int e = rq * G + j;
            const float cc = a.c[e];
            if (!(cc >= 0.0f && cc <= 1.0f)) bad = true;
            prod = __fmul_rn(prod, cc);
            if (a.a) a.a[e] = prod;
            keys[e] = prod > 0.0f ? ((unsigned long long)(~__float_as_uint(prod)) << 32) | (unsigned)e
                                  : kOutKey | (unsigned)e;
        }
        ell_s[rq] = 0;
        if (bad) atomicExch(&s_bad, 1);
    }
    for (int e = n + tid; e < npad; e += nt) keys[e] = ~0ull;
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            set_err(a.err, DSPARK_ERR_RANGE);
            *a.K_out = 0;
            *a.theta_best = 0.0;
        }
        for (int rq = tid; rq < R; rq += nt) a.ell[rq] = 0;
        return;
    }

    // 2. bitonic sort, ascending keys
    for (int k = 2; k <= npad; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npad; i += nt) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = keys[i], y = keys[ixj];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) {
                        keys[i] = y;
                        keys[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < npad; i += nt)
        if (keys[i] >= kOutKey && (i == 0 || keys[i - 1] < kOutKey)) s_pool = i;
    __syncthreads();
    const int pool = min(s_pool, n);

    // 3. tau in 2^-32 units: exact integer prefix sums of round(a * 2^32)
    const int chunk = (npad + nt - 1) / nt;
    const int i0 = min(tid * chunk, npad), i1 = min(i0 + chunk, npad);
    long long local = 0;
    for (int i = i0; i < i1; ++i) {
        if (i < pool) {
            const float av = __uint_as_float(~(unsigned)(keys[i] >> 32));
            local += __float2ll_rn(__fmul_rn(av, 4294967296.0f));
        }
    }
    const long long base = ((long long)R << 32);
    long long run = block_inclusive_scan(local, warp_tot) - local + base;
    if (tid == 0) units[0] = base;
    for (int i = i0; i < i1; ++i) {
        if (i < pool) {
            const float av = __uint_as_float(~(unsigned)(keys[i] >> 32));
            run += __float2ll_rn(__fmul_rn(av, 4294967296.0f));
        }
        units[i + 1] = run;
    }
    __syncthreads();

    // 4. Theta along the sorted pool
    double best_th = -1.0;
    int best_m = 0x7fffffff;
    int first = 0x7fffffff;
    for (int m = tid; m <= pool; m += nt) {
        const double th = theta_at(units[m], a.sps, a.B_min, R + m);
        if (th > best_th) {  // m increases within a thread: keeps the smallest m on ties
            best_th = th;
            best_m = m;
        }
        if (m >= 1 && first == 0x7fffffff) {
            const double prev = theta_at(units[m - 1], a.sps, a.B_min, R + m - 1);
            if (th <= prev) first = m;
        }
    }
    if (first != 0x7fffffff) atomicMin(&s_first, first);
    // argmax over threads: larger Theta, then smaller m
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const double th2 = __shfl_xor_sync(0xffffffffu, best_th, off);
        const int m2 = __shfl_xor_sync(0xffffffffu, best_m, off);
        if (th2 > best_th || (th2 == best_th && m2 < best_m)) {
            best_th = th2;
            best_m = m2;
        }
    }
    if ((tid & 31) == 0) {
        s_th[tid >> 5] = best_th;
        s_arg[tid >> 5] = best_m;
    }
    __syncthreads();
    if (tid < 32) {
        best_th = tid < (nt >> 5) ? s_th[tid] : -1.0;
        best_m = tid < (nt >> 5) ? s_arg[tid] : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double th2 = __shfl_xor_sync(0xffffffffu, best_th, off);
            const int m2 = __shfl_xor_sync(0xffffffffu, best_m, off);
            if (th2 > best_th || (th2 == best_th && m2 < best_m)) {
                best_th = th2;
                best_m = m2;
            }
        }
        if (tid == 0) s_arg[0] = best_m;
    }
    __syncthreads();
    const int K_cap = s_arg[0];
    int count = s_first == 0x7fffffff ? pool : s_first - 1;
    if (a.mode == DSPARK_SCHED_ASYNC && a.K_in != nullptr) {
        const int K = *a.K_in;
        if (K >= 0) count = min(K, pool);
    }

    // 5. verify lengths: l_r <- j for every admitted (r, j)
    for (int i = tid; i < count; i += nt) {
        const unsigned e = (unsigned)(keys[i] & 0xFFFFFFFFull);
        atomicMax(&ell_s[e / G], (int)(e % G) + 1);
    }
    __syncthreads();
    for (int rq = tid; rq < R; rq += nt) a.ell[rq] = ell_s[rq];
    if (tid == 0) {
        *a.K_out = K_cap;
        *a.theta_best = theta_at(units[count], a.sps, a.B_min, R + count);
    }
}

// ----- flattened batch tags: rows (r, 0..l_r) in request order -----------------
__global__ void __launch_bounds__(1024) build_tags_kernel(int R, int gamma, const int32_t *ell,
                                                          int32_t *tags, int32_t *N_out,
                                                          int32_t *err) {
    __shared__ long long warp_tot[32];
    const int nt = blockDim.x, tid = threadIdx.x;
    const int chunk = (R + nt - 1) / nt;
    const int r0 = min(tid * chunk, R), r1 = min(r0 + chunk, R);
    long long local = 0;
    for (int rq = r0; rq < r1; ++rq) {
        int l = ell[rq];
        if (l < 0 || l > gamma) {
            set_err(err, DSPARK_ERR_RANGE);
            l = 0;
        }
        local += 1 + l;
    }
    long long off = block_inclusive_scan(local, warp_tot) - local;
    for (int rq = r0; rq < r1; ++rq) {
        int l = ell[rq];
        if (l < 0 || l > gamma) l = 0;
        for (int j = 0; j <= l; ++j) {
            tags[2 * (off + j)] = rq;
            tags[2 * (off + j) + 1] = j;
        }
        off += 1 + l;
    }
    if (r1 == R && r0 < r1) *N_out = (int32_t)off;
    if (R == 0 && tid == 0) *N_out = 0;
}

}  // namespace

size_t schedule_smem_bytes(int R, int gamma) {
    int n = R * gamma, npad = 1;
    while (npad < n) npad <<= 1;
    return sizeof(unsigned long long) * (size_t)npad + sizeof(long long) * (size_t)(npad + 1) +
           sizeof(int) * (size_t)R;
}

cudaError_t launch_schedule(const dspark_sched_args &a, cudaStream_t s) {
    int n = a.R * a.gamma, npad = 1;
    while (npad < n) npad <<= 1;
    const size_t smem = schedule_smem_bytes(a.R, a.gamma);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    schedule_kernel<<<1, kSchedThreads, smem, s>>>(a, npad);
    return cudaGetLastError();
}

cudaError_t launch_build_tags(int R, int gamma, const int32_t *ell, int32_t *tags, int32_t *N_out,
                              int32_t *err, cudaStream_t s) {
    build_tags_kernel<<<1, 1024, 0, s>>>(R, gamma, ell, tags, N_out, err);
    return cudaGetLastError();
}

}  // namespace dspark
