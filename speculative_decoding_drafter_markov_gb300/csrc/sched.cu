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
//   2. 30-bit sort keys 0x3F800000 - bits(a) (a in (0, 1]; 0x3FFFFFFF marks an
//      entry outside the pool): ascending key order is a descending, and a
//      stable sort of the entries in flat-index order breaks ties by
//      (request, position).  Stable LSD radix sort in shared memory, 5-bit
//      digits, 6 passes: each warp ranks its items with five ballots (the
//      lanes sharing a digit), one block-wide scan over the (digit, warp)
//      counts places them;
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

// round(a 2^32) to the nearest integer, ties to even, for a in [0, 1]: the
// value __float2ll_rn(a * 2^32) has, from the bits (a = m 2^(E - 150))
__device__ __forceinline__ long long units_of(float a) {
    const uint32_t b = __float_as_uint(a);
    const int e = (int)(b >> 23);
    const uint32_t m = e ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
    const int sh = (e ? e : 1) - 118;
    if (sh >= 0) return (long long)m << sh;
    const int s = -sh;
    if (s >= 25) return 0;  // m 2^-s < 1/2
    const uint32_t q = m >> s, rem = m & ((1u << s) - 1u), half = 1u << (s - 1);
    return (long long)(q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u));
}

// u 2^-32 as a double, exactly, for u in [2^32, 2^53)
__device__ __forceinline__ double scaled_units(long long u) {
    const int msb = 63 - __clzll(u);
    const unsigned long long mant = ((unsigned long long)u << (52 - msb)) & 0xFFFFFFFFFFFFFull;
    return __longlong_as_double((long long)(((unsigned long long)(msb + 1023 - 32) << 52) | mant));
}

// comparisons of Theta values held as fp64 bit patterns
__device__ __forceinline__ bool th_plain(long long x) { return x >= 0 && x < 0x7FF0000000000000ll; }
__device__ __forceinline__ bool th_gt(long long x, long long y) {
    if (th_plain(x) && th_plain(y)) return x > y;
    return __longlong_as_double(x) > __longlong_as_double(y);
}
__device__ __forceinline__ bool th_le(long long x, long long y) {
    if (th_plain(x) && th_plain(y)) return x <= y;
    return __longlong_as_double(x) <= __longlong_as_double(y);
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

constexpr uint32_t kOutKey30 = 0x3FFFFFFFu;  // sorts after every a in (0, 1]
constexpr int kRadixBits = 5, kRadixPasses = 6, kBins = 1 << kRadixBits;
constexpr int kHistLd = 33;  // (digit, warp) counts at d * 33 + w: no two digits share a bank

// inclusive block scan of one int per thread (1024 threads)
__device__ int block_inclusive_scan_int(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += o;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int prefix = warp > 0 ? warp_tot[warp - 1] : 0;
    __syncthreads();
    return v + prefix;
}

// Stable LSD radix sort of CAP = 1024 IPT words (sort key in bits 32..61, flat
// index below) from `src`, result back in `src` (an even number of passes).
// Warp w owns positions [32 IPT w, 32 IPT (w + 1)) of the current order, item i
// of lane l being position 32 IPT w + 32 i + l, so (warp, item, lane) order is
// sequence order and ranking the items in that order keeps the sort stable.
// the lanes of the warp whose kRadixBits-bit digit is d, from the warp's
// per-bit ballots
__device__ __forceinline__ unsigned digit_lanes(const unsigned (&vote)[kRadixBits], int d) {
    unsigned m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < kRadixBits; ++b) m &= ((d >> b) & 1) ? vote[b] : ~vote[b];
    return m;
}

template <int IPT>
__device__ void radix_sort_keys(unsigned long long *src, unsigned long long *dst, int *hist, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int pass = 0; pass < kRadixPasses; ++pass) {
        const int shift = 32 + kRadixBits * pass;
        unsigned long long v[IPT];
        int off[IPT];
#pragma unroll
        for (int i = 0; i < IPT; ++i) v[i] = src[32 * IPT * warp + 32 * i + lane];
        // lane x keeps the running count of digit x over this warp's items
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int d = (int)(v[i] >> shift) & (kBins - 1);
            unsigned vote[kRadixBits];
#pragma unroll
            for (int b = 0; b < kRadixBits; ++b) vote[b] = __ballot_sync(0xffffffffu, (d >> b) & 1);
            const unsigned peers = digit_lanes(vote, d);
            off[i] = __shfl_sync(0xffffffffu, cnt, d) + __popc(peers & lt_mask);
            cnt += __popc(digit_lanes(vote, lane));
        }
        hist[lane * kHistLd + warp] = cnt;
        __syncthreads();
        // exclusive scan over (digit, warp) in digit-major order: 32 bins x 32 warps
        const int hs = (tid >> 5) * kHistLd + (tid & 31);
        const int c = hist[hs];
        const int incl = block_inclusive_scan_int(c, warp_tot);
        hist[hs] = incl - c;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int d = (int)(v[i] >> shift) & (kBins - 1);
            dst[hist[d * kHistLd + warp] + off[i]] = v[i];
        }
        __syncthreads();
        unsigned long long *t = src;
        src = dst;
        dst = t;
    }
}

template <int IPT>
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const dspark_sched_args a) {
    constexpr int npad = kSchedThreads * IPT;
    extern __shared__ unsigned long long sched_smem[];
    unsigned long long *keys = sched_smem;                     // [npad] sorted entries
    unsigned long long *tmp = keys + npad;                     // [npad] radix ping-pong
    long long *units = reinterpret_cast<long long *>(tmp);     // [npad + 1] after the sort
    int *ell_s = reinterpret_cast<int *>(tmp + npad + 1);      // [R]
    __shared__ long long warp_tot[32];
    __shared__ int hist[kBins * kHistLd];
    __shared__ int s_bad, s_pool, s_first;
    __shared__ long long s_th[32];
    __shared__ int s_arg[32];

    const int R = a.R, G = a.gamma, n = R * G, tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) {
        s_bad = 0;
        s_pool = 0;
        s_first = 0x7fffffff;
    }
    __syncthreads();

    // 1. prefix survival products (Algorithm 1, line 1) and sort keys (line 2);
    //    the confidences are staged in shared memory with coalesced loads first
    float *c_s = reinterpret_cast<float *>(tmp);  // free until the sort
    {
        float cv[IPT];  // all of a thread's loads in flight together
#pragma unroll
        for (int q = 0; q < IPT; ++q) cv[q] = tid + q * nt < n ? a.c[tid + q * nt] : 0.f;
#pragma unroll
        for (int q = 0; q < IPT; ++q)
            if (tid + q * nt < n) c_s[tid + q * nt] = cv[q];
    }
    __syncthreads();
    // one thread per request: the running products a_{r,1..G} (left to right, the
    // rounding of Algorithm 1's products) in place of its confidences
    bool bad = false;
    for (int rq = tid; rq < R; rq += nt) {
        float *cr = c_s + rq * G;
        float prod = 1.0f;
        for (int j = 0; j < G; ++j) {
            const float cc = cr[j];
            if (!(cc >= 0.0f && cc <= 1.0f)) bad = true;
            prod = __fmul_rn(prod, cc);
            cr[j] = prod;
        }
    }
    __syncthreads();
    // one thread per entry (r, j): its sort key
    int in_pool = 0;
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
        const int e = tid + q * nt;
        if (e >= n) continue;
        const float prod = c_s[e];
        if (a.a) a.a[e] = prod;
        const uint32_t k30 = prod > 0.0f ? 0x3F800000u - __float_as_uint(prod) : kOutKey30;
        in_pool += prod > 0.0f;
        keys[e] = ((unsigned long long)k30 << 32) | (unsigned)e;
    }
    for (int rq = tid; rq < R; rq += nt) ell_s[rq] = 0;
    if (bad) atomicExch(&s_bad, 1);
    for (int e = n + tid; e < npad; e += nt) keys[e] = ((unsigned long long)kOutKey30 << 32) | (unsigned)e;
    in_pool = __reduce_add_sync(0xffffffffu, in_pool);
    if ((tid & 31) == 0 && in_pool) atomicAdd(&s_pool, in_pool);
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

    // 2. stable radix sort, ascending keys
    radix_sort_keys<IPT>(keys, tmp, hist, reinterpret_cast<int *>(warp_tot));
    const int pool = s_pool;

    // 3. tau in 2^-32 units: exact integer prefix sums of round(a * 2^32)
    const int i0 = tid * IPT;
    long long u[IPT];
    long long local = 0;
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
        const int i = i0 + q;
        u[q] = i < pool ? units_of(__uint_as_float(0x3F800000u - (unsigned)(keys[i] >> 32))) : 0;
        local += u[q];
    }
    const long long base = ((long long)R << 32);
    long long run = block_inclusive_scan(local, warp_tot) - local + base;
    if (tid == 0) units[0] = base;
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
        run += u[q];
        units[i0 + q + 1] = run;
    }
    __syncthreads();

    // 4. Theta(m) = (tau_m 2^-32) SPS(R + m) once per prefix m, in place of
    //    units[m]: tau_m is exact in fp64 (units < 2^53, scaled by an exponent
    //    shift), so the one rounded multiply is the oracle's.  fp64 runs at a
    //    small fraction of the fp32 rate here, so the stop test and the argmax
    //    compare the values' bit patterns, which order like the values for
    //    non-negative finite doubles (else the fp64 comparison decides).
    long long *th = units;
    {
        double spv[IPT + 1];  // the table entries of this thread's prefixes, loads in flight together
#pragma unroll
        for (int q = 0; q <= IPT; ++q) spv[q] = tid + q * nt <= pool ? a.sps[R + tid + q * nt - a.B_min] : 0.0;
#pragma unroll
        for (int q = 0; q <= IPT; ++q) {
            const int m = tid + q * nt;
            if (m <= pool) th[m] = __double_as_longlong(__dmul_rn(scaled_units(units[m]), spv[q]));
        }
    }
    __syncthreads();
    long long best_th = 0;
    int best_m = 0x7fffffff;
    int first = 0x7fffffff;
    for (int m = tid; m <= pool; m += nt) {
        const long long t = th[m];
        if (best_m == 0x7fffffff || th_gt(t, best_th)) {  // m increases within a thread: smallest m on ties
            best_th = t;
            best_m = m;
        }
        if (m >= 1 && first == 0x7fffffff && th_le(t, th[m - 1])) first = m;
    }
    first = (int)__reduce_min_sync(0xffffffffu, (unsigned)first);
    if ((tid & 31) == 0 && first != 0x7fffffff) atomicMin(&s_first, first);
    // argmax over threads: larger Theta, then smaller m
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const long long th2 = __shfl_xor_sync(0xffffffffu, best_th, off);
        const int m2 = __shfl_xor_sync(0xffffffffu, best_m, off);
        if (m2 != 0x7fffffff &&
            (best_m == 0x7fffffff || th_gt(th2, best_th) || (th2 == best_th && m2 < best_m))) {
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
        best_th = tid < (nt >> 5) ? s_th[tid] : 0;
        best_m = tid < (nt >> 5) ? s_arg[tid] : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const long long th2 = __shfl_xor_sync(0xffffffffu, best_th, off);
            const int m2 = __shfl_xor_sync(0xffffffffu, best_m, off);
            if (m2 != 0x7fffffff &&
                (best_m == 0x7fffffff || th_gt(th2, best_th) || (th2 == best_th && m2 < best_m))) {
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
        *a.theta_best = __longlong_as_double(th[count]);
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

static int sched_ipt(int n) {
    int ipt = 1;
    while (kSchedThreads * ipt < n) ipt <<= 1;
    return ipt;
}

size_t schedule_smem_bytes(int R, int gamma) {
    const int npad = kSchedThreads * sched_ipt(R * gamma);
    return sizeof(unsigned long long) * (size_t)(2 * npad + 1) + sizeof(int) * (size_t)R;
}

template <int IPT>
static cudaError_t launch_schedule_t(const dspark_sched_args &a, size_t smem, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel<IPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    schedule_kernel<IPT><<<1, kSchedThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_schedule(const dspark_sched_args &a, cudaStream_t s) {
    const size_t smem = schedule_smem_bytes(a.R, a.gamma);
    switch (sched_ipt(a.R * a.gamma)) {
        case 1: return launch_schedule_t<1>(a, smem, s);
        case 2: return launch_schedule_t<2>(a, smem, s);
        case 4: return launch_schedule_t<4>(a, smem, s);
        case 8: return launch_schedule_t<8>(a, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_build_tags(int R, int gamma, const int32_t *ell, int32_t *tags, int32_t *N_out,
                              int32_t *err, cudaStream_t s) {
    build_tags_kernel<<<1, 1024, 0, s>>>(R, gamma, ell, tags, N_out, err);
    return cudaGetLastError();
}

}  // namespace dspark
