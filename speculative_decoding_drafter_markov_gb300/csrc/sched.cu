// sched.cu -- hardware-aware prefix scheduler and flattened-batch tags.
//
// DSpark digest, Module E and Algorithm 1: a_{r,j} = prod_{i<=j} c_{r,i}; the
// pool E = {(r,j): a_{r,j} > 0} sorted by a descending; admit greedily while
// Theta = tau * SPS(B) improves (break at the first non-improvement).  The
// production section replaces the break by a top-K of the current order with K
// taken from the confidences of two cycles earlier.
//
// A cluster of eight CTAs makes the decision (the pool holds at most 8192
// entries, one per thread; CTA c holds positions 1024 c .. 1024 c + 1023):
//   1. fp32 running products a (IEEE products, identical to any CPU);
//   2. 30-bit sort keys 0x3F800000 - bits(a) (a in (0, 1]; 0x3FFFFFFF marks an
//      entry outside the pool): ascending key order is a descending, and a
//      stable sort of the entries in flat-index order breaks ties by
//      (request, position).  Stable LSD radix sort in the cluster's shared
//      memory, 5-bit digits, 6 passes: each warp ranks its entries with five
//      ballots (the lanes sharing a digit); the (digit, warp) counts of the CTA
//      and the digit counts of the CTAs before it place them, and each entry
//      moves to the CTA that holds its new position;
//   3. tau as an exact integer prefix sum in 2^-32 units;
//   4. Theta(m) = (tau_m 2^-32) * SPS(R + m) for every prefix m in parallel;
//      the synchronous stop is the first m with Theta(m) <= Theta(m-1), the
//      capacity for cycle t+2 is argmax_m Theta(m) (smallest m on ties);
//   5. l_r = largest admitted position of request r.
#include <cooperative_groups.h>

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

// the lanes of the warp whose kRadixBits-bit digit is d, from the warp's
// per-bit ballots
__device__ __forceinline__ unsigned digit_lanes(const unsigned (&vote)[kRadixBits], int d) {
    unsigned m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < kRadixBits; ++b) m &= ((d >> b) & 1) ? vote[b] : ~vote[b];
    return m;
}

constexpr int kClusterCtas = 8;          // CTAs of the scheduler's cluster
constexpr int kCtaItems = kSchedThreads;  // sort positions per CTA: one per thread

// The scheduler on a cluster of kClusterCtas CTAs (distributed shared memory):
// CTA c holds positions c 1024 .. c 1024 + 1023 of the pool order (one entry a
// thread), so every per-entry step runs on eight SMs; the radix passes exchange
// the CTAs' digit counts and scatter the entries through the cluster's shared
// memory, and the prefix sums and reductions combine the CTAs' parts in CTA
// order.  Every CTA takes the same path (the decisions are cluster-wide), and
// none leaves while another may still read its shared memory.
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kSchedThreads)
    schedule_cluster_kernel(const dspark_sched_args a) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    __shared__ unsigned long long keys[2][kCtaItems];
    __shared__ int hist[kBins * kHistLd];  // (digit, warp) counts, then their prefix in the CTA
    __shared__ int dtot[kBins];             // this CTA's count of each digit (read by the others)
    __shared__ int gbase[kBins];            // first position of this CTA's entries of each digit
    __shared__ long long warp_tot[32];
    __shared__ long long s_th[kCtaItems];   // Theta(m) for m = c 1024 + t + 1
    __shared__ long long s_red_th[32];
    __shared__ int s_red_m[32];
    __shared__ int s_bad, s_pool, s_first;  // this CTA's parts, read by the others
    __shared__ long long s_ctot, s_best_th, s_th0;
    __shared__ int s_best_m;
    const int R = a.R, G = a.gamma, n = R * G, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int p0 = c * kCtaItems;  // this CTA's first position
    if (tid == 0) {
        s_bad = 0;
        s_pool = 0;
        s_first = 0x7fffffff;
    }
    // the verify lengths start at 0 (atomic maxima follow, after cluster barriers)
    for (int rq = c * kSchedThreads + tid; rq < R; rq += kClusterCtas * kSchedThreads) a.ell[rq] = 0;
    __syncthreads();

    // 1. survival products (Algorithm 1, line 1): one thread per request whose
    //    entries meet this CTA's range, the same left-to-right products; each
    //    entry's key (line 2) in flat-index order
    {
        const int rq0 = p0 / G, rq1 = min(R - 1, (p0 + kCtaItems - 1) / G);
        bool bad = false;
        int in_pool = 0;
        const int rq = rq0 + tid;
        if (p0 < n && rq <= rq1) {
            const float *cr = a.c + (size_t)rq * G;
            float prod = 1.0f;
            for (int j = 0; j < G; ++j) {
                const int e = rq * G + j;
                const float cc = cr[j];
                prod = __fmul_rn(prod, cc);
                if (e < p0 || e >= p0 + kCtaItems) continue;
                if (!(cc >= 0.0f && cc <= 1.0f)) bad = true;
                if (a.a) a.a[e] = prod;
                const uint32_t k30 = prod > 0.0f ? 0x3F800000u - __float_as_uint(prod) : kOutKey30;
                in_pool += prod > 0.0f;
                keys[0][e - p0] = ((unsigned long long)k30 << 32) | (unsigned)e;
            }
        }
        if (p0 + tid >= n) keys[0][tid] = ((unsigned long long)kOutKey30 << 32) | (unsigned)(p0 + tid);
        if (bad) atomicExch(&s_bad, 1);
        in_pool = __reduce_add_sync(0xffffffffu, in_pool);
        if (lane == 0 && in_pool) atomicAdd(&s_pool, in_pool);
    }
    cluster.sync();
    int bad = 0, pool = 0;
    for (int q = 0; q < kClusterCtas; ++q) {
        bad |= *cluster.map_shared_rank(&s_bad, q);
        pool += *cluster.map_shared_rank(&s_pool, q);
    }
    cluster.sync();  // every CTA has read the others' parts
    if (bad) {
        if (c == 0 && tid == 0) {
            set_err(a.err, DSPARK_ERR_RANGE);
            *a.K_out = 0;
            *a.theta_best = 0.0;
        }
        return;  // every CTA: the decision is the cluster's
    }

    // 2. stable LSD radix sort of the keys (bits 32..61), 5-bit digits: a warp
    //    ranks its 32 entries with five ballots; the CTA's (digit, warp) counts,
    //    the cluster's digit counts in CTA order and the rank give the new
    //    position, and the entry moves to the CTA that holds it
    const unsigned lt_mask = (1u << lane) - 1u;
    int cur = 0;
    for (int pass = 0; pass < kRadixPasses; ++pass) {
        const int shift = 32 + kRadixBits * pass;
        const unsigned long long v = keys[cur][tid];
        const int d = (int)(v >> shift) & (kBins - 1);
        unsigned vote[kRadixBits];
#pragma unroll
        for (int b = 0; b < kRadixBits; ++b) vote[b] = __ballot_sync(0xffffffffu, (d >> b) & 1);
        const int rank = __popc(digit_lanes(vote, d) & lt_mask);
        hist[lane * kHistLd + warp] = __popc(digit_lanes(vote, lane));  // entries of digit `lane`
        __syncthreads();
        {
            // warp d: the digit's counts over the CTA's warps, prefix and total
            const int dd = warp, w = lane;
            const int cnt = hist[dd * kHistLd + w];
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            hist[dd * kHistLd + w] = incl - cnt;
            if (lane == 31) dtot[dd] = incl;
        }
        cluster.sync();
        if (warp == 0) {
            // digit `lane`: its count in every CTA; where this CTA's entries of it start
            int tot = 0, before = 0;
            for (int q = 0; q < kClusterCtas; ++q) {
                const int t = *cluster.map_shared_rank(&dtot[lane], q);
                tot += t;
                if (q < c) before += t;
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            gbase[lane] = incl - tot + before;
        }
        __syncthreads();
        const int pos = gbase[d] + hist[d * kHistLd + warp] + rank;
        *cluster.map_shared_rank(&keys[cur ^ 1][pos & (kCtaItems - 1)], pos / kCtaItems) = v;
        cluster.sync();  // every entry placed; the digit counts read
        cur ^= 1;
    }

    // 3. tau in 2^-32 units: exact integer prefix sums of round(a 2^32) over the
    //    pool order, the CTAs' totals added in CTA order
    const unsigned long long kv = keys[cur][tid];
    const int i = p0 + tid;  // this entry's position
    const long long u = i < pool ? units_of(__uint_as_float(0x3F800000u - (unsigned)(kv >> 32))) : 0;
    const long long incl_u = block_inclusive_scan(u, warp_tot);
    if (tid == kSchedThreads - 1) s_ctot = incl_u;
    cluster.sync();
    const long long base = ((long long)R << 32);
    long long off_u = base;
    for (int q = 0; q < c; ++q) off_u += *cluster.map_shared_rank(&s_ctot, q);
    // 4. Theta(m) = (tau_m 2^-32) SPS(R + m) for the prefixes m = i + 1 (and m = 0
    //    at CTA 0), compared by bit pattern like the values (non-negative finite
    //    doubles), else by the fp64 comparison
    const int m = i + 1;
    const long long thm = m <= pool ? __double_as_longlong(__dmul_rn(scaled_units(off_u + incl_u),
                                                                      a.sps[R + m - a.B_min]))
                                    : 0;
    s_th[tid] = thm;
    if (c == 0 && tid == 0) s_th0 = __double_as_longlong(__dmul_rn(scaled_units(base), a.sps[R - a.B_min]));
    cluster.sync();
    // the stop test needs Theta(m - 1): the previous thread's, the previous CTA's
    // last, or Theta(0)
    long long prev = 0;
    if (tid > 0)
        prev = s_th[tid - 1];
    else
        prev = c == 0 ? s_th0 : *cluster.map_shared_rank(&s_th[kCtaItems - 1], c - 1);
    const long long th0 = *cluster.map_shared_rank(&s_th0, 0);
    int first = m <= pool && th_le(thm, prev) ? m : 0x7fffffff;
    // argmax over m (larger Theta, then smaller m); CTA 0 also holds m = 0
    long long best_th = m <= pool ? thm : 0;
    int best_m = m <= pool ? m : 0x7fffffff;
    if (c == 0 && tid == 0 && (best_m == 0x7fffffff || !th_gt(best_th, th0))) {
        best_th = th0;
        best_m = 0;
    }
    first = (int)__reduce_min_sync(0xffffffffu, (unsigned)first);
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
    if (lane == 0) {
        s_red_th[warp] = best_th;
        s_red_m[warp] = best_m;
        if (first != 0x7fffffff) atomicMin(&s_first, first);
    }
    __syncthreads();
    if (warp == 0) {
        best_th = s_red_th[lane];
        best_m = s_red_m[lane];
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
        if (lane == 0) {
            s_best_th = best_th;
            s_best_m = best_m;
        }
    }
    cluster.sync();
    // the cluster's argmax and first stop, from the CTAs' parts in CTA order
    int K_cap = 0x7fffffff, stop = 0x7fffffff;
    long long K_th = 0;
    for (int q = 0; q < kClusterCtas; ++q) {
        const int m2 = *cluster.map_shared_rank(&s_best_m, q);
        const long long th2 = *cluster.map_shared_rank(&s_best_th, q);
        if (m2 != 0x7fffffff && (K_cap == 0x7fffffff || th_gt(th2, K_th) || (th2 == K_th && m2 < K_cap))) {
            K_th = th2;
            K_cap = m2;
        }
        stop = min(stop, *cluster.map_shared_rank(&s_first, q));
    }
    int count = stop == 0x7fffffff ? pool : stop - 1;
    if (a.mode == DSPARK_SCHED_ASYNC && a.K_in != nullptr) {
        const int K = *a.K_in;
        if (K >= 0) count = min(K, pool);
    }
    // Theta at the admitted point: Theta(0) or the entry's of position count - 1
    if (count == 0) {
        if (c == 0 && tid == 0) *a.theta_best = __longlong_as_double(th0);
    } else if (count - 1 == i) {
        *a.theta_best = __longlong_as_double(thm);
    }
    if (c == 0 && tid == 0) *a.K_out = K_cap;

    // 5. verify lengths: l_r <- j for every admitted (r, j) (its position < count)
    if (i < count) {
        const unsigned e = (unsigned)(kv & 0xFFFFFFFFull);
        atomicMax(&a.ell[e / G], (int)(e % G) + 1);
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
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

cudaError_t launch_schedule(const dspark_sched_args &a, cudaStream_t s) {
    if (a.R * a.gamma > kClusterCtas * kCtaItems) return cudaErrorInvalidValue;
    schedule_cluster_kernel<<<kClusterCtas, kSchedThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_build_tags(int R, int gamma, const int32_t *ell, int32_t *tags, int32_t *N_out,
                              int32_t *err, cudaStream_t s) {
    build_tags_kernel<<<1, 1024, 0, s>>>(R, gamma, ell, tags, N_out, err);
    return cudaGetLastError();
}

}  // namespace dspark
