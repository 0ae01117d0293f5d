// train_loss.cu -- the drafter's training losses and their gradient.
//
// DSpark digest, Module F: three losses, each position weighted by
// w_k = exp(-(k - 1) / gamma) -- cross-entropy of the target's token under the
// draft distribution (eq. 9), the total variation ||p_d - p_t||_1 between the
// draft and target distributions (eq. 10), and binary cross-entropy of the
// confidence towards c* = 1 - ||p_d - p_t||_1 / 2 (eqs. 8, 11) -- combined as
// L = a_ce L_ce + a_tv L_tv + a_conf L_conf (eq. 12), averaged over the blocks.
//
// Every row needs three sweeps over its draft and target logits (the
// log-sum-exps; then the total variation and sum_v p_d sgn(p_d - p_t); then,
// when the gradient is wanted, dL/dzd), and neither later sweep can be folded
// into an earlier one: |p_d - p_t| does not factor through a running maximum.
// The sweeps are bound by instruction issue, so the arithmetic runs on fp32
// pairs (one f32x2 instruction per two elements), the running maximum on bf16
// pairs, and the gradient is written as dL/dzd_v = p_d,v f(sgn_v) - [v = x]
// a_ce w/B with f one of three row constants; the one-hot term is added after
// the sweep by the thread that owns column x.
//
// Resident kernel (the default): a cluster of kClusterCtas CTAs owns a row at a
// time, each CTA holding one contiguous slice of the row pair in shared memory,
// brought in by one bulk asynchronous copy per slice.  The three sweeps run out
// of shared memory; the per-slice partial (max, sum) pairs and (tv, msg) sums
// are exchanged over distributed shared memory between two cluster barriers.
// Two or three CTAs of different clusters share an SM, so while one waits on
// its copy, its barriers or its reductions the others sweep.  HBM sees each
// logit once and each gradient element once.
//
// Streaming kernel (when fewer than two slice pairs fit in an SM's shared
// memory, or no cluster can be placed): one persistent CTA per SM walks rows
// i = blockIdx.x, + gridDim.x, ...; the second and third sweeps read the row
// back through L2 (at most 152 rows x 2 x V x 2 bytes in flight, under L2's
// 129 MB for bf16 at V = 151936).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

#include <algorithm>
#include <mutex>

namespace dspark {

namespace {

constexpr int kThreads = 512;     // streaming kernel: one CTA per SM
constexpr int kResThreads = 256;  // resident kernel: two CTAs per SM
constexpr int kWarps = kThreads / 32;
constexpr int kLoads = 4;  // 16-byte loads of each row per thread and iteration (streaming kernel)

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 16 bytes of logits: kPairs fp32 pairs (elements 2q, 2q + 1) and their maximum
template <typename T>
struct Chunk;

template <>
struct Chunk<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    static __device__ __forceinline__ uint32_t word(const uint4 &r, int q) {
        return q == 0 ? r.x : q == 1 ? r.y : q == 2 ? r.z : r.w;
    }
    static __device__ __forceinline__ float2 pair(const uint4 &r, int q) {
        const uint32_t w = word(r, q);
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ __nv_bfloat162 as_b2(uint32_t w) {
        __nv_bfloat162 b;
        *reinterpret_cast<uint32_t *>(&b) = w;
        return b;
    }
    static __device__ __forceinline__ float max(const uint4 &r) {
        const __nv_bfloat162 m = __hmax2(__hmax2(as_b2(r.x), as_b2(r.y)), __hmax2(as_b2(r.z), as_b2(r.w)));
        return fmaxf(__low2float(m), __high2float(m));
    }
};

template <>
struct Chunk<float> {
    static constexpr int kPairs = 2;
    static __device__ __forceinline__ float2 pair(const uint4 &r, int q) {
        return q == 0 ? make_float2(__uint_as_float(r.x), __uint_as_float(r.y))
                      : make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    static __device__ __forceinline__ float max(const uint4 &r) {
        return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                     fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
    }
};

// Online log-sum-exp state of one thread: m = running maximum, S = sum of
// 2^(x log2e - m log2e) over the elements seen, kept as a pair of partial sums.
struct Lse {
    float m = -INFINITY, mL = 0.f;
    float2 S = make_float2(0.f, 0.f);
};

template <typename T>
__device__ __forceinline__ void lse_feed(Lse &st, const uint4 &r) {
    const float cm = Chunk<T>::max(r);
    if (cm > st.m) {  // a new maximum: rescale (S is 0 while m = -inf)
        const float f = ex2((st.m - cm) * kLog2e);
        st.S = make_float2(st.S.x * f, st.S.y * f);
        st.m = cm;
        st.mL = cm * kLog2e;
    }
    const float2 l2 = make_float2(kLog2e, kLog2e), nm = make_float2(-st.mL, -st.mL);
#pragma unroll
    for (int q = 0; q < Chunk<T>::kPairs; ++q) {
        const float2 a = fma2(Chunk<T>::pair(r, q), l2, nm);
        st.S = add2(st.S, make_float2(ex2(a.x), ex2(a.y)));
    }
}

__device__ __forceinline__ void lse_merge(float &m, float &S, float m2, float S2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) {
        S = 0.f;
    } else {
        S = S * ex2((m - M) * kLog2e) + S2 * ex2((m2 - M) * kLog2e);
    }
    m = M;
}

// Block-wide (max, sum) of two online states, merged in a fixed tree order;
// every thread gets the block's (m, S) for both rows in md, Sd, mt, St.
template <int NT>
__device__ void block_lse2(const Lse &d, const Lse &t, float &md, float &Sd, float &mt, float &St,
                           float4 *red) {
    constexpr int NW = NT / 32;
    md = d.m; Sd = d.S.x + d.S.y; mt = t.m; St = t.S.x + t.S.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lse_merge(md, Sd, __shfl_xor_sync(0xffffffffu, md, off), __shfl_xor_sync(0xffffffffu, Sd, off));
        lse_merge(mt, St, __shfl_xor_sync(0xffffffffu, mt, off), __shfl_xor_sync(0xffffffffu, St, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = make_float4(md, Sd, mt, St);
    __syncthreads();
    if (warp == 0) {
        const float4 p = lane < NW ? red[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        md = p.x; Sd = p.y; mt = p.z; St = p.w;
#pragma unroll
        for (int off = NW / 2; off > 0; off >>= 1) {
            lse_merge(md, Sd, __shfl_xor_sync(0xffffffffu, md, off), __shfl_xor_sync(0xffffffffu, Sd, off));
            lse_merge(mt, St, __shfl_xor_sync(0xffffffffu, mt, off), __shfl_xor_sync(0xffffffffu, St, off));
        }
        if (lane == 0) red[NW] = make_float4(md, Sd, mt, St);
    }
    __syncthreads();
    const float4 r = red[NW];
    md = r.x; Sd = r.y; mt = r.z; St = r.w;
}

// block-wide sums of a and b (fixed tree order), returned in every thread
template <int NT>
__device__ void block_sum2(float &a, float &b, float4 *red) {
    constexpr int NW = NT / 32;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = make_float4(a, b, 0.f, 0.f);
    __syncthreads();
    if (warp == 0) {
        const float4 p = lane < NW ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        a = p.x; b = p.y;
#pragma unroll
        for (int off = NW / 2; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
        }
        if (lane == 0) red[NW] = make_float4(a, b, 0.f, 0.f);
    }
    __syncthreads();
    a = red[NW].x;
    b = red[NW].y;
}

// (max, sum) pairs of the warps of a CTA merged into red[NW] by warp 0, in a
// fixed tree order (the CTA's threads must pass a barrier before reading it)
template <int NT>
__device__ void cta_lse2(const Lse &d, const Lse &t, float4 *red) {
    constexpr int NW = NT / 32;
    float md = d.m, Sd = d.S.x + d.S.y, mt = t.m, St = t.S.x + t.S.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lse_merge(md, Sd, __shfl_xor_sync(0xffffffffu, md, off), __shfl_xor_sync(0xffffffffu, Sd, off));
        lse_merge(mt, St, __shfl_xor_sync(0xffffffffu, mt, off), __shfl_xor_sync(0xffffffffu, St, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = make_float4(md, Sd, mt, St);
    __syncthreads();
    if (warp == 0) {
        const float4 p = lane < NW ? red[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        md = p.x; Sd = p.y; mt = p.z; St = p.w;
#pragma unroll
        for (int off = NW / 2; off > 0; off >>= 1) {
            lse_merge(md, Sd, __shfl_xor_sync(0xffffffffu, md, off), __shfl_xor_sync(0xffffffffu, Sd, off));
            lse_merge(mt, St, __shfl_xor_sync(0xffffffffu, mt, off), __shfl_xor_sync(0xffffffffu, St, off));
        }
        if (lane == 0) red[NW] = make_float4(md, Sd, mt, St);
    }
}

// sums of a and b over the CTA into red[NW] by warp 0 (fixed tree order)
template <int NT>
__device__ void cta_sum2(float a, float b, float4 *red) {
    constexpr int NW = NT / 32;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = make_float4(a, b, 0.f, 0.f);
    __syncthreads();
    if (warp == 0) {
        const float4 p = lane < NW ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        a = p.x; b = p.y;
#pragma unroll
        for (int off = NW / 2; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
        }
        if (lane == 0) red[NW] = make_float4(a, b, 0.f, 0.f);
    }
}

// Row constants of sweeps 2 and 3: 2^(x log2e - lse log2e) = softmax(x).
struct RowScale {
    float2 l2, nld, nlt;  // (log2e, log2e), -lse_d log2e, -lse_t log2e
    __device__ RowScale(float lse_d, float lse_t)
        : l2(make_float2(kLog2e, kLog2e)),
          nld(make_float2(-lse_d * kLog2e, -lse_d * kLog2e)),
          nlt(make_float2(-lse_t * kLog2e, -lse_t * kLog2e)) {}
};

// sweep 2 over 16 bytes: ||p_d - p_t||_1 and sum_v p_d sgn(log p_d - log p_t)
template <typename T>
__device__ __forceinline__ void tv_chunk(const uint4 &rd, const uint4 &rt, const RowScale &rs, float2 &tv,
                                         float &msg) {
#pragma unroll
    for (int q = 0; q < Chunk<T>::kPairs; ++q) {
        const float2 ad = fma2(Chunk<T>::pair(rd, q), rs.l2, rs.nld);
        const float2 at = fma2(Chunk<T>::pair(rt, q), rs.l2, rs.nlt);
        const float2 pd = make_float2(ex2(ad.x), ex2(ad.y));
        const float2 dd = sub2(pd, make_float2(ex2(at.x), ex2(at.y)));
        tv = add2(tv, make_float2(fabsf(dd.x), fabsf(dd.y)));
        msg += ad.x > at.x ? pd.x : (ad.x < at.x ? -pd.x : 0.f);
        msg += ad.y > at.y ? pd.y : (ad.y < at.y ? -pd.y : 0.f);
    }
}

// sweep 3 over 16 bytes: p_d,v f_v with f_v = kp, km or k0 as log p_d >, < or =
// log p_t, written as fp32 with streaming stores (the one-hot term comes later)
template <typename T>
__device__ __forceinline__ void grad_chunk(const uint4 &rd, const uint4 &rt, const RowScale &rs, float kp,
                                           float km, float k0, float4 *gz) {
    float2 g[Chunk<T>::kPairs];
#pragma unroll
    for (int q = 0; q < Chunk<T>::kPairs; ++q) {
        const float2 ad = fma2(Chunk<T>::pair(rd, q), rs.l2, rs.nld);
        const float2 at = fma2(Chunk<T>::pair(rt, q), rs.l2, rs.nlt);
        const float2 f = make_float2(ad.x > at.x ? kp : (ad.x < at.x ? km : k0),
                                     ad.y > at.y ? kp : (ad.y < at.y ? km : k0));
        g[q] = mul2(make_float2(ex2(ad.x), ex2(ad.y)), f);
    }
#pragma unroll
    for (int q = 0; q < Chunk<T>::kPairs; q += 2) __stcs(gz + q / 2, make_float4(g[q].x, g[q].y, g[q + 1].x, g[q + 1].y));
}

// the gradient's three row constants: w/B (a_ce + a_tv (sgn - msg)) for sgn = +1, -1, 0
struct GradScale {
    float kp, km, k0, gce;
    __device__ GradScale(const dspark_train_loss_args &a, float wk, float msg) {
        const float gw = wk / (float)a.B;
        gce = a.a_ce * gw;
        const float gtv = a.a_tv * gw;
        k0 = gce - gtv * msg;
        kp = k0 + gtv;
        km = k0 - gtv;
    }
    // the full gradient at one column, one-hot term included
    __device__ float at(float zd, float zt, const RowScale &rs, bool onehot) const {
        const float ad = fmaf(zd, kLog2e, rs.nld.x), at_ = fmaf(zt, kLog2e, rs.nlt.x);
        const float f = ad > at_ ? kp : (ad < at_ ? km : k0);
        return ex2(ad) * f - (onehot ? gce : 0.f);
    }
};

// The row's terms (one thread): ce, c*, bce into the row outputs, the weighted
// loss totals (fp64 atomics) and dL/ds_i = a_conf w/B (sigmoid(s_i) - c*).
template <typename T>
__device__ void row_terms(const dspark_train_loss_args &a, int i, float wk, float lse_d, float lse_t, float tv,
                          int xs, bool tok_ok) {
    const float zx = tok_ok ? to_f32(static_cast<const T *>(a.zd)[(size_t)i * a.V + xs]) : 0.f;
    const float ce = lse_d - zx;
    const float cstar = 1.f - 0.5f * tv;
    const float si = a.s[i];
    const float sp = si > 0.f ? si + log1pf(expf(-si)) : log1pf(expf(si));
    const float bce = sp - cstar * si;
    if (a.row) {
        float *ro = a.row + (size_t)i * 6;
        ro[0] = lse_d; ro[1] = lse_t; ro[2] = ce; ro[3] = tv; ro[4] = cstar; ro[5] = bce;
    }
    if (tok_ok) {
        const double w = (double)wk / a.B;
        atomicAdd(a.loss + 0, w * ce);
        atomicAdd(a.loss + 1, w * tv);
        atomicAdd(a.loss + 2, w * bce);
        atomicAdd(a.loss + 3, w * ((double)a.a_ce * ce + (double)a.a_tv * tv + (double)a.a_conf * bce));
    }
    if (a.grad_s) a.grad_s[i] = a.a_conf * wk / (float)a.B * (1.f / (1.f + expf(-si)) - cstar);
}

// ---------------------------------------------------------------- streaming kernel
template <typename T>
__global__ void __launch_bounds__(kThreads, 1) train_loss_kernel(const dspark_train_loss_args a) {
    __shared__ float4 red[kWarps + 1];
    constexpr int kVec = 16 / sizeof(T);
    const int N = a.B * a.gamma, V = a.V, nv = V / kVec;
    const uint64_t keep = tc::policy_evict_last(), once = tc::policy_evict_first();
    for (int i = blockIdx.x; i < N; i += gridDim.x) {
        const int k = i % a.gamma + 1;
        const float wk = expf(-(float)(k - 1) / (float)a.gamma);
        const T *zd = static_cast<const T *>(a.zd) + (size_t)i * V;
        const T *zt = static_cast<const T *>(a.zt) + (size_t)i * V;
        const uint4 *rd = reinterpret_cast<const uint4 *>(zd);
        const uint4 *rt = reinterpret_cast<const uint4 *>(zt);
        const int xs = a.xs[i];
        const bool tok_ok = xs >= 0 && xs < V;
        if (!tok_ok && threadIdx.x == 0) set_err(a.err, DSPARK_ERR_RANGE);

        // sweep 1: log-sum-exp of both rows (kept in L2 for the next sweeps)
        Lse sd, st;
        for (int c0 = threadIdx.x; c0 < nv; c0 += kLoads * kThreads) {
            uint4 raw_d[kLoads], raw_t[kLoads];
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const int c = c0 + q * kThreads;
                if (c < nv) {
                    raw_d[q] = tc::ld_global_hint(rd + c, keep);
                    raw_t[q] = tc::ld_global_hint(rt + c, keep);
                }
            }
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                if (c0 + q * kThreads < nv) {
                    lse_feed<T>(sd, raw_d[q]);
                    lse_feed<T>(st, raw_t[q]);
                }
            }
        }
        float md, Sd, mt, St;
        block_lse2<kThreads>(sd, st, md, Sd, mt, St, red);
        const float lse_d = md + logf(Sd), lse_t = mt + logf(St);
        const RowScale rs(lse_d, lse_t);

        // sweep 2: ||p_d - p_t||_1 and sum_v p_d sgn(p_d - p_t)
        float2 tv2 = make_float2(0.f, 0.f);
        float msg = 0.f;
        for (int c0 = threadIdx.x; c0 < nv; c0 += kLoads * kThreads) {
            uint4 raw_d[kLoads], raw_t[kLoads];
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const int c = c0 + q * kThreads;
                if (c < nv) {
                    raw_d[q] = tc::ld_global_hint(rd + c, a.grad_z ? keep : once);
                    raw_t[q] = tc::ld_global_hint(rt + c, a.grad_z ? keep : once);
                }
            }
#pragma unroll
            for (int q = 0; q < kLoads; ++q)
                if (c0 + q * kThreads < nv) tv_chunk<T>(raw_d[q], raw_t[q], rs, tv2, msg);
        }
        float tv = tv2.x + tv2.y;
        block_sum2<kThreads>(tv, msg, red);

        if (threadIdx.x == 0) row_terms<T>(a, i, wk, lse_d, lse_t, tv, xs, tok_ok);

        // sweep 3: dL/dzd; the one-hot column is rewritten after the sweep's store
        if (a.grad_z) {
            const GradScale gs(a, wk, msg);
            float4 *gz = reinterpret_cast<float4 *>(a.grad_z + (size_t)i * V);
            for (int c = threadIdx.x; c < nv; c += kThreads)
                grad_chunk<T>(tc::ld_global_hint(rd + c, once), tc::ld_global_hint(rt + c, once), rs, gs.kp, gs.km,
                              gs.k0, gz + c * kVec / 4);
            __syncthreads();
            if (threadIdx.x == 0 && tok_ok)
                a.grad_z[(size_t)i * V + xs] = gs.at(to_f32(zd[xs]), to_f32(zt[xs]), rs, true);
        }
    }
}

// ---------------------------------------------------------------- resident kernel
constexpr int kClusterCtas = 8;       // CTAs sharing one row (the portable cluster size)
constexpr uint32_t kBulkChunk = 32768;  // bytes per bulk copy

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// all threads of all CTAs of the cluster; shared-memory writes before it are
// visible to every CTA of the cluster after it
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the 16 bytes at shared address `p` of cluster CTA `rank`
__device__ __forceinline__ float4 ld_cluster_f4(const void *p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(tc::smem_u32(p)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}
// bulk asynchronous copy global -> this CTA's shared memory (16-byte aligned
// addresses, a multiple of 16 bytes), counted on `bar`
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(tc::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar)), "l"(policy)
        : "memory");
}

// shared memory after the slice pair; red1[NW] and red2[NW] are the CTA's
// partials of sweeps 1 and 2 that the other CTAs of the cluster read, merged
// by warp 0 into `row` for the CTA
struct ResTail {
    float4 red1[kResThreads / 32 + 1];
    float4 red2[kResThreads / 32 + 1];
    float4 row;  // the row's (lse_d, lse_t) after sweep 1, (tv, msg) after sweep 2
    uint64_t full;
    int abort;
};

// Cluster CTA `rank` owns columns [rank L, rank L + L) of every row of its
// cluster (rows cluster, + clusters, ...); its shared memory holds
// [zd slice | zt slice] of the current row.
template <typename T>
__global__ void __launch_bounds__(kResThreads, 2) train_loss_resident(const dspark_train_loss_args a, int L) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int kVec = 16 / sizeof(T);
    const size_t slice_bytes = (size_t)L * sizeof(T);
    ResTail &tl = *reinterpret_cast<ResTail *>(smem + 2 * slice_bytes);
    const uint32_t rank = cluster_ctarank(), C = cluster_nctarank();
    const int cl = (int)cluster_id_x(), ncl = (int)cluster_count_x();
    const int N = a.B * a.gamma, V = a.V, tid = threadIdx.x;
    const int col0 = (int)rank * L;
    const int len = max(0, min(L, V - col0));
    const int nch = len / kVec;
    const uint32_t bytes = (uint32_t)len * sizeof(T);
    const uint64_t once = tc::policy_evict_first();

    if (tid == 0) {
        tc::mbar_init(&tl.full, 1);
        tl.abort = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();

    int issued = 0;  // loads issued (thread 0)
    auto issue = [&](int row) {
        uint64_t *bar = &tl.full;
        ++issued;
        if (bytes == 0) {
            tc::mbar_arrive(bar);
            return;
        }
        tc::mbar_expect_tx(bar, 2 * bytes);
        unsigned char *dst = smem;
        const size_t off = ((size_t)row * V + col0) * sizeof(T);
        const unsigned char *zd = static_cast<const unsigned char *>(a.zd) + off;
        const unsigned char *zt = static_cast<const unsigned char *>(a.zt) + off;
        for (uint32_t o = 0; o < bytes; o += kBulkChunk) {
            const uint32_t n = min(kBulkChunk, bytes - o);
            bulk_g2s(dst + o, zd + o, n, bar, once);
            bulk_g2s(dst + slice_bytes + o, zt + o, n, bar, once);
        }
    };
    if (tid == 0 && cl < N) issue(cl);

    const uint4 *sd = reinterpret_cast<const uint4 *>(smem);
    const uint4 *sz = reinterpret_cast<const uint4 *>(smem + slice_bytes);
    int j = 0;
    for (int i = cl; i < N; i += ncl, ++j) {
        tc::mbar_wait(&tl.full, (uint32_t)j & 1u, &tl.abort, a.err);
        const int k = i % a.gamma + 1;
        const float wk = expf(-(float)(k - 1) / (float)a.gamma);

        // sweep 1: (max, sum) of both slices; warp 0 merges the cluster's
        // partials in rank order, so all CTAs of the cluster agree
        constexpr int NW = kResThreads / 32;
        const int lane = tid & 31;
        Lse ld, lt;
        for (int c = tid; c < nch; c += kResThreads) {
            lse_feed<T>(ld, sd[c]);
            lse_feed<T>(lt, sz[c]);
        }
        cta_lse2<kResThreads>(ld, lt, tl.red1);
        cluster_sync();
        if (tid < 32) {
            const float4 p = lane < (int)C ? ld_cluster_f4(&tl.red1[NW], lane) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
            float m1 = __shfl_sync(0xffffffffu, p.x, 0), s1 = __shfl_sync(0xffffffffu, p.y, 0);
            float m2 = __shfl_sync(0xffffffffu, p.z, 0), s2 = __shfl_sync(0xffffffffu, p.w, 0);
            for (int r = 1; r < (int)C; ++r) {
                lse_merge(m1, s1, __shfl_sync(0xffffffffu, p.x, r), __shfl_sync(0xffffffffu, p.y, r));
                lse_merge(m2, s2, __shfl_sync(0xffffffffu, p.z, r), __shfl_sync(0xffffffffu, p.w, r));
            }
            if (tid == 0) tl.row = make_float4(m1 + logf(s1), m2 + logf(s2), 0.f, 0.f);
        }
        __syncthreads();
        const float lse_d = tl.row.x, lse_t = tl.row.y;
        const RowScale rs(lse_d, lse_t);

        // sweep 2: ||p_d - p_t||_1 and sum_v p_d sgn(p_d - p_t), summed in rank order
        float2 tv2 = make_float2(0.f, 0.f);
        float msg = 0.f;
        for (int c = tid; c < nch; c += kResThreads) tv_chunk<T>(sd[c], sz[c], rs, tv2, msg);
        cta_sum2<kResThreads>(tv2.x + tv2.y, msg, tl.red2);
        cluster_sync();
        if (tid < 32) {
            const float4 p = lane < (int)C ? ld_cluster_f4(&tl.red2[NW], lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            float t = __shfl_sync(0xffffffffu, p.x, 0), m = __shfl_sync(0xffffffffu, p.y, 0);
            for (int r = 1; r < (int)C; ++r) {
                t += __shfl_sync(0xffffffffu, p.x, r);
                m += __shfl_sync(0xffffffffu, p.y, r);
            }
            if (tid == 0) tl.row = make_float4(t, m, 0.f, 0.f);
        }
        __syncthreads();
        const float tv = tl.row.x;
        msg = tl.row.y;

        const int xs = a.xs[i];
        const bool tok_ok = xs >= 0 && xs < V;
        if (rank == 0 && tid == 0) {
            if (!tok_ok) set_err(a.err, DSPARK_ERR_RANGE);
            row_terms<T>(a, i, wk, lse_d, lse_t, tv, xs, tok_ok);
        }

        // sweep 3: dL/dzd over the slice; the one-hot column is rewritten after
        // the sweep's store by the CTA that holds it
        if (a.grad_z) {
            const GradScale gs(a, wk, msg);
            float4 *gz = reinterpret_cast<float4 *>(a.grad_z + (size_t)i * V + col0);
            for (int c = tid; c < nch; c += kResThreads) grad_chunk<T>(sd[c], sz[c], rs, gs.kp, gs.km, gs.k0, gz + c * kVec / 4);
        }

        // the sweeps are done: thread 0 rewrites the one-hot column (after the
        // sweep's store of it) and brings in this cluster's next row
        __syncthreads();
        if (tid == 0) {
            if (a.grad_z && tok_ok && xs >= col0 && xs < col0 + len) {
                const GradScale gs(a, wk, msg);
                const T *ed = reinterpret_cast<const T *>(sd), *et = reinterpret_cast<const T *>(sz);
                a.grad_z[(size_t)i * V + xs] = gs.at(to_f32(ed[xs - col0]), to_f32(et[xs - col0]), rs, true);
            }
            if (!tl.abort && i + ncl < N) issue(i + ncl);
        }
    }
    // let this CTA's copy land (a no-op unless a wait gave up), and keep its
    // shared memory alive until the other CTAs have read its partials
    if (tid == 0 && issued > 0) tc::mbar_wait_drain(&tl.full, (uint32_t)(issued - 1) & 1u, a.err);
    cluster_sync();
}

}  // namespace

namespace {

// Shared memory and cluster count of the resident kernel for one (dtype, V).
// It is used only when two CTAs fit on an SM (their overlap is what hides each
// CTA's copy, barriers and reductions); clusters = how many the device holds
// at once, 0 when it is not used.
struct ResidentPlan {
    int L = 0, clusters = 0;
    size_t smem = 0;
};

template <typename T>
ResidentPlan plan_resident(int V) {
    static std::mutex mu;
    static int cached_V = -1, cached_dev = -1;
    static ResidentPlan cached;
    ResidentPlan p;
    int dev = 0, per_sm = 0, reserved = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return p;
    std::lock_guard<std::mutex> lock(mu);
    if (V == cached_V && dev == cached_dev) return cached;
    constexpr int kVec = 16 / sizeof(T);
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return p;
    p.L = ((V + kClusterCtas - 1) / kClusterCtas + kVec - 1) / kVec * kVec;
    p.smem = 2 * (size_t)p.L * sizeof(T) + sizeof(ResTail);
    if (2 * (p.smem + reserved) <= (size_t)per_sm) {
        auto kern = train_loss_resident<T>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
            return p.clusters = 0, p;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kClusterCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(kClusterCtas);
        cfg.blockDim = dim3(kResThreads);
        cfg.dynamicSmemBytes = p.smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&p.clusters, kern, &cfg) != cudaSuccess) p.clusters = 0;
    }
    cudaGetLastError();  // a refused query leaves the streaming kernel in charge
    cached_V = V;
    cached_dev = dev;
    cached = p;
    return p;
}

template <typename T>
cudaError_t launch_typed(const dspark_train_loss_args &a, cudaStream_t s) {
    const int N = a.B * a.gamma;
    const ResidentPlan p = plan_resident<T>(a.V);
    if (p.clusters > 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kClusterCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(kClusterCtas * (unsigned)std::min(p.clusters, N));
        cfg.blockDim = dim3(kResThreads);
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, train_loss_resident<T>, a, p.L);
    }
    const int grid = std::max(1, std::min(sm_count(), N));
    train_loss_kernel<T><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_train_losses(const dspark_train_loss_args &a, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(a.loss, 0, 4 * sizeof(double), s);
    if (e != cudaSuccess) return e;
    return a.dtype == DSPARK_BF16 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace dspark
