// train_loss.cu -- the drafter's training losses and their gradient.
//
// DSpark digest, Module F: three losses, each position weighted by
// w_k = exp(-(k - 1) / gamma) -- cross-entropy of the target's token under the
// draft distribution (eq. 9), the total variation ||p_d - p_t||_1 between the
// draft and target distributions (eq. 10), and binary cross-entropy of the
// confidence towards c* = 1 - ||p_d - p_t||_1 / 2 (eqs. 8, 11) -- combined as
// L = a_ce L_ce + a_tv L_tv + a_conf L_conf (eq. 12), averaged over the blocks.
//
// One persistent CTA per SM walks rows i = blockIdx.x, + gridDim.x, ...  A row
// takes two passes over its draft and target logits (the log-sum-exps, then
// the total variation and sum_v p_d sgn(p_d - p_t)) and, when the gradient is
// wanted, a third that writes dL/dzd.  With one row per SM in flight (at most
// 152 rows x 2 x V x 2 bytes, under L2's 129 MB for bf16 at V = 151936) the
// second and third passes read the row back from L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dspark {

namespace {

constexpr int kThreads = 512;
constexpr int kLoads = 4;  // 16-byte loads of each row per thread and iteration

template <typename T>
__device__ __forceinline__ void widen(const uint4 &raw, float (&x)[16 / sizeof(T)]) {
    const T *v = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int j = 0; j < (int)(16 / sizeof(T)); ++j) x[j] = to_f32(v[j]);
}

// online (max, sum of exp(x - max)) over a run of values
__device__ __forceinline__ void lse_feed(float &m, float &S, const float *x, int n) {
    float cm = m;
    for (int j = 0; j < n; ++j) cm = fmaxf(cm, x[j]);
    if (cm > m) {
        S = (m == -INFINITY) ? 0.f : S * ex2((m - cm) * kLog2e);
        m = cm;
    }
    const float mL = m * kLog2e;
    float acc = 0.f;
    for (int j = 0; j < n; ++j) acc += ex2(fmaf(x[j], kLog2e, -mL));
    S += acc;
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

// block-wide reduction of two (max, sum) pairs; every thread gets the result
__device__ void block_lse2(float &md, float &Sd, float &mt, float &St, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lse_merge(md, Sd, __shfl_xor_sync(0xffffffffu, md, off), __shfl_xor_sync(0xffffffffu, Sd, off));
        lse_merge(mt, St, __shfl_xor_sync(0xffffffffu, mt, off), __shfl_xor_sync(0xffffffffu, St, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[4 * warp] = md; red[4 * warp + 1] = Sd; red[4 * warp + 2] = mt; red[4 * warp + 3] = St;
    }
    __syncthreads();
    md = red[0]; Sd = red[1]; mt = red[2]; St = red[3];
    for (int w = 1; w < kThreads / 32; ++w) {  // fixed order: the same result in every thread
        lse_merge(md, Sd, red[4 * w], red[4 * w + 1]);
        lse_merge(mt, St, red[4 * w + 2], red[4 * w + 3]);
    }
    __syncthreads();
}

__device__ void block_sum2(float &a, float &b, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[2 * warp] = a;
        red[2 * warp + 1] = b;
    }
    __syncthreads();
    a = 0.f;
    b = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) {
        a += red[2 * w];
        b += red[2 * w + 1];
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) train_loss_kernel(const dspark_train_loss_args a) {
    __shared__ float red[4 * (kThreads / 32)];
    constexpr int kVec = 16 / sizeof(T);
    const int N = a.B * a.gamma, V = a.V, nv = V / kVec;
    const float invB = 1.0f / (float)a.B;
    const uint64_t keep = tc::policy_evict_last(), once = tc::policy_evict_first();
    for (int i = blockIdx.x; i < N; i += gridDim.x) {
        const int k = i % a.gamma + 1;
        const float wk = expf(-(float)(k - 1) / (float)a.gamma);
        const uint4 *rd = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.zd) + (size_t)i * V);
        const uint4 *rt = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.zt) + (size_t)i * V);
        const int xs = a.xs[i];
        const bool tok_ok = xs >= 0 && xs < V;
        if (!tok_ok && threadIdx.x == 0) set_err(a.err, DSPARK_ERR_RANGE);

        // pass 1: log-sum-exp of both rows (kept in L2 for the next passes)
        float md = -INFINITY, Sd = 0.f, mt = -INFINITY, St = 0.f;
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
                    float x[kVec];
                    widen<T>(raw_d[q], x);
                    lse_feed(md, Sd, x, kVec);
                    widen<T>(raw_t[q], x);
                    lse_feed(mt, St, x, kVec);
                }
            }
        }
        block_lse2(md, Sd, mt, St, red);
        const float lse_d = md + logf(Sd), lse_t = mt + logf(St);
        const float ld2 = lse_d * kLog2e, lt2 = lse_t * kLog2e;

        // pass 2: ||p_d - p_t||_1 and sum_v p_d sgn(p_d - p_t)
        float tv = 0.f, msg = 0.f;
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
            for (int q = 0; q < kLoads; ++q) {
                if (c0 + q * kThreads < nv) {
                    float xd[kVec], xt[kVec];
                    widen<T>(raw_d[q], xd);
                    widen<T>(raw_t[q], xt);
#pragma unroll
                    for (int j = 0; j < kVec; ++j) {
                        const float ad = fmaf(xd[j], kLog2e, -ld2), at = fmaf(xt[j], kLog2e, -lt2);
                        const float pd = ex2(ad), pt = ex2(at);
                        tv += fabsf(pd - pt);
                        msg += ad > at ? pd : (ad < at ? -pd : 0.f);  // the sign pass 3 uses
                    }
                }
            }
        }
        block_sum2(tv, msg, red);

        // the row's terms (thread 0)
        if (threadIdx.x == 0) {
            const float zx = tok_ok ? to_f32(static_cast<const T *>(a.zd)[(size_t)i * V + xs]) : 0.f;
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
            if (a.grad_s) a.grad_s[i] = a.a_conf * wk * invB * (1.f / (1.f + expf(-si)) - cstar);
        }

        // pass 3: dL/dzd = w/B [a_ce (p_d - onehot) + a_tv p_d (sgn - msg)], four floats per store
        if (a.grad_z) {
            const float gw = wk * invB, gce = a.a_ce * gw, gtv = a.a_tv * gw;
            float4 *gz = reinterpret_cast<float4 *>(a.grad_z + (size_t)i * V);
            for (int c = threadIdx.x; c < nv; c += kThreads) {
                float xd[kVec], xt[kVec];
                widen<T>(tc::ld_global_hint(rd + c, once), xd);
                widen<T>(tc::ld_global_hint(rt + c, once), xt);
                float g[kVec];
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    // sgn(p_d - p_t) = sgn(log p_d - log p_t): the target's exponential is not needed
                    const float ad = fmaf(xd[j], kLog2e, -ld2), at = fmaf(xt[j], kLog2e, -lt2);
                    const float pd = ex2(ad);
                    const float sg = ad > at ? 1.f : (ad < at ? -1.f : 0.f);
                    const int v = c * kVec + j;
                    g[j] = gce * (pd - (v == xs ? 1.f : 0.f)) + gtv * pd * (sg - msg);
                }
#pragma unroll
                for (int j = 0; j < kVec; j += 4)
                    __stcs(gz + (c * kVec + j) / 4, make_float4(g[j], g[j + 1], g[j + 2], g[j + 3]));
            }
        }
    }
}

}  // namespace

cudaError_t launch_train_losses(const dspark_train_loss_args &a, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(a.loss, 0, 4 * sizeof(double), s);
    if (e != cudaSuccess) return e;
    int grid = sm_count();
    if (grid < 1) grid = 1;
    const int N = a.B * a.gamma;
    if (grid > N) grid = N;
    if (a.dtype == DSPARK_BF16)
        train_loss_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
    else
        train_loss_kernel<float><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
