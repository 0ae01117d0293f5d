// draft.cu -- semi-autoregressive draft step kernels (CUDA cores).
//
// DSpark digest, eq. (4): p_k(v) is a softmax over U_k(v) + B_k(v); eq. (5)
// Markov bias B_k = W_1[x_{k-1}] W_2; eq. (6) RNN bias B_k = W_2^T tanh(W_o z_k);
// eq. (7) confidence c_k = sigma(w^T [h_k ; W_1[x_{k-1}]]).
//
// One draft step is two launches:
//   draft_step_simt  vocabulary-sliced: each CTA owns 64 vocabulary entries,
//                    keeps that slice of W_2 in shared memory, and for every
//                    request contracts the bias operand with it, adds U_k and
//                    folds the result into the sum of exponentials and the
//                    two-level draw (its 16-entry blocks raced on their masses,
//                    the entry of a block by inverse CDF).  Output: one partial
//                    per (request, slice); no logit ever reaches global memory.
//   draft_reduce     one CTA per request merges its partials in a fixed order
//                    (deterministic), writes x_k, log q_k(x_k), lse_k and the
//                    confidence c_k.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "rnn_step.cuh"

namespace dspark {

namespace {

constexpr int kSliceV = 64;     // vocabulary entries per CTA
constexpr int kRowsPerPass = 8; // requests per pass over the slice
constexpr int kThreads = 128;   // 16 vocabulary quads x 8 requests

template <typename T, bool kRnn>
__global__ void __launch_bounds__(kThreads) draft_step_simt(const DraftStep p) {
    extern __shared__ float smem[];
    const int r = p.r, ld = r + 1;
    float *W2s = smem;                    // [64][r + 1]
    float *Es = smem + kSliceV * ld;      // [8][r + 1]
    const T *W2t = static_cast<const T *>(p.W2t);
    const T *W1 = static_cast<const T *>(p.W1);
    const T *U = static_cast<const T *>(p.U);
    const int slice = blockIdx.x, vbase = slice * kSliceV;

    for (int e = threadIdx.x; e < kSliceV * r; e += kThreads) {
        const int vv = e / r, i = e - vv * r, v = vbase + vv;
        W2s[vv * ld + i] = v < p.V ? to_f32(W2t[(size_t)v * r + i]) : 0.f;
    }
    const int quad = threadIdx.x & 15, sub = threadIdx.x >> 4;
    const int v0 = vbase + quad * 4;
    const PhiloxKey key = philox_key(p.seed);
    const uint32_t c3 = philox_ctr3(p.cycle, 0);

    for (int row0 = 0; row0 < p.R; row0 += kRowsPerPass) {
        __syncthreads();
        for (int e = threadIdx.x; e < kRowsPerPass * r; e += kThreads) {
            const int rr = e / r, i = e - rr * r, row = row0 + rr;
            float val = 0.f;
            if (row < p.R) {
                if (kRnn) {
                    val = p.A_op[(size_t)row * p.a_stride + i];
                } else {
                    int xp = p.x_prev[(size_t)row * p.x_stride];
                    if (xp < 0 || xp >= p.V) {
                        if (i == 0) set_err(p.err, DSPARK_ERR_RANGE);
                        xp = 0;
                    }
                    val = to_f32(W1[(size_t)xp * r + i]);
                }
            }
            Es[rr * ld + i] = val;
        }
        __syncthreads();

        const int row = row0 + sub;
        const float *e = Es + sub * ld;
        const float *w0 = W2s + (quad * 4) * ld;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < r; ++i) {
            const float ev = e[i];
            acc[0] = fmaf(ev, w0[i], acc[0]);
            acc[1] = fmaf(ev, w0[ld + i], acc[1]);
            acc[2] = fmaf(ev, w0[2 * ld + i], acc[2]);
            acc[3] = fmaf(ev, w0[3 * ld + i], acc[3]);
        }
        // Four lanes (quads 4i .. 4i + 3) hold vocabulary block b = v0 / 16 of this
        // request: the block's maximum and quad sums by shuffles, the same block
        // sum and race score in each of the four, then level 2 of the draw from
        // the block's aligned sums; the lane whose quad holds the drawn entry
        // keeps the block as its candidate.  Entries at or beyond V carry
        // z = -inf (weight 0); a block wholly beyond V has no mass.
        RowState st;
        row_init(st);
        {
            const T *Urow = U + ((size_t)min(row, p.R - 1) * p.gamma + (p.k - 1)) * (size_t)p.V;
            float z[4], e[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) z[j] = (v0 + j < p.V) ? acc[j] + to_f32(Urow[v0 + j]) : -INFINITY;
            float mb = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const float mL = mb * kLog2e;
#pragma unroll
            for (int j = 0; j < 4; ++j) e[j] = mb == -INFINITY ? 0.f : ex2(fmaf(z[j], kLog2e, -mL));
            const float p0 = e[0] + e[1], p1 = e[2] + e[3], qs = p0 + p1;
            const int base = threadIdx.x & ~3;
            float q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = __shfl_sync(0xffffffffu, qs, base + i);
            const float o0 = q[0] + q[1], o1 = q[2] + q[3], Sb = o0 + o1;
            if (row < p.R && mb > -INFINITY && Sb > 0.f) {
                st.m = mb;
                st.mL = mL;
                st.S = qs;  // the request's sum over the slice is the sum of its quads
                const int vb = v0 & ~15, qi_self = quad & 3;
                const uint4 words = philox4x32_10(
                    make_uint4((uint32_t)(vb >> 5), (uint32_t)p.k, (uint32_t)row, c3), key);
                const bool odd = (vb & 16) != 0;
                const uint32_t wr = odd ? words.z : words.x, we = odd ? words.w : words.y;
                const float score = mb + kLn2 * lg2(Sb) - log_exp_variate(one_minus_uniform(wr));
                float t = uniform_of(we) * Sb;
                const bool r1 = t >= o0 && o1 > 0.f;
                t = r1 ? t - o0 : t;
                const float qL = r1 ? q[2] : q[0], qR = r1 ? q[3] : q[1];
                const bool r2 = t >= qL && qR > 0.f;
                t = r2 ? t - qL : t;
                if (((r1 ? 2 : 0) | (r2 ? 1 : 0)) == qi_self) {
                    const bool r3 = t >= p0 && p1 > 0.f;
                    t = r3 ? t - p0 : t;
                    const float eL = r3 ? e[2] : e[0], eR = r3 ? e[3] : e[1];
                    const int j = 2 * (r3 ? 1 : 0) + (t >= eL && eR > 0.f ? 1 : 0);
                    st.best = score;
                    st.idx = v0 + j;
                    st.zbest = select_of(z, j);
                }
            }
        }
        // merge the 16 quads of this request (lanes differing in bits 0..3)
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
            const float m = __shfl_xor_sync(0xffffffffu, st.m, off);
            const float S = __shfl_xor_sync(0xffffffffu, st.S, off);
            const float b = __shfl_xor_sync(0xffffffffu, st.best, off);
            const float zb = __shfl_xor_sync(0xffffffffu, st.zbest, off);
            const int ix = __shfl_xor_sync(0xffffffffu, st.idx, off);
            row_merge(st, m, S, b, zb, ix);
        }
        if (quad == 0 && row < p.R)
            p.part[(size_t)row * p.nparts + slice] = make_partial(st.m, st.S, st.best, st.zbest, st.idx);
    }
}

constexpr int kReduceThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kReduceThreads) draft_reduce_kernel(const DraftReduce p) {
    __shared__ float s_m[kReduceThreads], s_S[kReduceThreads], s_b[kReduceThreads],
        s_z[kReduceThreads], s_dot[kReduceThreads];
    __shared__ int s_i[kReduceThreads];
    const int row = blockIdx.x, tid = threadIdx.x;
    RowState st;
    row_init(st);
    for (int t = tid; t < p.nparts; t += kReduceThreads) {
        const DraftPartial q = p.part[(size_t)row * p.nparts + t];
        row_merge(st, q.m, q.S, q.best, q.zbest, q.idx);
    }
    // confidence logit w^T [h_k ; W_1[x_{k-1}]]
    int xp = p.x_prev[(size_t)row * p.x_stride];
    if (xp < 0 || xp >= p.V) xp = 0;  // reported by the step kernel
    const T *h = static_cast<const T *>(p.h) + ((size_t)row * p.gamma + (p.k - 1)) * (size_t)p.d;
    const T *e = static_cast<const T *>(p.W1) + (size_t)xp * p.r;
    float dot = 0.f;
    for (int j = tid; j < p.d; j += kReduceThreads) dot = fmaf(p.w[j], to_f32(h[j]), dot);
    for (int i = tid; i < p.r; i += kReduceThreads) dot = fmaf(p.w[p.d + i], to_f32(e[i]), dot);

    s_m[tid] = st.m; s_S[tid] = st.S; s_b[tid] = st.best; s_z[tid] = st.zbest; s_i[tid] = st.idx;
    s_dot[tid] = dot;
    __syncthreads();
    for (int half = kReduceThreads / 2; half > 0; half >>= 1) {
        if (tid < half) {
            RowState a{s_m[tid], s_m[tid] * kLog2e, s_S[tid], s_b[tid], s_z[tid], s_i[tid]};
            row_merge(a, s_m[tid + half], s_S[tid + half], s_b[tid + half], s_z[tid + half],
                      s_i[tid + half]);
            s_m[tid] = a.m; s_S[tid] = a.S; s_b[tid] = a.best; s_z[tid] = a.zbest; s_i[tid] = a.idx;
            s_dot[tid] += s_dot[tid + half];
        }
        __syncthreads();
    }
    if (tid == 0) {
        const size_t o = (size_t)row * p.gamma + (p.k - 1);
        float lse = s_m[0] + logf(s_S[0]);
        int idx = s_i[0];
        if (idx < 0 || !isfinite(lse)) {
            set_err(p.err, DSPARK_ERR_NONFINITE);
            idx = 0;
        }
        p.x[o] = idx;
        p.lse[o] = lse;
        p.logq[o] = s_z[0] - lse;
        const float T_k = p.sts_T ? p.sts_T[p.k - 1] : 1.0f;
        p.c[o] = 1.0f / (1.0f + expf(-s_dot[0] / T_k));
        if (p.conf_logit) p.conf_logit[o] = s_dot[0];
    }
}

// ---------------------------------------------------------------- RNN head
template <typename T>
__global__ void __launch_bounds__(256) rnn_hproj_kernel(int M, int d, int r, const T *h, const T *W,
                                                        float *Hpre) {
    __shared__ float As[16][68], Bs[16][68];
    const int N = 3 * r, ldw = 2 * r + d;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += 16) {
        for (int e = threadIdx.x; e < 1024; e += 256) {
            const int mm = e >> 4, kk = e & 15;
            As[kk][mm] = (m0 + mm < M && k0 + kk < d) ? to_f32(h[(size_t)(m0 + mm) * d + k0 + kk]) : 0.f;
            Bs[kk][mm] = (n0 + mm < N && k0 + kk < d)
                             ? to_f32(W[(size_t)(n0 + mm) * ldw + 2 * r + k0 + kk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
            if (m < M && n < N) Hpre[(size_t)m * N + n] = acc[i][j];
        }
}

// One step of eq. (6) after the h_k part, one tile (rnn_step.cuh) per CTA.
// The state is double-buffered (s_in -> s_out) since every CTA reads whole
// rows of s_{k-1}.
struct CtaSync {
    __device__ void operator()() const { __syncthreads(); }
};

template <typename T>
__global__ void __launch_bounds__(rnn::kThreads, 1) rnn_step_kernel(const RnnStep p) {
    extern __shared__ float sh[];
    rnn::step_tile<T>(p, sh, blockIdx.x * rnn::kIB, blockIdx.y * rnn::kRB, threadIdx.x, CtaSync{});
}

}  // namespace

int draft_step_nparts(int V) { return (V + kSliceV - 1) / kSliceV; }

template <typename T, bool kRnn>
static cudaError_t launch_step_t(const DraftStep &p, cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)(kSliceV + kRowsPerPass) * (p.r + 1);
    auto kern = draft_step_simt<T, kRnn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<p.nparts, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_draft_step(const DraftStep &p, cudaStream_t s) {
    const bool rnn = p.A_op != nullptr;
    if (p.dtype == DSPARK_BF16)
        return rnn ? launch_step_t<__nv_bfloat16, true>(p, s) : launch_step_t<__nv_bfloat16, false>(p, s);
    return rnn ? launch_step_t<float, true>(p, s) : launch_step_t<float, false>(p, s);
}

cudaError_t launch_draft_reduce(const DraftReduce &p, cudaStream_t s) {
    if (p.dtype == DSPARK_BF16)
        draft_reduce_kernel<__nv_bfloat16><<<p.R, kReduceThreads, 0, s>>>(p);
    else
        draft_reduce_kernel<float><<<p.R, kReduceThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rnn_hproj(int M, int d, int r, int dtype, const void *h, const void *W,
                             float *Hpre, cudaStream_t s) {
    dim3 grid((3 * r + 63) / 64, (M + 63) / 64);
    if (dtype == DSPARK_BF16)
        rnn_hproj_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            M, d, r, static_cast<const __nv_bfloat16 *>(h), static_cast<const __nv_bfloat16 *>(W), Hpre);
    else
        rnn_hproj_kernel<float><<<grid, 256, 0, s>>>(M, d, r, static_cast<const float *>(h),
                                                     static_cast<const float *>(W), Hpre);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_rnn_step_t(const RnnStep &p, cudaStream_t s) {
    const size_t smem = rnn::tile_smem_bytes(p.r);
    auto kern = rnn_step_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((p.r + rnn::kIB - 1) / rnn::kIB, (p.R + rnn::kRB - 1) / rnn::kRB);
    kern<<<grid, rnn::kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rnn_step(const RnnStep &p, cudaStream_t s) {
    // 16 requests x 8 entries per CTA (512 threads; 83 KB of shared memory at r = 256)
    if (p.dtype == DSPARK_BF16) return launch_rnn_step_t<__nv_bfloat16>(p, s);
    return launch_rnn_step_t<float>(p, s);
}

}  // namespace dspark
