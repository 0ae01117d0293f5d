// verify.cu -- lossless verification over the flattened variable-length batch.
//
// "DSpark explained", section 06: draw x ~ q, accept with probability
// min(1, p(x)/q(x)), otherwise resample from norm(max(0, p - q)); along a
// block the rule runs position by position and stops at the first rejection
// (DSpark digest, overview step 3).  Rows of the target batch are tagged with
// (request, position) as in the digest's production section.
//
// Three launches:
//   verify_phase1  one CTA per flattened row: log-sum-exp of the target row,
//                  log p of the drafted token, the Philox acceptance test, and
//                  an atomicMin of rejected positions per request (min is order
//                  independent, so the result is deterministic).
//   verify_phase2  vocabulary-sliced like the draft step: per request it
//                  recomputes q at the first rejected position (U + bias operand
//                  x W_2, never stored) and races over max(0, p - q) and over p.
//   verify_final   one CTA per request merges the slices and writes the
//                  accepted tokens, the correction / bonus token and the anchor.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "verify_common.cuh"

namespace dspark {

namespace {

constexpr int kSliceV = 64;
constexpr int kRowsPerPass = 8;
constexpr int kThreads = 128;
constexpr int kNone = 0x7fffffff;

__global__ void verify_init(int R, int gamma, VerifyWs w) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < R * (gamma + 1)) w.row_of[i] = -1;
    if (i < kVerifyMaxMTiles) w.done[i] = 0;
    if (i < R) {
        w.first_rej[i] = kNone;
        w.ell[i] = -1;
        w.win[i] = 0ull;
    }
}

template <typename T>
__device__ __forceinline__ void feed_lse(float &m, float &S, const float *x, int n) {
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < n; ++j) cm = fmaxf(cm, x[j]);
    if (cm > m) {
        S *= ex2((m - cm) * kLog2e);
        m = cm;
    }
    const float mL = m * kLog2e;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < n; ++j) acc += ex2(fmaf(x[j], kLog2e, -mL));
    S += acc;
}

template <typename T>
__global__ void __launch_bounds__(256) verify_phase1(const dspark_verify_args a, VerifyWs w) {
    const int i = blockIdx.x, tid = threadIdx.x;
    const int N = a.N_dev ? min(*a.N_dev, a.N) : a.N;
    if (i >= N) return;
    const int rq = a.tags[2 * i], pos = a.tags[2 * i + 1];
    bool ok = rq >= 0 && rq < a.R && pos >= 0 && pos <= a.gamma;
    if (ok) {
        if (pos == 0)
            ok = (i == 0) || a.tags[2 * (i - 1)] != rq;
        else
            ok = i > 0 && a.tags[2 * (i - 1)] == rq && a.tags[2 * (i - 1) + 1] == pos - 1;
    }
    if (!ok) {
        if (tid == 0) set_err(a.err, DSPARK_ERR_INVAL);
        return;
    }
    const T *row = static_cast<const T *>(a.T) + (size_t)i * a.V;
    float m = -INFINITY, S = 0.f;
    constexpr int kVec = 16 / sizeof(T);
    if (a.V % kVec == 0) {
        const uint4 *row4 = reinterpret_cast<const uint4 *>(row);
        const int nv = a.V / kVec;
        const uint64_t pol = tc::policy_evict_first();  // each target row is read once here
        // kLoads 16-byte loads in flight per thread, then one max / rescale for all of them
        constexpr int kLoads = 4;
        const int step = kLoads * (int)blockDim.x;
        int c0 = tid;
        for (; c0 + (kLoads - 1) * (int)blockDim.x < nv; c0 += step) {
            uint4 raw[kLoads];
#pragma unroll
            for (int q = 0; q < kLoads; ++q) raw[q] = tc::ld_global_hint(row4 + c0 + q * blockDim.x, pol);
            float x[kLoads * kVec];
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const T *vals = reinterpret_cast<const T *>(&raw[q]);
#pragma unroll
                for (int j = 0; j < kVec; ++j) x[q * kVec + j] = to_f32(vals[j]);
            }
            feed_lse<T>(m, S, x, kLoads * kVec);
        }
        for (int c = c0; c < nv; c += blockDim.x) {
            const uint4 raw = tc::ld_global_hint(row4 + c, pol);
            const T *vals = reinterpret_cast<const T *>(&raw);
            float x[kVec];
#pragma unroll
            for (int j = 0; j < kVec; ++j) x[j] = to_f32(vals[j]);
            feed_lse<T>(m, S, x, kVec);
        }
    } else {
        for (int v = tid; v < a.V; v += blockDim.x) {
            const float x = to_f32(row[v]);
            feed_lse<T>(m, S, &x, 1);
        }
    }
    __shared__ float s_m[256], s_S[256];
    s_m[tid] = m;
    s_S[tid] = S;
    __syncthreads();
    for (int half = blockDim.x / 2; half > 0; half >>= 1) {
        if (tid < half) {
            const float m2 = s_m[tid + half], S2 = s_S[tid + half];
            const float M = fmaxf(s_m[tid], m2);
            s_S[tid] = M == -INFINITY ? 0.f
                                      : s_S[tid] * ex2((s_m[tid] - M) * kLog2e) + S2 * ex2((m2 - M) * kLog2e);
            s_m[tid] = M;
        }
        __syncthreads();
    }
    if (tid != 0) return;
    const float lse = s_m[0] + logf(s_S[0]);
    w.lse_p[i] = lse;
    if (a.lse_p) a.lse_p[i] = lse;
    if (atomicCAS(&w.row_of[rq * (a.gamma + 1) + pos], -1, i) != -1) set_err(a.err, DSPARK_ERR_INVAL);
    const bool test = pos < a.gamma && i + 1 < N && a.tags[2 * (i + 1)] == rq;
    if (test) {
        const int tok = a.x[(size_t)rq * a.gamma + pos];
        if (tok < 0 || tok >= a.V) {
            set_err(a.err, DSPARK_ERR_RANGE);
            if (a.logp) a.logp[i] = NAN;
            atomicMin(&w.first_rej[rq], pos);
            return;
        }
        const float logp = to_f32(row[tok]) - lse;
        const uint4 words = philox4x32_10(
            make_uint4(0u, (uint32_t)pos, (uint32_t)rq, philox_ctr3(a.cycle, 1)), philox_key(a.seed));
        const float u = uniform_of(words.x);
        const bool accept = logf(u) < logp - a.logq[(size_t)rq * a.gamma + pos];
        if (!accept) atomicMin(&w.first_rej[rq], pos);
        if (a.logp) a.logp[i] = logp;
    } else {
        w.ell[rq] = pos;
        if (a.logp) a.logp[i] = NAN;
    }
}

struct RowMeta {
    int residual;   // 1: residual race needed, 0: bonus (p only), -1: skip
    int n;          // position of the final sample
    int row;        // flattened row of that position
    float lse_p, lse_q;
};

template <typename T, bool kRnn>
__global__ void __launch_bounds__(kThreads) verify_phase2(const dspark_verify_args a, VerifyWs w) {
    extern __shared__ float smem[];
    const int r = a.r, ld = r + 1;
    float *W2s = smem;
    float *Es = smem + kSliceV * ld;
    __shared__ RowMeta meta[kRowsPerPass];
    const T *W2t = static_cast<const T *>(a.W2t);
    const T *W1 = static_cast<const T *>(a.W1);
    const T *U = static_cast<const T *>(a.U);
    const T *Tm = static_cast<const T *>(a.T);
    const int slice = blockIdx.x, vbase = slice * kSliceV;
    for (int e = threadIdx.x; e < kSliceV * r; e += kThreads) {
        const int vv = e / r, i = e - vv * r, v = vbase + vv;
        W2s[vv * ld + i] = v < a.V ? to_f32(W2t[(size_t)v * r + i]) : 0.f;
    }
    const int quad = threadIdx.x & 15, sub = threadIdx.x >> 4;
    const int v0 = vbase + quad * 4;
    const PhiloxKey key = philox_key(a.seed);
    const uint32_t c3 = philox_ctr3(a.cycle, 2);

    for (int row0 = 0; row0 < a.R; row0 += kRowsPerPass) {
        __syncthreads();
        if (threadIdx.x < kRowsPerPass) {
            const int rq = row0 + threadIdx.x;
            RowMeta mt{-1, 0, 0, 0.f, 0.f};
            if (rq < a.R) {
                const int ell = w.ell[rq];
                if (ell >= 0) {
                    const int fr = w.first_rej[rq];
                    mt.residual = fr < ell ? 1 : 0;
                    mt.n = fr < ell ? fr : ell;
                    mt.row = w.row_of[rq * (a.gamma + 1) + mt.n];
                    if (mt.row < 0) {
                        mt.residual = -1;
                    } else {
                        mt.lse_p = w.lse_p[mt.row];
                        if (mt.residual) mt.lse_q = a.lse[(size_t)rq * a.gamma + mt.n];
                    }
                } else if (slice == 0) {
                    set_err(a.err, DSPARK_ERR_INVAL);  // request missing from the batch
                }
            }
            meta[threadIdx.x] = mt;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kRowsPerPass * r; e += kThreads) {
            const int rr = e / r, i = e - rr * r, rq = row0 + rr;
            float val = 0.f;
            const RowMeta mt = meta[rr];
            if (rq < a.R && mt.residual == 1) {
                if (kRnn) {
                    val = a.A[((size_t)rq * a.gamma + mt.n) * (size_t)r + i];
                } else {
                    int xn = mt.n == 0 ? a.anchor[rq] : a.x[(size_t)rq * a.gamma + mt.n - 1];
                    if (xn < 0 || xn >= a.V) xn = 0;
                    val = to_f32(W1[(size_t)xn * r + i]);
                }
            }
            Es[rr * ld + i] = val;
        }
        __syncthreads();

        const int rq = row0 + sub;
        const RowMeta mt = meta[sub];
        Race res, pr;
        race_init(res);
        race_init(pr);
        if (rq < a.R && mt.residual >= 0 && v0 < a.V) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (mt.residual) {
                const float *e = Es + sub * ld;
                const float *w0 = W2s + (quad * 4) * ld;
                for (int i = 0; i < r; ++i) {
                    const float ev = e[i];
                    acc[0] = fmaf(ev, w0[i], acc[0]);
                    acc[1] = fmaf(ev, w0[ld + i], acc[1]);
                    acc[2] = fmaf(ev, w0[2 * ld + i], acc[2]);
                    acc[3] = fmaf(ev, w0[3 * ld + i], acc[3]);
                }
            }
            const uint4 words = philox4x32_10(
                make_uint4((uint32_t)(v0 >> 2), (uint32_t)mt.n, (uint32_t)rq, c3), key);
            const T *trow = Tm + (size_t)mt.row * a.V;
            const T *urow = U + ((size_t)rq * a.gamma + mt.n) * (size_t)a.V;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = v0 + j;
                if (v >= a.V) continue;
                const float t = one_minus_uniform(word_lane(words, j));
                const float p = ex2((to_f32(trow[v]) - mt.lse_p) * kLog2e);
                race_feed(pr, p, t, v);
                if (mt.residual) {
                    const float q = ex2((acc[j] + to_f32(urow[v]) - mt.lse_q) * kLog2e);
                    race_feed(res, fmaxf(p - q, 0.f), t, v);
                }
            }
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
            const float b1 = __shfl_xor_sync(0xffffffffu, res.best, off);
            const int i1 = __shfl_xor_sync(0xffffffffu, res.idx, off);
            const float b2 = __shfl_xor_sync(0xffffffffu, pr.best, off);
            const int i2 = __shfl_xor_sync(0xffffffffu, pr.idx, off);
            race_merge(res.best, res.idx, b1, i1);
            race_merge(pr.best, pr.idx, b2, i2);
        }
        if (quad == 0 && rq < a.R)
            w.part[(size_t)rq * w.nparts + slice] = VerifyPartial{res.best, pr.best, res.idx, pr.idx};
    }
}

__global__ void __launch_bounds__(256) verify_final(const dspark_verify_args a, VerifyWs w) {
    __shared__ float s_b1[256], s_b2[256];
    __shared__ int s_i1[256], s_i2[256];
    const int rq = blockIdx.x, tid = threadIdx.x;
    float b1 = -INFINITY, b2 = -INFINITY;
    int i1 = -1, i2 = -1;
    for (int t = tid; t < w.nparts; t += blockDim.x) {
        const VerifyPartial q = w.part[(size_t)rq * w.nparts + t];
        race_merge(b1, i1, q.best_res, q.idx_res);
        race_merge(b2, i2, q.best_p, q.idx_p);
    }
    s_b1[tid] = b1; s_i1[tid] = i1; s_b2[tid] = b2; s_i2[tid] = i2;
    __syncthreads();
    for (int half = blockDim.x / 2; half > 0; half >>= 1) {
        if (tid < half) {
            race_merge(s_b1[tid], s_i1[tid], s_b1[tid + half], s_i1[tid + half]);
            race_merge(s_b2[tid], s_i2[tid], s_b2[tid + half], s_i2[tid + half]);
        }
        __syncthreads();
    }
    // A rejected position whose residual max(0, p - q) came out empty (p equal to
    // q to rounding everywhere) samples p instead, with the same stream-2 noise:
    // when the slices did not run that race, this CTA runs it over the whole row.
    __shared__ int s_fallback;
    if (tid == 0) {
        const int ell = w.ell[rq];
        s_fallback = ell >= 0 && w.first_rej[rq] < ell && s_i1[0] < 0 && s_i2[0] < 0;
    }
    __syncthreads();
    if (s_fallback) {
        const int n = w.first_rej[rq];
        const int row = w.row_of[rq * (a.gamma + 1) + n];
        Race pr;
        race_init(pr);
        if (row >= 0) {
            const float lsep = w.lse_p[row] * kLog2e;
            const PhiloxKey key = philox_key(a.seed);
            const uint32_t c3 = philox_ctr3(a.cycle, 2);
            for (int v0 = 4 * tid; v0 < a.V; v0 += 4 * blockDim.x) {
                const uint4 words =
                    philox4x32_10(make_uint4((uint32_t)(v0 >> 2), (uint32_t)n, (uint32_t)rq, c3), key);
                for (int j = 0; j < 4 && v0 + j < a.V; ++j) {
                    const size_t at = (size_t)row * a.V + v0 + j;
                    const float tv = a.dtype == DSPARK_BF16
                                         ? __bfloat162float(static_cast<const __nv_bfloat16 *>(a.T)[at])
                                         : static_cast<const float *>(a.T)[at];
                    race_feed(pr, ex2(fmaf(tv, kLog2e, -lsep)), one_minus_uniform(word_lane(words, j)), v0 + j);
                }
            }
        }
        __syncthreads();
        s_b2[tid] = pr.best;
        s_i2[tid] = pr.idx;
        __syncthreads();
        for (int half = blockDim.x / 2; half > 0; half >>= 1) {
            if (tid < half) race_merge(s_b2[tid], s_i2[tid], s_b2[tid + half], s_i2[tid + half]);
            __syncthreads();
        }
    }
    if (tid != 0) return;
    write_outcome(a, w, rq, s_i1[0], s_i2[0]);
}

template <typename T, bool kRnn>
cudaError_t launch_phase2(const dspark_verify_args &a, const VerifyWs &w, cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)(kSliceV + kRowsPerPass) * (a.r + 1);
    auto kern = verify_phase2<T, kRnn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<w.nparts, kThreads, smem, s>>>(a, w);
    return cudaGetLastError();
}

}  // namespace

size_t verify_ws_bytes(int R, int gamma, int V, int N) {
    const int nparts = (V + kSliceV - 1) / kSliceV;
    return align256(sizeof(float) * (size_t)N) + align256(sizeof(int32_t) * (size_t)R) * 2 +
           align256(sizeof(int32_t) * (size_t)R * (gamma + 1)) +
           align256(sizeof(VerifyPartial) * (size_t)R * nparts) + align256(sizeof(int) * kVerifyMaxMTiles) +
           align256(sizeof(unsigned long long) * (size_t)R);
}

VerifyWs verify_ws_carve(void *ws, int R, int gamma, int V, int N) {
    char *p = static_cast<char *>(ws);
    VerifyWs w;
    w.nparts = (V + kSliceV - 1) / kSliceV;
    w.lse_p = reinterpret_cast<float *>(p);
    p += align256(sizeof(float) * (size_t)N);
    w.first_rej = reinterpret_cast<int32_t *>(p);
    p += align256(sizeof(int32_t) * (size_t)R);
    w.ell = reinterpret_cast<int32_t *>(p);
    p += align256(sizeof(int32_t) * (size_t)R);
    w.row_of = reinterpret_cast<int32_t *>(p);
    p += align256(sizeof(int32_t) * (size_t)R * (gamma + 1));
    w.part = reinterpret_cast<VerifyPartial *>(p);
    p += align256(sizeof(VerifyPartial) * (size_t)R * w.nparts);
    w.done = reinterpret_cast<int *>(p);
    p += align256(sizeof(int) * kVerifyMaxMTiles);
    w.win = reinterpret_cast<unsigned long long *>(p);
    return w;
}

cudaError_t launch_verify(const dspark_verify_args &a, const VerifyWs &w, cudaStream_t s) {
    const int n_init = a.R * (a.gamma + 1) > kVerifyMaxMTiles ? a.R * (a.gamma + 1) : kVerifyMaxMTiles;  // >= R
    verify_init<<<(n_init + 255) / 256, 256, 0, s>>>(a.R, a.gamma, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.N > 0) {
        if (a.dtype == DSPARK_BF16)
            verify_phase1<__nv_bfloat16><<<a.N, 256, 0, s>>>(a, w);
        else
            verify_phase1<float><<<a.N, 256, 0, s>>>(a, w);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const bool rnn = a.A != nullptr;
    VerifyWs wf = w;  // the tensor-core path sets its own partial count
    if (verify_tc_supported(a)) {
        // the last CTA of each M-tile merges the slices and writes the outcome itself
        e = launch_verify_phase2_tc(a, wf, s);
        return e;
    }
    if (a.dtype == DSPARK_BF16)
        e = rnn ? launch_phase2<__nv_bfloat16, true>(a, w, s) : launch_phase2<__nv_bfloat16, false>(a, w, s);
    else
        e = rnn ? launch_phase2<float, true>(a, w, s) : launch_phase2<float, false>(a, w, s);
    if (e != cudaSuccess) return e;
    verify_final<<<a.R, 256, 0, s>>>(a, wf);
    return cudaGetLastError();
}

}  // namespace dspark
