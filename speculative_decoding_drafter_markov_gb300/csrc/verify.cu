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
//                  x W_2, never stored) and sums max(0, p - q) and p per slice.
//   verify_final   one warp per request: the inverse-CDF draw of the correction
//                  (or bonus) token over the slice sums, then over the chosen
//                  slice's weights recomputed with phase 2's arithmetic, and the
//                  accepted tokens, that token and the anchor.
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

__global__ void verify_init(int R, int gamma, VerifyWs w, int ttot_words) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    // the tensor-core phase adds into its tile sums: zero them (16 bytes a store)
    for (int j = i; 2 * j < ttot_words; j += gridDim.x * blockDim.x)
        reinterpret_cast<uint4 *>(w.ttot)[j] = make_uint4(0u, 0u, 0u, 0u);
    if (i < R * (gamma + 1)) w.row_of[i] = -1;
    if (i < kVerifyMaxMTiles) {
        w.done[i] = 0;
        w.tctr[i] = 0;
    }
    if (i < R) {
        w.first_rej[i] = kNone;
        w.ell[i] = -1;
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
    int residual;   // 1: residual draw, 0: bonus (p only), -1: skip
    int n;          // position of the final sample
    int row;        // flattened row of that position
    float lse_p, lse_q;
};

// The weights of vocabulary entries v0 .. v0 + 3 of one request: the residual
// max(0, p - q) (zero unless the request rejected) and p; entries at or beyond V
// weigh zero.  w2 points at the staged W_2^T row of v0 (rows ld apart), e at
// the bias operand (W_1[x_n] or A_{n+1}); the same arithmetic serves the slice
// sums and the final search, so both see the same weights.
template <typename T, bool kRnn>
__device__ __forceinline__ void slice_weights(const dspark_verify_args &a, const RowMeta &mt, const float *w2,
                                              const float *e, int ld, int rq, int v0, float (&wr)[4],
                                              float (&wp)[4]) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (mt.residual == 1) {
        for (int i = 0; i < a.r; ++i) {
            const float ev = e[i];
            acc[0] = fmaf(ev, w2[i], acc[0]);
            acc[1] = fmaf(ev, w2[ld + i], acc[1]);
            acc[2] = fmaf(ev, w2[2 * ld + i], acc[2]);
            acc[3] = fmaf(ev, w2[3 * ld + i], acc[3]);
        }
    }
    const T *trow = static_cast<const T *>(a.T) + (size_t)mt.row * a.V;
    const T *urow = static_cast<const T *>(a.U) + ((size_t)rq * a.gamma + mt.n) * (size_t)a.V;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int v = v0 + j;
        wr[j] = wp[j] = 0.f;
        if (v >= a.V) continue;
        const float p = ex2((to_f32(trow[v]) - mt.lse_p) * kLog2e);
        wp[j] = p;
        if (mt.residual == 1) {
            const float q = ex2((acc[j] + to_f32(urow[v]) - mt.lse_q) * kLog2e);
            wr[j] = fmaxf(p - q, 0.f);
        }
    }
}

template <typename T, bool kRnn>
__global__ void __launch_bounds__(kThreads) verify_phase2(const dspark_verify_args a, VerifyWs w) {
    extern __shared__ float smem[];
    const int r = a.r, ld = r + 1;
    float *W2s = smem;
    float *Es = smem + kSliceV * ld;
    __shared__ RowMeta meta[kRowsPerPass];
    const T *W2t = static_cast<const T *>(a.W2t);
    const T *W1 = static_cast<const T *>(a.W1);
    const int slice = blockIdx.x, vbase = slice * kSliceV;
    for (int e = threadIdx.x; e < kSliceV * r; e += kThreads) {
        const int vv = e / r, i = e - vv * r, v = vbase + vv;
        W2s[vv * ld + i] = v < a.V ? to_f32(W2t[(size_t)v * r + i]) : 0.f;
    }
    const int quad = threadIdx.x & 15, sub = threadIdx.x >> 4;
    const int v0 = vbase + quad * 4;

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
        float sres = 0.f, sp = 0.f;  // this thread's 4 weights of the two draws
        if (rq < a.R && mt.residual >= 0 && v0 < a.V) {
            float wr[4], wp[4];
            slice_weights<T, kRnn>(a, mt, W2s + (quad * 4) * ld, Es + sub * ld, ld, rq, v0, wr, wp);
            sres = (wr[0] + wr[1]) + (wr[2] + wr[3]);
            sp = (wp[0] + wp[1]) + (wp[2] + wp[3]);
        }
        // the slice's sums over its 16 quads (a fixed tree)
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) {
            sres += __shfl_xor_sync(0xffffffffu, sres, off);
            sp += __shfl_xor_sync(0xffffffffu, sp, off);
        }
        if (quad == 0 && rq < a.R) w.part[(size_t)rq * w.nparts + slice] = VerifyPartial{sres, sp};
    }
}

// One warp per request: the correction / bonus draw by inverse CDF over the
// slice sums, then over the 64 weights of the chosen slice, recomputed with the
// same arithmetic as phase 2.  A rejected position whose residual max(0, p - q)
// came out empty (p equal to q to rounding everywhere) draws from p instead.
template <typename T, bool kRnn>
__global__ void __launch_bounds__(32) verify_final(const dspark_verify_args a, VerifyWs w) {
    __shared__ float Es[512];  // the bias operand (r <= 512)
    const int rq = blockIdx.x, lane = threadIdx.x;
    const int ell = w.ell[rq];
    if (ell < 0) {
        if (lane == 0) write_outcome(a, w, rq, -1, -1);
        return;
    }
    const int fr = w.first_rej[rq];
    RowMeta mt;
    mt.residual = fr < ell ? 1 : 0;
    mt.n = fr < ell ? fr : ell;
    mt.row = w.row_of[rq * (a.gamma + 1) + mt.n];
    if (mt.row < 0) {
        if (lane == 0) write_outcome(a, w, rq, -1, -1);
        return;
    }
    mt.lse_p = w.lse_p[mt.row];
    mt.lse_q = mt.residual ? a.lse[(size_t)rq * a.gamma + mt.n] : 0.f;
    const VerifyPartial *part = w.part + (size_t)rq * w.nparts;
    // the residual's total decides whether its draw is possible
    float below = 0.f, total = 0.f;
    bool use_res = mt.residual == 1;
    if (use_res) {
        warp_cdf_search(w.nparts, 0.f, INFINITY, [&](int i) { return part[i].sum_res; }, &below, &total);
        use_res = total > 0.f;
    }
    if (!use_res) warp_cdf_search(w.nparts, 0.f, INFINITY, [&](int i) { return part[i].sum_p; }, &below, &total);
    const float target = correction_uniform(a.seed, a.cycle, mt.n, rq) * total;
    const int sl = use_res ? warp_cdf_search(w.nparts, 0.f, target, [&](int i) { return part[i].sum_res; }, &below)
                           : warp_cdf_search(w.nparts, 0.f, target, [&](int i) { return part[i].sum_p; }, &below);
    int y = -1;
    if (sl >= 0) {
        // the slice's 64 weights: lane l takes entries 4 (l % 16) .. + 3 (lanes 16-31 repeat them)
        const int r = a.r, vbase = sl * kSliceV;
        const T *W2t = static_cast<const T *>(a.W2t);
        if (use_res) {
            for (int i = lane; i < r; i += 32) {
                float val;
                if (kRnn) {
                    val = a.A[((size_t)rq * a.gamma + mt.n) * (size_t)r + i];
                } else {
                    int xn = mt.n == 0 ? a.anchor[rq] : a.x[(size_t)rq * a.gamma + mt.n - 1];
                    if (xn < 0 || xn >= a.V) xn = 0;
                    val = to_f32(static_cast<const T *>(a.W1)[(size_t)xn * r + i]);
                }
                Es[i] = val;
            }
        }
        float wv[4] = {0.f, 0.f, 0.f, 0.f};
        const int quad = lane & 15, v0 = vbase + 4 * quad;
        {
            // the quad's weights, W_2^T read from global memory in phase 2's order
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            __syncwarp();
            if (use_res) {
                for (int i = 0; i < r; ++i) {
                    const float ev = Es[i];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (v0 + j < a.V) acc[j] = fmaf(ev, to_f32(W2t[(size_t)(v0 + j) * r + i]), acc[j]);
                }
            }
            const T *trow = static_cast<const T *>(a.T) + (size_t)mt.row * a.V;
            const T *urow = static_cast<const T *>(a.U) + ((size_t)rq * a.gamma + mt.n) * (size_t)a.V;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = v0 + j;
                if (v >= a.V) continue;
                const float p = ex2((to_f32(trow[v]) - mt.lse_p) * kLog2e);
                if (use_res) {
                    const float q = ex2((acc[j] + to_f32(urow[v]) - mt.lse_q) * kLog2e);
                    wv[j] = fmaxf(p - q, 0.f);
                } else {
                    wv[j] = p;
                }
            }
        }
        float b2 = 0.f;
        const int e = warp_cdf_search(kSliceV, below, target,
                                      [&](int i) {
                                          const float x0 = __shfl_sync(0xffffffffu, wv[0], i >> 2),
                                                      x1 = __shfl_sync(0xffffffffu, wv[1], i >> 2),
                                                      x2 = __shfl_sync(0xffffffffu, wv[2], i >> 2),
                                                      x3 = __shfl_sync(0xffffffffu, wv[3], i >> 2);
                                          const int j = i & 3;
                                          return j == 0 ? x0 : j == 1 ? x1 : j == 2 ? x2 : x3;
                                      },
                                      &b2);
        y = e >= 0 ? vbase + e : -1;
    }
    if (lane == 0) write_outcome(a, w, rq, use_res ? y : -1, use_res ? -1 : y);
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
           align256(sizeof(VerifyPartial) * (size_t)R * nparts) + align256(sizeof(int) * kVerifyMaxMTiles) * 2 +
           align256(sizeof(float) * (size_t)R * ((V + 15) / 16)) + align256(sizeof(unsigned long long) * ((size_t)R * ((V + 63) / 64 + ((V + 63) / 64 + 31) / 32) + 1));
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
    w.tctr = reinterpret_cast<int *>(p);
    p += align256(sizeof(int) * kVerifyMaxMTiles);
    w.csum = reinterpret_cast<float *>(p);
    p += align256(sizeof(float) * (size_t)R * ((V + 15) / 16));
    w.ttot = reinterpret_cast<unsigned long long *>(p);
    return w;
}

cudaError_t launch_verify(const dspark_verify_args &a, const VerifyWs &w, cudaStream_t s) {
    const bool tc = verify_tc_supported(a);
    const int nt = tc ? verify_tc_tiles(a) : 0;
    const int ttot_words = a.R * (nt + (nt + 31) / 32);  // rounded up to even below
    const int n_init = a.R * (a.gamma + 1) > kVerifyMaxMTiles ? a.R * (a.gamma + 1) : kVerifyMaxMTiles;  // >= R
    verify_init<<<(n_init + 255) / 256, 256, 0, s>>>(a.R, a.gamma, w, (ttot_words + 1) & ~1);
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
    if (tc) {
        // the last CTA of each M-tile merges the slices and writes the outcome itself
        e = launch_verify_phase2_tc(a, wf, s);
        return e;
    }
    if (a.dtype == DSPARK_BF16)
        e = rnn ? launch_phase2<__nv_bfloat16, true>(a, w, s) : launch_phase2<__nv_bfloat16, false>(a, w, s);
    else
        e = rnn ? launch_phase2<float, true>(a, w, s) : launch_phase2<float, false>(a, w, s);
    if (e != cudaSuccess) return e;
    if (a.dtype == DSPARK_BF16)
        rnn ? verify_final<__nv_bfloat16, true><<<a.R, 32, 0, s>>>(a, wf)
            : verify_final<__nv_bfloat16, false><<<a.R, 32, 0, s>>>(a, wf);
    else
        rnn ? verify_final<float, true><<<a.R, 32, 0, s>>>(a, wf) : verify_final<float, false><<<a.R, 32, 0, s>>>(a, wf);
    return cudaGetLastError();
}

}  // namespace dspark
