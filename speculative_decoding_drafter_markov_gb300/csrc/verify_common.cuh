// verify_common.cuh -- pieces of the verification outcome shared by the
// CUDA-core and tensor-core second phases.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dspark {

// [E] section 06 along the prefix: the accepted drafted tokens, then the
// correction (the residual draw i_res at the first rejection; the draw i_p from
// p when the residual was empty) or, all accepted, the bonus token i_p; the
// next anchor is that token.  Requests missing from the batch
// (ell < 0) get -1 everywhere.
__device__ __forceinline__ void write_outcome(const dspark_verify_args &a, const VerifyWs &w, int rq, int i_res,
                                              int i_p) {
    const int ell = w.ell[rq];
    int32_t *out = a.out_tokens + (size_t)rq * (a.gamma + 1);
    if (ell < 0) {
        a.n_accept[rq] = 0;
        for (int j = 0; j <= a.gamma; ++j) out[j] = -1;
        a.next_anchor[rq] = -1;
        return;
    }
    const int fr = w.first_rej[rq];
    const bool residual = fr < ell;
    const int n = residual ? fr : ell;
    int y = (residual && i_res >= 0) ? i_res : i_p;
    if (y < 0) {
        set_err(a.err, DSPARK_ERR_NONFINITE);
        y = 0;
    }
    a.n_accept[rq] = n;
    for (int j = 0; j <= a.gamma; ++j) out[j] = j < n ? a.x[(size_t)rq * a.gamma + j] : (j == n ? y : -1);
    a.next_anchor[rq] = y;
}

// write_outcome by one warp (all lanes), the drawn token y (-1: none), the
// tokens written lane-parallel
__device__ __forceinline__ void write_outcome_warp(const dspark_verify_args &a, const VerifyWs &w, int rq, int y) {
    const int lane = threadIdx.x & 31;
    const int ell = w.ell[rq];
    int32_t *out = a.out_tokens + (size_t)rq * (a.gamma + 1);
    if (ell < 0) {
        for (int j = lane; j <= a.gamma; j += 32) out[j] = -1;
        if (lane == 0) {
            a.n_accept[rq] = 0;
            a.next_anchor[rq] = -1;
        }
        return;
    }
    const int fr = w.first_rej[rq];
    const int n = fr < ell ? fr : ell;
    if (y < 0) {
        if (lane == 0) set_err(a.err, DSPARK_ERR_NONFINITE);
        y = 0;
    }
    for (int j = lane; j <= a.gamma; j += 32) out[j] = j < n ? a.x[(size_t)rq * a.gamma + j] : (j == n ? y : -1);
    if (lane == 0) {
        a.n_accept[rq] = n;
        a.next_anchor[rq] = y;
    }
}

// The correction / bonus token is an inverse-CDF draw from the weights w (the
// residual max(0, p - q), or p): one uniform u from Philox stream 2 with
// counter (0, n, request, cycle << 2 | 2), word 0, the target u * sum(w), and the
// first vocabulary entry whose cumulative weight exceeds it.  Sums run in fp32
// in a fixed order (below), so the draw is deterministic.
__device__ __forceinline__ float correction_uniform(uint64_t seed, uint64_t cycle, int n, int rq) {
    const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)n, (uint32_t)rq, philox_ctr3(cycle, 2)),
                                  philox_key(seed));
    return uniform_of(w.x);
}

// Tile sums of the tensor-core phase in fixed point: a thread's share of a
// tile, a sum of probabilities (at most 1 up to rounding), clamped to [0, 2]
// (NaN to 0) and truncated to a multiple of 2^-47, so that integer addition --
// exact and independent of order -- holds up to 2^16 shares without overflow.
constexpr float kFixScale = 140737488355328.f;  // 2^47
__device__ __forceinline__ unsigned long long to_fixed(float x) {
    return __float2ull_rz(fminf(fmaxf(x, 0.f), 2.f) * kFixScale);
}

// One warp (all lanes) over cnt consecutive non-negative weights get(i), i <
// cnt, taken 32 at a time with an inclusive warp scan and a running carry that
// starts at `base` (the order of the additions is fixed).  With target >= 0:
// returns the first i whose cumulative weight exceeds `target` and its
// exclusive cumulative in *below; when the target is never passed (it sits at
// the total, to rounding), the last i with a positive weight; -1 when all are
// zero.  *total receives base + the sum of all cnt weights (the same
// additions), when the scan ran to the end.  NB groups of 32 are fetched before
// they are scanned (their loads in flight together); the result does not
// depend on NB.
template <int NB = 1, class Get>
__device__ __forceinline__ int warp_cdf_search(int cnt, float base, float target, Get &&get, float *below,
                                               float *total = nullptr) {
    const int lane = threadIdx.x & 31;
    float carry = base, below_last = base;
    int last = -1;
    for (int i0 = 0; i0 < cnt; i0 += 32 * NB) {
        float vb[NB];
#pragma unroll
        for (int g = 0; g < NB; ++g) {
            const int i = i0 + 32 * g + lane;
            vb[g] = i < cnt ? get(i) : 0.f;
        }
#pragma unroll
        for (int g = 0; g < NB; ++g) {
            const float v = fmaxf(vb[g], 0.f);  // NaN and negative weights count as zero
            float incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const float cum_in = carry + incl, cum_ex = cum_in - v;
            const unsigned pos = __ballot_sync(0xffffffffu, v > 0.f);
            const unsigned hit = __ballot_sync(0xffffffffu, v > 0.f && cum_in > target);
            if (hit) {
                const int l = __ffs(hit) - 1;
                *below = __shfl_sync(0xffffffffu, cum_ex, l);
                return i0 + 32 * g + l;
            }
            if (pos) {
                const int l = 31 - __clz(pos);
                last = i0 + 32 * g + l;
                below_last = __shfl_sync(0xffffffffu, cum_ex, l);
            }
            carry = __shfl_sync(0xffffffffu, cum_in, 31);
        }
    }
    *below = below_last;
    if (total) *total = carry;
    return last;
}

// One warp: the sum of cnt non-negative weights get(i) (NaN and negative count
// as zero), NB per lane fetched together; lane-strided partial sums, then a
// fixed tree over the lanes, the same value on every lane.
template <int NB, class Get>
__device__ __forceinline__ float warp_weight_sum(int cnt, Get &&get) {
    const int lane = threadIdx.x & 31;
    float acc = 0.f;
    for (int i0 = 0; i0 < cnt; i0 += 32 * NB) {
        float vb[NB];
#pragma unroll
        for (int g = 0; g < NB; ++g) {
            const int i = i0 + 32 * g + lane;
            vb[g] = i < cnt ? get(i) : 0.f;
        }
#pragma unroll
        for (int g = 0; g < NB; ++g) acc += fmaxf(vb[g], 0.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
    return __shfl_sync(0xffffffffu, acc, 0);
}

}  // namespace dspark
