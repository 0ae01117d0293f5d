// rnn_step.cuh -- one tile of the RNN head's state update, eq. (6) of the
// DSpark digest after the h_k part:
//   G = W[:, :2r] [s_{k-1} ; W_1[x_{k-1}]] + Hpre_k,
//   s_k = sigma(G_g) s_{k-1} + (1 - sigma(G_g)) tanh(G_c),   A_k = tanh(G_o).
// A tile is kIB gate entries i0 .. i0 + kIB - 1 of kRB requests q0 ..: the
// 3 kIB rows of W and the kRB input vectors z are staged in shared memory as
// fp32, and kKS adjacent lanes share each (request, entry), lane ks taking the
// 16-byte groups 4 ks, 4 ks + 16, ... of the 2r inputs, then a two-step shuffle
// sum.  Rows are padded by 16 words: 16-byte aligned, and two weight rows read
// by one quarter-warp sit 64 bytes apart in the banks.  kThreads threads run a
// tile; `sync` is their barrier.  Used by the standalone update kernel (the
// CUDA-core path) and, between the steps, by the tensor-core draft launch that
// runs all the steps.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace rnn {

constexpr int kIB = 8;                     // gate entries per tile
constexpr int kKS = 4;                     // lanes sharing one (request, entry)
constexpr int kRB = 16;                    // requests per tile
constexpr int kThreads = kRB * kIB * kKS;  // 512

// shared memory of a tile: [3 kIB + kRB][2r + 16] fp32, then kRB tokens
__host__ __device__ constexpr size_t tile_smem_bytes(int r) {
    return sizeof(float) * (size_t)(3 * kIB + kRB) * (size_t)(2 * r + 16) + sizeof(int) * kRB;
}

// x_{k-1} of request rq: the token array, or the packed race winner of the
// previous step when x_win is set (no winner reads as token 0; the draft's
// finaliser reports that case)
__device__ __forceinline__ int token(const RnnStep &p, int rq) {
    if (p.x_win) {
        const int x = winner_index(__ldcg(p.x_win + rq));
        return x >= 0 && x < p.V ? x : 0;
    }
    const int x = p.x_prev[(size_t)rq * p.x_stride];
    if (x < 0 || x >= p.V) {
        set_err(p.err, DSPARK_ERR_RANGE);
        return 0;
    }
    return x;
}

template <typename T, class Sync>
__device__ void step_tile(const RnnStep &p, float *sh, int i0, int q0, int tid, Sync sync) {
    const int r = p.r, K = 2 * r, ld = K + 16;
    float *Ws = sh;                  // [3 kIB][ld]: rows g r + i0 + ii, g = gate
    float *Zs = sh + 3 * kIB * ld;   // [kRB][ld]
    int *s_xp = reinterpret_cast<int *>(Zs + kRB * ld);
    const int ldw = 2 * r + p.d;
    const T *W = static_cast<const T *>(p.W);
    const T *W1 = static_cast<const T *>(p.W1);
    if (tid < kRB) s_xp[tid] = q0 + tid < p.R ? token(p, q0 + tid) : 0;
    sync();
    constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
    if (r % kVec == 0 && ldw % kVec == 0) {
        // 16-byte loads, several in flight per thread (the loops are unrolled)
        const int cpr = K / kVec;  // chunks per staged row
#pragma unroll 4
        for (int e = tid; e < 3 * kIB * cpr; e += kThreads) {
            const int row = e / cpr, c = e - row * cpr;
            const int g = row / kIB, i = i0 + (row - g * kIB);
            float *dst = Ws + row * ld + c * kVec;
            if (i < r) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(W + (size_t)(g * r + i) * ldw + c * kVec);
                const T *vals = reinterpret_cast<const T *>(&raw);
#pragma unroll
                for (int k = 0; k < kVec; ++k) dst[k] = to_f32(vals[k]);
            } else {
#pragma unroll
                for (int k = 0; k < kVec; ++k) dst[k] = 0.f;
            }
        }
#pragma unroll 4
        for (int e = tid; e < kRB * cpr; e += kThreads) {
            const int q = e / cpr, c = e - q * cpr, rq = q0 + q, j = c * kVec;
            float *dst = Zs + q * ld + j;
            if (rq >= p.R) {
#pragma unroll
                for (int k = 0; k < kVec; ++k) dst[k] = 0.f;
            } else if (j < r) {
                // the state buffers alternate between steps and other CTAs of a
                // multi-step launch write them: read through L2, not L1
                const float *src = p.s_in + (size_t)rq * r + j;
#pragma unroll
                for (int k = 0; k < kVec; k += 4) {
                    const float4 f = __ldcg(reinterpret_cast<const float4 *>(src + k));
                    dst[k] = f.x; dst[k + 1] = f.y; dst[k + 2] = f.z; dst[k + 3] = f.w;
                }
            } else {
                const uint4 raw = *reinterpret_cast<const uint4 *>(W1 + (size_t)s_xp[q] * r + (j - r));
                const T *vals = reinterpret_cast<const T *>(&raw);
#pragma unroll
                for (int k = 0; k < kVec; ++k) dst[k] = to_f32(vals[k]);
            }
        }
    } else {
        for (int e = tid; e < 3 * kIB * K; e += kThreads) {
            const int row = e / K, j = e - row * K;
            const int g = row / kIB, i = i0 + (row - g * kIB);
            Ws[row * ld + j] = i < r ? to_f32(W[(size_t)(g * r + i) * ldw + j]) : 0.f;
        }
        for (int e = tid; e < kRB * K; e += kThreads) {
            const int q = e / K, j = e - q * K, rq = q0 + q;
            float v = 0.f;
            if (rq < p.R) v = j < r ? __ldcg(p.s_in + (size_t)rq * r + j) : to_f32(W1[(size_t)s_xp[q] * r + (j - r)]);
            Zs[q * ld + j] = v;
        }
    }
    // this thread's (request, entry, input share); the h-projection terms are
    // loaded now, off the dependence chain of the dot products
    const int ks = tid % kKS, qi = tid / kKS;
    const int q = qi / kIB, ii = qi - q * kIB;
    const int rq = q0 + q, i = i0 + ii;
    const bool out = ks == 0 && rq < p.R && i < r;
    float hg = 0.f, hc = 0.f, ho = 0.f;
    if (out) {
        const float *hp = p.Hpre + ((size_t)rq * p.gamma + (p.k - 1)) * (size_t)(3 * r);
        hg = hp[i];
        hc = hp[r + i];
        ho = hp[2 * r + i];
    }
    sync();
    const float *z = Zs + q * ld;
    const float *wg = Ws + ii * ld, *wc = Ws + (kIB + ii) * ld, *wo = Ws + (2 * kIB + ii) * ld;
    float gg = 0.f, gc = 0.f, go = 0.f;
    for (int j = 4 * ks; j + 4 <= K; j += 4 * kKS) {
        const float4 zv = *reinterpret_cast<const float4 *>(z + j);
        const float4 a = *reinterpret_cast<const float4 *>(wg + j);
        const float4 b = *reinterpret_cast<const float4 *>(wc + j);
        const float4 c = *reinterpret_cast<const float4 *>(wo + j);
        gg = fmaf(a.x, zv.x, gg); gg = fmaf(a.y, zv.y, gg); gg = fmaf(a.z, zv.z, gg); gg = fmaf(a.w, zv.w, gg);
        gc = fmaf(b.x, zv.x, gc); gc = fmaf(b.y, zv.y, gc); gc = fmaf(b.z, zv.z, gc); gc = fmaf(b.w, zv.w, gc);
        go = fmaf(c.x, zv.x, go); go = fmaf(c.y, zv.y, go); go = fmaf(c.z, zv.z, go); go = fmaf(c.w, zv.w, go);
    }
    if (ks == 0)
        for (int j = K & ~3; j < K; ++j) {  // K % 4 trailing inputs
            const float zj = z[j];
            gg = fmaf(wg[j], zj, gg);
            gc = fmaf(wc[j], zj, gc);
            go = fmaf(wo[j], zj, go);
        }
#pragma unroll
    for (int off = 1; off < kKS; off <<= 1) {
        gg += __shfl_xor_sync(0xffffffffu, gg, off);
        gc += __shfl_xor_sync(0xffffffffu, gc, off);
        go += __shfl_xor_sync(0xffffffffu, go, off);
    }
    if (out) {
        gg += hg;
        gc += hc;
        go += ho;
        const float g = 1.0f / (1.0f + expf(-gg));
        p.s_out[(size_t)rq * r + i] = g * z[i] + (1.0f - g) * tanhf(gc);
        p.A[((size_t)rq * p.gamma + (p.k - 1)) * (size_t)r + i] = tanhf(go);
    }
    sync();  // the staged rows may be overwritten by the next tile
}

}  // namespace rnn
}  // namespace dspark
