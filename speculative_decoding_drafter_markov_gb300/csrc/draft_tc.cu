// draft_tc.cu -- the draft step on the 5th-generation tensor cores.
//
// DSpark digest eq. (5): B_k = W_1[x_{k-1}] W_2 (Markov head) or eq. (6)
// B_k = W_2^T tanh(W_o z_k) (RNN head), contracted on tcgen05 into TMEM and
// consumed in place by the eq. (4) epilogue: U_k add, sum of exponentials,
// the two-level draw (16-entry blocks raced on their masses with Philox
// words, the winning block's entry by inverse CDF).  No logit reaches global memory.  The pipeline (TMA rings
// of W_2^T slabs and U_k tiles, MMA warp, per-warp TMEM epilogue) is tc_pipe.cuh;
// this file supplies the bias operand, the per-tile epilogue and the merge.
//
// Markov head: the operand E = W_1[x_{k-1}] is exact in bf16.  RNN head: the
// fp32 operand A_k is split into bf16 hi + lo parts (two MMAs per K-step).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "rnn_step.cuh"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace dspark {

namespace {

struct TcParams {
    int R, V, r, d, gamma;
    int k;       // first step of the launch (1..gamma)
    int nsteps;  // steps k .. k + nsteps - 1
    int step_index;  // counter index of step k (1 for the first step since the counters were zeroed)
    int phase0;      // cross-CTA synchronisation points earlier launches of the draft passed
    const __nv_bfloat16 *W1;
    const __nv_bfloat16 *W2t;  // [V, r] (the W_2^T tiles of the first step are pulled into L2 early)
    const int32_t *x_prev;  // token x_{k-1} of row i at x_prev[i * x_stride]
    int x_stride;
    const float *A_op;  // RNN: operand of row i for step k at A_op[i * a_stride], else null
    int a_stride;       // (step k + j: A_op + j r)
    const __nv_bfloat16 *h;  // [R, gamma, d]
    const float *w;          // [d + r]
    const float *sts_T;      // [gamma] or null
    uint64_t seed, cycle;
    PhiloxRoundKeys rk;  // of seed
    DraftPartial *part;  // [gamma][R][nparts]: step partials, by counter index - 1
    unsigned long long *winners;  // [gamma][R] packed race winners, zero at the start of the call
    int *counters;  // [n_mtiles]: partials published (per M-tile), zero at the start of the call
    int32_t *x;
    float *logq, *lse, *c;   // [R, gamma]
    float *conf_logit;       // [R, gamma] or null
    int nparts;  // vocabulary ranges (CTAs per M-tile)
    int n_mtiles;
    int32_t *err;
    RnnStep rnn;  // RNN head: the state update's inputs (s_in holds s_{k-1})
    unsigned char *a_stage;  // RNN head: [n_mtiles][kRnnStageBytes] prepared operands
};

// eq. (7): c_k = sigma(w^T [h_k ; W_1[x_{k-1}]] / T_k) of one request (token
// xp = x_{k-1}) by one warp: lanes over 16-byte chunks, four in flight, then a
// fixed shuffle tree; lane 0 writes.  Computed after the launch's last step.
__device__ __forceinline__ void confidence_warp(const TcParams &p, int k, int grow, int xp, int lane) {
    const __nv_bfloat16 *h = p.h + ((size_t)grow * p.gamma + (k - 1)) * (size_t)p.d;
    const __nv_bfloat16 *e = p.W1 + (size_t)xp * p.r;
    float dot = 0.f;
    if ((p.d & 7) == 0) {
        const int hc = p.d / 8, nc = hc + p.r / 8;
#pragma unroll 4
        for (int ch = lane; ch < nc; ch += 32) {
            const uint4 raw = ch < hc ? *reinterpret_cast<const uint4 *>(h + ch * 8)
                                      : *reinterpret_cast<const uint4 *>(e + (ch - hc) * 8);
            const float *wv = p.w + ch * 8;
            const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dot = fmaf(wv[2 * i], tcp::bf16_lo(v[i]), dot);
                dot = fmaf(wv[2 * i + 1], tcp::bf16_hi(v[i]), dot);
            }
        }
    } else {
        for (int j = lane; j < p.d + p.r; j += 32)
            dot = fmaf(p.w[j], __bfloat162float(j < p.d ? h[j] : e[j - p.d]), dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) {
        const float T_k = p.sts_T ? p.sts_T[k - 1] : 1.0f;
        const size_t o = (size_t)grow * p.gamma + (k - 1);
        p.c[o] = 1.0f / (1.0f + expf(-dot / T_k));
        if (p.conf_logit) p.conf_logit[o] = dot;
    }
}

__device__ __forceinline__ int ld_acquire(const int *ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// bounded wait until *ctr >= target (a counter other CTAs of the launch raise)
__device__ __forceinline__ bool wait_counter(const int *ctr, int target, int32_t *err,
                                             uint64_t limit_ns = tc::kWaitLimitNs) {
    const uint64_t t0 = tc::globaltimer_ns();
    while (ld_acquire(ctr) < target) {
        if (tc::globaltimer_ns() - t0 > limit_ns) {
            set_err(err, DSPARK_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

// token x_{k-1} of request grow (held in s.tok), checked against the vocabulary
__device__ __forceinline__ int load_token(const TcParams &p, int grow, const int32_t *xp, int stride) {
    if (grow >= p.R) return -1;
    int x = xp[(size_t)grow * stride];
    if (x < 0 || x >= p.V) {
        set_err(p.err, DSPARK_ERR_RANGE);
        x = 0;
    }
    return x;
}

// the bias operand of the M-tile in the swizzled K-major layout: W_1[x_{k-1}]
// (tokens in s.tok) or the split fp32 RNN operand; threads tid, tid + nthr, ...
template <class P>
__device__ __forceinline__ void gather_operand(const TcParams &p, const typename P::State &s, int m0, int k,
                                               int tid, int nthr) {
    const int chunks_per_row = p.r / 8;
    const float *A_k = P::KSPLIT == 2 ? p.A_op + (size_t)(k - p.k) * p.r : nullptr;
    if (P::KSPLIT == 1 && nthr == tcp::kEpiThreads) {
        // the epilogue threads at a step boundary: all of a thread's row loads in
        // flight together (MV rows x r / 8 chunks <= 8 per thread), then the stores
        constexpr int kMax = P::MV * 32 / tcp::kEpiThreads;
        uint4 v[kMax];
#pragma unroll
        for (int n = 0; n < kMax; ++n) {
            const int e = tid + n * tcp::kEpiThreads, row = e / chunks_per_row, c = e - row * chunks_per_row;
            const int xp = e < P::MV * chunks_per_row ? s.tok[row] : -1;
            v[n] = xp >= 0 ? *reinterpret_cast<const uint4 *>(p.W1 + (size_t)xp * p.r + c * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int n = 0; n < kMax; ++n) {
            const int e = tid + n * tcp::kEpiThreads, row = e / chunks_per_row, c = e - row * chunks_per_row;
            if (e < P::MV * chunks_per_row) P::put_a(s, row, c, 0, v[n]);
        }
        return;
    }
    for (int e = tid; e < P::MV * chunks_per_row; e += nthr) {
        const int row = e / chunks_per_row, c = e - row * chunks_per_row;
        const int grow = m0 + row;
        if (P::KSPLIT == 1) {
            const int xp = s.tok[row];
            const uint4 val = xp >= 0 ? *reinterpret_cast<const uint4 *>(p.W1 + (size_t)xp * p.r + c * 8)
                                      : make_uint4(0u, 0u, 0u, 0u);
            P::put_a(s, row, c, 0, val);
        } else {
            float xs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (grow < p.R) {
                // written by other CTAs of the launch: read through L2
                const float4 *src = reinterpret_cast<const float4 *>(A_k + (size_t)grow * p.a_stride + c * 8);
                const float4 a0 = __ldcg(src), a1 = __ldcg(src + 1);
                xs[0] = a0.x; xs[1] = a0.y; xs[2] = a0.z; xs[3] = a0.w;
                xs[4] = a1.x; xs[5] = a1.y; xs[6] = a1.z; xs[7] = a1.w;
            }
            uint4 hi, lo;
            tcp::split8(xs, hi, lo);
            P::put_a(s, row, c, 0, hi);
            P::put_a(s, row, c, 1, lo);
        }
    }
}

// Finalise row gr of step k from its nparts partials, by one warp (lanes stride
// over the partials, then a fixed shuffle tree): x_k, lse_k, log q_k(x_k),
// written by lane 0.
__device__ __forceinline__ void finalise_row(const TcParams &p, const DraftPartial *part, int gr, int k, int lane) {
    RowState f;
    row_init(f);
    // a lane's partials four at a time: the loads of a batch in flight together,
    // then merged in order
    constexpr int kBatch = 4;
    for (int q0 = 0; lane + 32 * q0 < p.nparts; q0 += kBatch) {
        DraftPartial pq[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = lane + 32 * (q0 + q);
            if (i < p.nparts) pq[q] = load_partial_cg(part + (size_t)gr * p.nparts + i);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q)
            if (lane + 32 * (q0 + q) < p.nparts) row_merge(f, pq[q].m, pq[q].S, pq[q].best, pq[q].zbest, pq[q].idx);
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float m = __shfl_xor_sync(0xffffffffu, f.m, off);
        const float S = __shfl_xor_sync(0xffffffffu, f.S, off);
        const float bb = __shfl_xor_sync(0xffffffffu, f.best, off);
        const float zb = __shfl_xor_sync(0xffffffffu, f.zbest, off);
        const int ix = __shfl_xor_sync(0xffffffffu, f.idx, off);
        row_merge(f, m, S, bb, zb, ix);
    }
    if (lane == 0) {
        const size_t o = (size_t)gr * p.gamma + (k - 1);
        const float lse = f.m + logf(f.S);
        int idx = f.idx;
        if (idx < 0 || !isfinite(lse)) {
            set_err(p.err, DSPARK_ERR_NONFINITE);
            idx = 0;
        }
        p.x[o] = idx;
        p.lse[o] = lse;
        p.logq[o] = f.zbest - lse;
    }
}

// Cross-CTA synchronisation point of the M-tile (all epilogue threads call it):
// with `publish`, this CTA's writes so far become visible and it counts itself
// (else it did so already); then it waits (bounded) until every CTA of the
// M-tile has reached synchronisation point number `phase`.  Returns false (and
// raises the abort flag) when the wait ran out or the CTA had aborted.
template <class P>
__device__ __forceinline__ bool mtile_sync(const TcParams &p, typename P::State &s, int *ctr, int phase, int et,
                                           bool publish) {
    if (publish) tc::named_bar_sync(1, tcp::kEpiThreads);
    if (et == 0) {
        if (publish) {
            __threadfence();  // cumulative over the CTA's writes before the barrier
            atomicAdd(ctr, 1);
        }
        *s.flag = !*s.abort_flag && wait_counter(ctr, phase * p.nparts, p.err) ? 1 : 0;
    }
    tc::named_bar_sync(1, tcp::kEpiThreads);
    if (!*s.flag) {
        *s.abort_flag = 1;
        return false;
    }
    __threadfence();
    return true;
}

// RNN head, eq. (6): the state update of step k for the M-tile's requests --
//   G = W[:, :2r] [s_{k-1} ; W_1[x_{k-1}]] + Hpre_k,
//   s_k = sigma(G_g) s_{k-1} + (1 - sigma(G_g)) tanh(G_c),   A_k = tanh(G_o),
// with x_{k-1} the launch's input token at its first step, else step k-1's race
// winner.  Tiles of kRQ requests x kIE gate entries spread over the M-tile's
// CTAs; a tile stages its 3 kIE weight rows and kRQ input vectors in fp32 in the
// operand region (free between two steps' contractions).  Thread (ks, ii, qb)
// takes the K inputs 4 (ks + kKS g), g = 0.., of entry ii for the kQB requests of
// block qb (one weight load serves kQB requests), then kKS lanes sum by
// shuffles.  Besides s_k and the fp32 A_k, each tile writes its 16-byte chunk of
// the operand -- A_k split into bf16 hi + lo, in the shared-memory layout of the
// contraction -- to the M-tile's staging buffer, which every CTA of the M-tile
// then bulk-copies into its operand region.
namespace rnnt {
constexpr int kRQ = 32;  // requests per tile
constexpr int kIE = 8;   // gate entries per tile (one 16-byte operand chunk)
constexpr int kKS = 8;   // lanes sharing one (entry, request block)
constexpr int kQB = 4;   // requests per thread
constexpr int kWLoads = 3;  // 16-byte weight chunks per thread (r <= 256)
constexpr int kZLoads = 4;  // 16-byte chunks of the state inputs per thread (r <= 256)
static_assert(kKS * kIE * (kRQ / kQB) == tcp::kEpiThreads, "one thread per (ks, entry, request block)");
static_assert(kWLoads * tcp::kEpiThreads >= 3 * kIE * 64 && kZLoads * tcp::kEpiThreads >= kRQ * 64 &&
                  (kZLoads / 2) * tcp::kEpiThreads >= kRQ * 32,
              "r <= 256");
// shared memory: [3 kIE + kRQ][2r + 4] fp32, the tile's pre-activations from
// the h projection [kRQ][3 kIE] fp32, A_k [kRQ][kIE] fp32, kRQ tokens
__host__ __device__ constexpr int smem_bytes(int r) {
    return 4 * (3 * kIE + kRQ) * (2 * r + 4) + 4 * kRQ * 3 * kIE + 4 * kRQ * kIE + 4 * kRQ;
}
}  // namespace rnnt

__device__ __forceinline__ float4 bf16x8_lo4(const uint4 &v) {
    return make_float4(tcp::bf16_lo(v.x), tcp::bf16_hi(v.x), tcp::bf16_lo(v.y), tcp::bf16_hi(v.y));
}
__device__ __forceinline__ float4 bf16x8_hi4(const uint4 &v) {
    return make_float4(tcp::bf16_lo(v.z), tcp::bf16_hi(v.z), tcp::bf16_lo(v.w), tcp::bf16_hi(v.w));
}

template <class P>
__device__ __forceinline__ void rnn_state_update(const TcParams &p, const typename P::State &s, int m0, int m_tile,
                                                 int cv, int k, int et) {
    static_assert(P::kABytes - P::kMergeBytes >= rnnt::smem_bytes(256), "state-update tile in the operand region");
    static_assert(P::kABytes == (int)kRnnStageBytes, "staging buffer holds one operand region");
    // the state buffers alternate: p.rnn.s_in holds s_{k-1} at the launch's first step
    const bool odd = ((k - p.k) & 1) != 0;
    const float *s_in = odd ? p.rnn.s_out : p.rnn.s_in;
    float *s_out = odd ? const_cast<float *>(p.rnn.s_in) : p.rnn.s_out;
    // x_{k-1}: the launch's input tokens at its first step, else step k-1's race winners
    const unsigned long long *x_win =
        k == p.k ? nullptr : p.winners + (size_t)(p.step_index + (k - 1 - p.k) - 1) * p.R;
    const int r = p.r, K = 2 * r, ld = K + 4, ldw = 2 * r + p.d;
    float *Ws = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(P::merge_scratch(s)) + P::kMergeBytes);
    float *Zs = Ws + 3 * rnnt::kIE * ld;
    float *Hs = Zs + rnnt::kRQ * ld;
    float *As = Hs + rnnt::kRQ * 3 * rnnt::kIE;
    int *xs = reinterpret_cast<int *>(As + rnnt::kRQ * rnnt::kIE);
    const __nv_bfloat16 *W = static_cast<const __nv_bfloat16 *>(p.rnn.W);
    unsigned char *stage = p.a_stage + (size_t)m_tile * kRnnStageBytes;
    const int ni = r / rnnt::kIE;
    const int nq = (min(P::MV, p.R - m0) + rnnt::kRQ - 1) / rnnt::kRQ;
    const int ks = et % rnnt::kKS, ii = (et / rnnt::kKS) % rnnt::kIE, qb = et / (rnnt::kKS * rnnt::kIE);
    const int cpr = K / 8;  // 16-byte chunks of a staged weight row
    const int nw = 3 * rnnt::kIE * cpr;
    const bool wvec = (ldw & 7) == 0;  // rows of W start on 16-byte boundaries
    for (int t = cv; t < ni * nq; t += p.nparts) {
        const int i0 = (t % ni) * rnnt::kIE, q0 = m0 + (t / ni) * rnnt::kRQ;
        if (et < rnnt::kRQ) {
            int x = 0;
            if (q0 + et < p.R) {
                if (x_win) {
                    x = winner_index(__ldcg(x_win + q0 + et));
                    if (x < 0 || x >= p.V) x = 0;  // no winner: reported by the finaliser
                } else {
                    x = load_token(p, q0 + et, p.x_prev, p.x_stride);
                }
            }
            xs[et] = x;
        }
        tc::named_bar_sync(1, tcp::kEpiThreads);
        // All of a thread's loads in flight together: weight rows g r + i0 + e
        // (g: gate, candidate, output), the inputs [s_{k-1} ; W_1[x_{k-1}]] of the
        // tile's requests and their h-projection terms; then widened to fp32.
        // the state part of the inputs moves as 16-byte chunks of 4 fp32, the
        // embedding part as 16-byte chunks of 8 bf16
        const int cs = r / 4, ce = r / 8;
        uint4 wr[rnnt::kWLoads], zs[rnnt::kZLoads];
#pragma unroll
        for (int n = 0; n < rnnt::kWLoads; ++n) {
            const int e = et + n * tcp::kEpiThreads;
            if (wvec && e < nw) {
                const int row = e / cpr, c = e - row * cpr;
                const int g = row / rnnt::kIE, i = i0 + (row - g * rnnt::kIE);
                wr[n] = *reinterpret_cast<const uint4 *>(W + (size_t)(g * r + i) * ldw + c * 8);
            }
        }
#pragma unroll
        for (int n = 0; n < rnnt::kZLoads; ++n) {
            const int e = et + n * tcp::kEpiThreads, q = e / cs, rq = q0 + q;
            // the state buffers alternate between steps and other CTAs write them: L2 reads
            if (e < rnnt::kRQ * cs && rq < p.R)
                zs[n] = __ldcg(reinterpret_cast<const uint4 *>(s_in + (size_t)rq * r) + (e - q * cs));
        }
        for (int e = et; e < rnnt::kRQ * 3 * rnnt::kIE; e += tcp::kEpiThreads) {
            const int q = e / (3 * rnnt::kIE), gi = e - q * 3 * rnnt::kIE, g = gi / rnnt::kIE;
            const int rq = q0 + q, i = i0 + (gi - g * rnnt::kIE);
            Hs[e] = rq < p.R ? p.rnn.Hpre[((size_t)rq * p.gamma + (k - 1)) * (size_t)(3 * r) + g * r + i] : 0.f;
        }
#pragma unroll
        for (int n = 0; n < rnnt::kWLoads; ++n) {
            const int e = et + n * tcp::kEpiThreads;
            if (wvec && e < nw) {
                const int row = e / cpr, c = e - row * cpr;
                float4 *dst = reinterpret_cast<float4 *>(Ws + row * ld + c * 8);
                dst[0] = bf16x8_lo4(wr[n]);
                dst[1] = bf16x8_hi4(wr[n]);
            }
        }
        if (!wvec) {
            for (int e = et; e < 3 * rnnt::kIE * K; e += tcp::kEpiThreads) {
                const int row = e / K, j = e - row * K;
                const int g = row / rnnt::kIE, i = i0 + (row - g * rnnt::kIE);
                Ws[row * ld + j] = __bfloat162float(W[(size_t)(g * r + i) * ldw + j]);
            }
        }
#pragma unroll
        for (int n = 0; n < rnnt::kZLoads; ++n) {
            const int e = et + n * tcp::kEpiThreads, q = e / cs;
            if (e < rnnt::kRQ * cs) {
                const uint4 v = q0 + q < p.R ? zs[n] : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(Zs + q * ld + 4 * (e - q * cs)) = v;
            }
        }
        uint4 ze[rnnt::kZLoads / 2];
#pragma unroll
        for (int n = 0; n < rnnt::kZLoads / 2; ++n) {
            const int e = et + n * tcp::kEpiThreads, q = e / ce, rq = q0 + q;
            if (e < rnnt::kRQ * ce && rq < p.R)
                ze[n] = *reinterpret_cast<const uint4 *>(p.W1 + (size_t)xs[q] * r + 8 * (e - q * ce));
        }
#pragma unroll
        for (int n = 0; n < rnnt::kZLoads / 2; ++n) {
            const int e = et + n * tcp::kEpiThreads, q = e / ce;
            if (e < rnnt::kRQ * ce) {
                float4 *dst = reinterpret_cast<float4 *>(Zs + q * ld + r + 8 * (e - q * ce));
                if (q0 + q < p.R) {
                    dst[0] = bf16x8_lo4(ze[n]);
                    dst[1] = bf16x8_hi4(ze[n]);
                } else {
                    dst[0] = dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
        tc::named_bar_sync(1, tcp::kEpiThreads);
        // dot products on paired lanes: (even, odd) inputs of each float4 half
        float2 acc[rnnt::kQB][3];
#pragma unroll
        for (int q = 0; q < rnnt::kQB; ++q) acc[q][0] = acc[q][1] = acc[q][2] = make_float2(0.f, 0.f);
        const float *wg = Ws + ii * ld, *wc = Ws + (rnnt::kIE + ii) * ld, *wo = Ws + (2 * rnnt::kIE + ii) * ld;
        const float *zb0 = Zs + qb * rnnt::kQB * ld;
        for (int j = 4 * ks; j < K; j += 4 * rnnt::kKS) {
            const float4 a = *reinterpret_cast<const float4 *>(wg + j);
            const float4 b = *reinterpret_cast<const float4 *>(wc + j);
            const float4 c = *reinterpret_cast<const float4 *>(wo + j);
#pragma unroll
            for (int q = 0; q < rnnt::kQB; ++q) {
                const float4 z = *reinterpret_cast<const float4 *>(zb0 + q * ld + j);
                const float2 z0 = make_float2(z.x, z.y), z1 = make_float2(z.z, z.w);
                acc[q][0] = fma2(make_float2(a.z, a.w), z1, fma2(make_float2(a.x, a.y), z0, acc[q][0]));
                acc[q][1] = fma2(make_float2(b.z, b.w), z1, fma2(make_float2(b.x, b.y), z0, acc[q][1]));
                acc[q][2] = fma2(make_float2(c.z, c.w), z1, fma2(make_float2(c.x, c.y), z0, acc[q][2]));
            }
        }
        float sum[rnnt::kQB][3];
#pragma unroll
        for (int q = 0; q < rnnt::kQB; ++q)
#pragma unroll
            for (int g = 0; g < 3; ++g) sum[q][g] = acc[q][g].x + acc[q][g].y;
#pragma unroll
        for (int off = 1; off < rnnt::kKS; off <<= 1)
#pragma unroll
            for (int q = 0; q < rnnt::kQB; ++q)
#pragma unroll
                for (int g = 0; g < 3; ++g) sum[q][g] += __shfl_xor_sync(0xffffffffu, sum[q][g], off);
        if (ks == 0) {
            const int i = i0 + ii;
#pragma unroll
            for (int q = 0; q < rnnt::kQB; ++q) {
                const int ql = qb * rnnt::kQB + q, rq = q0 + ql;
                const float *h3 = Hs + ql * 3 * rnnt::kIE + ii;
                const float gg = sum[q][0] + h3[0], gc = sum[q][1] + h3[rnnt::kIE], go = sum[q][2] + h3[2 * rnnt::kIE];
                const float g = 1.0f / (1.0f + expf(-gg));
                const float a_out = tanhf(go);
                if (rq < p.R) {
                    s_out[(size_t)rq * r + i] = g * Zs[ql * ld + i] + (1.0f - g) * tanhf(gc);
                    p.rnn.A[((size_t)rq * p.gamma + (k - 1)) * (size_t)r + i] = a_out;
                }
                As[ql * rnnt::kIE + ii] = rq < p.R ? a_out : 0.f;
            }
        }
        tc::named_bar_sync(1, tcp::kEpiThreads);
        // the operand chunk (entries i0 .. i0 + 7) of each request of the tile, hi and lo parts
        if (et < rnnt::kRQ && q0 + et < p.R) {
            const int row = q0 - m0 + et;
            uint4 hi, lo;
            tcp::split8(As + et * rnnt::kIE, hi, lo);
            *reinterpret_cast<uint4 *>(stage + P::a_offset(row, i0 / 8, 0)) = hi;
            *reinterpret_cast<uint4 *>(stage + P::a_offset(row, i0 / 8, 1)) = lo;
        }
        tc::named_bar_sync(1, tcp::kEpiThreads);  // the scratch is reused by the next tile
    }
    // the staged chunks are read by other CTAs' bulk copies (async proxy)
    tc::fence_proxy_async_global();
}

// RNN head: one thread copies the M-tile's prepared operand (the kslabs used K
// slabs of the hi and lo parts) from the staging buffer into the operand region
// and, once it has landed, lets the MMA warp go.  `use` counts the copies of
// the launch (the barrier's phase).
template <class P>
__device__ __forceinline__ bool rnn_load_operand(const TcParams &p, typename P::State &s, int m_tile, int use) {
    const unsigned char *stage = p.a_stage + (size_t)m_tile * kRnnStageBytes;
    const int kslabs = p.r / 64;
    tc::fence_proxy_async_global();
    tc::mbar_expect_tx(s.opbar, (uint32_t)(2 * kslabs * P::kSlabA));
    for (int part = 0; part < 2; ++part)
        for (int j = 0; j < kslabs; ++j) {
            const int slab = j + 4 * part;
            tc::bulk_load(s.sA + slab * P::kSlabA, stage + slab * P::kSlabA, (uint32_t)P::kSlabA, s.opbar);
        }
    if (!tc::mbar_wait_drain(s.opbar, (uint32_t)use & 1u, p.err)) {
        *s.abort_flag = 1;
        return false;
    }
    tc::mbar_arrive(s.aready);
    return true;
}

// One launch runs draft steps k .. k + nsteps - 1 of one decoding cycle.  CTA
// (m_tile, cv) owns requests m0 .. m0 + MV - 1 and the vocabulary tiles
// cv, cv + nparts, cv + 2 nparts, ... (about an equal share).  Per step:
// contraction + eq. (4) epilogue over the columns, a merge into one partial
// per request (kept per step) and the race winner folded into a per-(step,
// request) 64-bit maximum.  Once every CTA of the M-tile has published
// (bounded wait; the launch is cooperative, so all are resident) each reads
// the winners x_k of its rows and gathers the next operand W_1[x_k] right away
// -- the producer has already streamed the next step's first W_2^T slabs and U
// tiles.  Nothing else sits between two steps: the rows' lse_k and log q_k
// (which need every CTA's partial) and the confidences c_k (x_{k-1} from the
// per-step winner words) are computed after the last step, spread over the
// CTAs' warps.
template <class P>
__global__ void __launch_bounds__(P::kThreads, 1)
    draft_step_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmU,
                  const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    typename P::State s = P::carve(smem_raw);
    P::init(s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.n_mtiles, cv = blockIdx.x / p.n_mtiles;
    const int m0 = m_tile * P::MV;
    // the CTA's vocabulary tiles: every nparts-th BN-wide tile, starting at tile
    // cv, so the CTAs of an M-tile stream neighbouring pieces of each U row at
    // the same time (DRAM page locality); the last tile may end at V
    const int n_vtiles = (p.V + P::BN - 1) / P::BN;
    const int c0 = cv * P::BN, c1 = p.V, tstride = p.nparts * P::BN;
    const int ntiles = (n_vtiles - cv + p.nparts - 1) / p.nparts;
    const int kslabs = p.r / 64;
    int *ctr = p.counters + m_tile;

    // 0. the first step reads this CTA's W_2^T tiles from DRAM: start them towards L2
    //    now, while the tokens and the first operand are gathered (one M-tile only:
    //    with several, the M-tiles' CTAs would pull the same tiles; measured no gain)
    if (threadIdx.x == P::MV && p.n_mtiles == 1) {
        for (int t = 0; t < ntiles; ++t) {
            const int n0 = c0 + t * tstride, rows = min(P::BN, p.V - n0);
            tc::prefetch_l2_bulk(p.W2t + (size_t)n0 * p.r, (uint32_t)(rows * p.r * 2));
        }
    }
    // 1. the M-tile's tokens x_{k-1} (one load per row, all in flight together)
    if (threadIdx.x < P::MV) s.tok[threadIdx.x] = load_token(p, m0 + threadIdx.x, p.x_prev, p.x_stride);
    __syncthreads();  // tokens, barriers, thresholds, TMEM
    P::ready(s);

    // 2. first bias operand, before the W_2 / U streams compete for bandwidth (the
    //    RNN head's first operand needs the state update, below)
    if (P::KSPLIT == 1) {
        gather_operand<P>(p, s, m0, p.k, threadIdx.x, P::kThreads);
        tc::fence_proxy_async_smem();
    }
    __syncthreads();  // operand complete

    if (warp == tcp::kProducerWarp) {
        if (lane == 0) {
            tc::prefetch_tmap(&tmB);
            tc::prefetch_tmap(&tmU);
        }
        __syncwarp();
        if (lane == 0) P::producer_w2(s, &tmB, c0, tstride, ntiles, kslabs, p.nsteps, p.err);
        __syncwarp();
    } else if (warp == tcp::kUWarp) {
        if (lane == 0) P::producer_u(s, &tmU, c0, tstride, ntiles, p.nsteps, p.k - 1, m0, p.err);
        __syncwarp();
    } else if (warp == tcp::kMmaWarp) {
        if (lane == 0) P::mma(s, ntiles, kslabs, p.nsteps, p.err, P::KSPLIT == 1 ? 1 : 0);
        __syncwarp();
    } else {
        const int et = threadIdx.x;
        const int row = P::epi_row(), col0 = P::epi_col0();
        const int grow = m0 + row;
        const bool row_live = grow < p.R;
        const uint32_t c3 = philox_ctr3(p.cycle, 0);
        float *mg = P::merge_scratch(s);
        int phase = p.phase0;  // cross-CTA synchronisation points passed
        int op_copies = 0;     // RNN head: operand copies issued
        if constexpr (P::KSPLIT == 2) {
            // RNN head: the state update of the first step, then its operand A_k
            rnn_state_update<P>(p, s, m0, m_tile, cv, p.k, et);
            if (mtile_sync<P>(p, s, ctr, ++phase, et, true) && et == 0) rnn_load_operand<P>(p, s, m_tile, op_copies);
            ++op_copies;
        }
        for (int step = 0; step < p.nsteps && !*s.abort_flag; ++step) {
            const int k = p.k + step, q = p.step_index + step;
            DraftPartial *part = p.part + (size_t)(q - 1) * p.R * p.nparts;
            unsigned long long *win = p.winners + (size_t)(q - 1) * p.R;

            RowState st;
            row_init(st);
            const PhiloxRow prow = philox_row((uint32_t)k, (uint32_t)grow, p.rk);
            // Thresholds shared by all CTAs: a block only needs its entry drawn when
            // it beats the row's best block so far, wherever that was found.  The
            // step's winner word of a request (win[row], raised by every CTA) holds
            // the packed score of some block of the row, so any value read from it
            // is a valid threshold, however stale.  Once per tile one thread per
            // request (the leader) forwards the CTA's best when it beats what it
            // last saw and brings the global best into the CTA; its read is issued
            // a tile ahead so the L2 latency stays off the tile loop.
            const bool leader = row_live && warp < (P::DUAL ? 2 : 4);
            unsigned long long *gwin = win + (row_live ? grow : m0);
            unsigned long long g_next = leader ? tc::ld_relaxed_gpu_u64(gwin) : 0ull, g_sent = 0ull;
            uint2 w_odd = make_uint2(0u, 0u);  // the odd block's words of the last Philox call
            P::epilogue(s, step * ntiles, c0, tstride, ntiles, p.err,
                        [&](int, int n0, int cofs, const uint32_t *acc, const unsigned char *sU) {
                if (leader && cofs == 0) {
                    const unsigned long long g = g_next, loc = P::read_thr(s, row);
                    if (loc > g && loc > g_sent) {
                        atomicMax(gwin, loc);
                        g_sent = loc;
                    }
                    if (g > loc) P::publish_thr(s, row, g);
                    g_next = tc::ld_relaxed_gpu_u64(gwin);
                }
                const int cb = col0 + cofs, vb = n0 + cb;  // the block's first column: in the tile, in V
                if (vb >= c1) return;
                // block b = vb / 16 draws words 2 (b mod 2), 2 (b mod 2) + 1 of the Philox
                // call (b / 2, k, request, cycle): an even block and the odd one after it,
                // when the same warp takes it next, share one call
                uint32_t wr, we;
                const bool odd = (vb & 16) != 0;
                if (!odd || cofs == 0) {
                    const uint4 w4 = philox4x32_10((uint32_t)(vb >> 5), c3, prow, p.rk);
                    wr = odd ? w4.z : w4.x;
                    we = odd ? w4.w : w4.y;
                    w_odd = make_uint2(w4.z, w4.w);
                } else {
                    wr = w_odd.x;
                    we = w_odd.y;
                }
                float z[16];
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    const uint4 uu = P::u_oct(sU, row, cb + 8 * o);
                    const uint32_t u[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 zz = add2(make_float2(__uint_as_float(acc[8 * o + 2 * i]),
                                                           __uint_as_float(acc[8 * o + 2 * i + 1])),
                                               make_float2(tcp::bf16_lo(u[i]), tcp::bf16_hi(u[i])));
                        z[8 * o + 2 * i] = zz.x;
                        z[8 * o + 2 * i + 1] = zz.y;
                    }
                }
                if (vb + 16 > c1) {
                    // the vocabulary ends inside this block
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (vb + j >= c1) z[j] = -INFINITY;
                }
                if (block_feed16(st, z, vb, wr, we, P::read_thr(s, row)) && row_live)
                    P::publish_thr(s, row, pack_winner(st.best, st.idx));
            });

            // The next step needs only x_k: fold the CTA's winner of each request (its
            // shared threshold word, which holds the best of all its threads) into the
            // step's winner word and publish right away; the partials (m, S, ...) that
            // lse_k and log q_k need after the last step follow off this path.  Only the
            // last step publishes after its partials, since they are read right after.
            tc::named_bar_sync(1, tcp::kEpiThreads);  // every warp past its last accumulator
            const bool last = step + 1 == p.nsteps;
            if (!last) {
                if (et < P::MV && m0 + et < p.R) {
                    const unsigned long long wbest = s.thr[et];
                    if (wbest != 0ull) atomicMax(win + m0 + et, wbest);
                }
                tc::named_bar_sync(1, tcp::kEpiThreads);
                if (et == 0) {
                    __threadfence();  // cumulative over the CTA's writes before the barrier
                    atomicAdd(ctr, 1);
                }
            }
            // merge the TPR threads of each request (fixed warp order) into this CTA's partial
            mg[et] = st.m;
            mg[tcp::kEpiThreads + et] = st.S;
            mg[2 * tcp::kEpiThreads + et] = st.best;
            mg[3 * tcp::kEpiThreads + et] = st.zbest;
            reinterpret_cast<int *>(mg)[4 * tcp::kEpiThreads + et] = st.idx;
            tc::named_bar_sync(1, tcp::kEpiThreads);
            if (et < P::MV) s.thr[et] = 0ull;  // the next step starts afresh
            if (et < P::MV && m0 + et < p.R) {
                RowState f;
                row_init(f);
                const int wstep = P::DUAL ? 2 : 4;  // warps holding the same request
                for (int w = et >> 5; w < tcp::kEpiWarps; w += wstep) {
                    const int src = w * 32 + (et & 31);
                    row_merge(f, mg[src], mg[tcp::kEpiThreads + src], mg[2 * tcp::kEpiThreads + src],
                              mg[3 * tcp::kEpiThreads + src], reinterpret_cast<int *>(mg)[4 * tcp::kEpiThreads + src]);
                }
                part[(size_t)(m0 + et) * p.nparts + cv] = make_partial(f.m, f.S, f.best, f.zbest, f.idx);
                if (last && f.idx >= 0) atomicMax(win + m0 + et, pack_winner(f.best, f.idx));
            }
            if (last) {
                tc::named_bar_sync(1, tcp::kEpiThreads);
                if (et == 0) {
                    __threadfence();
                    atomicAdd(ctr, 1);
                }
            } else if (et < P::MV && m0 + et < p.R) {
                // pull the W_1 row of the request's best token so far into L2: the winning
                // CTA's candidate is there when the next operand is gathered
                const unsigned long long wnow = tc::ld_relaxed_gpu_u64(win + m0 + et);
                const int xi = wnow != 0ull ? winner_index(wnow) : -1;
                if (xi >= 0 && xi < p.V) {
                    const char *rowp = reinterpret_cast<const char *>(p.W1 + (size_t)xi * p.r);
                    for (int b = 0; b < p.r * 2; b += 128) tc::prefetch_l2(rowp + b);
                }
            }

            // wait (bounded) until every CTA of the M-tile has published this step
            if (!mtile_sync<P>(p, s, ctr, ++phase, et, false)) break;
            if (step + 1 < p.nsteps) {
                // x_k of the M-tile's rows (the next step's x_{k-1})
                if (et < P::MV) {
                    int x = -1;
                    if (m0 + et < p.R) {
                        x = winner_index(__ldcg(win + m0 + et));
                        if (x < 0 || x >= p.V) x = 0;  // no winner: reported by the finaliser
                    }
                    s.tok[et] = x;
                }
                tc::named_bar_sync(1, tcp::kEpiThreads);
                if constexpr (P::KSPLIT == 2) {
                    // RNN head: the state update of step k + 1 over the M-tile's CTAs,
                    // then its operand A_{k+1} (prepared by those CTAs) is copied in
                    rnn_state_update<P>(p, s, m0, m_tile, cv, k + 1, et);
                    if (!mtile_sync<P>(p, s, ctr, ++phase, et, true)) break;
                    if (et == 0) rnn_load_operand<P>(p, s, m_tile, op_copies);
                    ++op_copies;
                } else {
                    // the next operand W_1[x_k], then the MMA warp goes
                    gather_operand<P>(p, s, m0, k + 1, et, tcp::kEpiThreads);
                    P::operand_written(s, et);
                }
            }
        }
        // lse_k and log q_k of every step of the launch: (step, request) pairs of
        // the M-tile over all its CTAs' warps, one pair per warp at a time
        if (!*s.abort_flag) {
            const int npairs = p.nsteps * P::MV;
            for (int pi = cv * tcp::kEpiWarps + warp; pi < npairs; pi += p.nparts * tcp::kEpiWarps) {
                const int si = pi / P::MV, i = pi - si * P::MV;
                if (m0 + i < p.R)
                    finalise_row(p, p.part + (size_t)(p.step_index + si - 1) * p.R * p.nparts, m0 + i, p.k + si, lane);
            }
            // the confidences c_k of every (step, request) pair of the M-tile, spread
            // over all its CTAs' warps (kept off the step boundary, where the slowest
            // CTA of the M-tile would carry them); x_{k-1} is the launch's input token
            // for its first step, else the previous step's winner (as the operand took it)
            for (int pi = cv * tcp::kEpiWarps + warp; pi < p.nsteps * P::MV; pi += p.nparts * tcp::kEpiWarps) {
                const int si = pi / P::MV, gr = m0 + (pi - si * P::MV);
                if (gr >= p.R) continue;
                int xp;
                if (si == 0) {
                    xp = load_token(p, gr, p.x_prev, p.x_stride);
                } else {
                    xp = winner_index(__ldcg(p.winners + (size_t)(p.step_index + si - 2) * p.R + gr));
                    if (xp < 0 || xp >= p.V) xp = 0;
                }
                confidence_warp(p, p.k + si, gr, xp, lane);
            }
        }
    }
    P::teardown(s);
}

// Self-check of the two bounded waits the tensor-core kernels use, on a
// condition that nothing satisfies unless the caller set it: mode 0 waits for
// *flag >= target like the cross-CTA counter waits; mode 1 waits on an
// mbarrier phase that completes only when target <= 0 (one arrival), like the
// pipeline waits.  Either returns after limit_ns with DSPARK_ERR_TIMEOUT in
// *err instead of hanging.
__global__ void wait_selfcheck_kernel(const int *flag, int target, int mode, uint64_t limit_ns, int32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (mode == 0) {
        wait_counter(flag, target, err, limit_ns);
        return;
    }
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
    if (target <= 0) tc::mbar_arrive(&bar);
    tc::mbar_wait(&bar, 0u, &abort_flag, err, limit_ns);
}

// pipeline configurations
// Pipe<requests per M-tile, vocabulary tile, W_2^T slab ring, U ring, operand split>
using DraftM64 = tcp::Pipe<64, 256, 3, 4, 1>;   // Markov, R <= 64 (U in 128-column parts)
using DraftM128 = tcp::Pipe<128, 256, 2, 3, 1>;  // Markov, 128 requests per M-tile (U in 128-column parts)
using DraftRnn = tcp::Pipe<128, 128, 2, 2, 2>;  // RNN (fp32 operand split hi/lo: 128 KB, so a 2-slot W_2^T ring)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class P>
cudaError_t launch_cfg(const DraftStep &p, int nparts, int n_mtiles, cudaStream_t s) {
    CUtensorMap tmB, tmU;
    if (!encode_w2t_map(&tmB, p.W2t, p.V, p.r, P::BN)) return cudaErrorInvalidValue;
    if (!encode_u_map(&tmU, p.U, p.R, p.gamma, p.V, P::MV)) return cudaErrorInvalidValue;
    TcParams tp;
    tp.R = p.R; tp.V = p.V; tp.r = p.r; tp.d = p.d; tp.gamma = p.gamma; tp.k = p.k;
    tp.nsteps = p.nsteps > 0 ? p.nsteps : 1;
    tp.step_index = p.step_index;
    tp.phase0 = p.phase0;
    tp.h = static_cast<const __nv_bfloat16 *>(p.h); tp.w = p.w; tp.sts_T = p.sts_T;
    tp.counters = p.counters;
    tp.x = p.x_out; tp.logq = p.logq; tp.lse = p.lse; tp.c = p.c;
    tp.conf_logit = p.conf_logit;
    tp.W1 = static_cast<const __nv_bfloat16 *>(p.W1);
    tp.W2t = static_cast<const __nv_bfloat16 *>(p.W2t);
    tp.x_prev = p.x_prev; tp.x_stride = p.x_stride;
    tp.A_op = p.A_op; tp.a_stride = p.a_stride;
    tp.seed = p.seed; tp.cycle = p.cycle;
    tp.rk = philox_round_keys(p.seed);
    tp.part = p.part; tp.nparts = nparts;
    tp.winners = p.winners;
    tp.n_mtiles = n_mtiles;
    tp.err = p.err;
    tp.rnn = p.rnn;
    tp.a_stage = p.a_stage;
    auto kern = draft_step_tc<P>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kBytes);
    if (e != cudaSuccess) return e;
    // cooperative: the CTAs wait for one another at the end of the step
    void *args[] = {&tmB, &tmU, &tp};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(n_mtiles * nparts),
                                       dim3(P::kThreads), args, (size_t)P::kBytes, s);
}

}  // namespace

// ---------------------------------------------------------------- host helpers
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool tc_available() { return encode_fn() != nullptr && sm_count() > 0; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// W_2^T [V, r] bf16: boxes of 64 K-elements (128 bytes, swizzled) x BN rows
bool encode_w2t_map(CUtensorMap *m, const void *W2t, int V, int r, int BN) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)V};
    const cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(W2t), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// a bf16 [rows, K] matrix with row stride ld elements (K-major): boxes of 64
// K-elements (128 bytes, swizzled) x box_rows rows
bool encode_kmajor_map(CUtensorMap *m, const void *base, int rows, int K, int ld, int box_rows) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// U [R, gamma, V] bf16: boxes of 64 vocabulary entries x 1 step x MV requests
bool encode_u_map(CUtensorMap *m, const void *U, int R, int gamma, int V, int MV) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)gamma * V * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)MV};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(U), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_kernels_enabled() {
    static const bool on = [] {
        const char *v = getenv("DSPARK_DRAFT_KERNEL");
        return !(v && v[0] == 's');  // "simt": CUDA-core kernels only
    }();
    return on;
}

bool draft_step_tc_supported(const DraftStep &p) {
    return tc_kernels_enabled() && p.dtype == DSPARK_BF16 && p.r % 64 == 0 && p.r >= 64 && p.r <= 256 &&
           p.V % 8 == 0 && aligned16(p.U) && aligned16(p.W1) && aligned16(p.W2t) &&
           (p.A_op == nullptr || (aligned16(p.A_op) && p.a_stride % 4 == 0)) && tc_available();
}

void tc_grid_shape(int R, int V, int MV, int BN, int *nparts, int *n_mtiles) {
    const int mt = (R + MV - 1) / MV;
    int g = sm_count() / mt;
    if (g < 1) g = 1;
    const int nv = (V + BN - 1) / BN;
    if (g > nv) g = nv;
    *nparts = g;
    *n_mtiles = mt;
}

void draft_step_tc_shape(int R, int V, bool rnn, int *nparts, int *n_mtiles) {
    if (rnn) tc_grid_shape(R, V, DraftRnn::MV, DraftRnn::BN, nparts, n_mtiles);
    else if (R <= 64) tc_grid_shape(R, V, DraftM64::MV, DraftM64::BN, nparts, n_mtiles);
    else tc_grid_shape(R, V, DraftM128::MV, DraftM128::BN, nparts, n_mtiles);
}

cudaError_t launch_wait_selfcheck(const int *flag, int target, int mode, uint64_t limit_ns, int32_t *err,
                                  cudaStream_t s) {
    wait_selfcheck_kernel<<<1, 1, 0, s>>>(flag, target, mode, limit_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_draft_step_tc(const DraftStep &p, cudaStream_t s) {
    const bool rnn = p.A_op != nullptr;
    int nparts = 0, mt = 0;
    draft_step_tc_shape(p.R, p.V, rnn, &nparts, &mt);
    if (nparts != p.nparts) return cudaErrorInvalidValue;
    if (rnn) return launch_cfg<DraftRnn>(p, nparts, mt, s);
    if (p.R <= 64) return launch_cfg<DraftM64>(p, nparts, mt, s);
    return launch_cfg<DraftM128>(p, nparts, mt, s);
}

}  // namespace dspark
