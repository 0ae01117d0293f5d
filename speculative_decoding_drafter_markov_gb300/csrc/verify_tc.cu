// verify_tc.cu -- verification phase 2 on the tensor cores.
//
// "DSpark explained" section 06: at the first rejected position n of request
// r the correction is drawn from norm(max(0, p_n - q_{n+1})); if every
// scheduled token passed, the bonus token is drawn from p_{l_r}.  q_{n+1}
// needs the draft logits of step n+1 again: U_{n+1} + (bias operand) W_2.
// That contraction runs on tcgen05 exactly like the draft step (shared
// pipeline in tc_pipe.cuh); the epilogue streams the target row p_n and the
// base-logit row U_{n+1} of each request from global memory, forms the weights
// (the residual, or p for the bonus) and keeps only their 16-column chunk sums
// and each CTA's total.  After the M-tile's CTAs meet, one warp per request
// draws the token by inverse CDF with the stream-2 uniform: CTA, chunk, entry.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tc_pipe.cuh"
#include "verify_common.cuh"

namespace dspark {

namespace {

// Per-thread staging of the target and base rows: every epilogue thread copies
// the 32 + 32 bytes of its next 16-column chunk with cp.async while it works on
// the current one (two stages).  Stage s, piece k (0-1 target, 2-3 base, 16 B
// each) of thread et sits at ((s 4 + k) kEpiThreads + et) 16: a warp's reads of
// one piece are 32 consecutive 16-byte words (no bank conflicts).
constexpr int kStagePieces = 4;
constexpr int kStageBytes = 2 * kStagePieces * tcp::kEpiThreads * 16;

struct VerifyTcParams {
    int R, V, r, gamma;
    const __nv_bfloat16 *T, *U, *W1, *W2t;
    const float *A;  // RNN bias operands [R, gamma, r] or null
    const int32_t *anchor, *x;
    const float *lse;  // draft log-sum-exp [R, gamma]
    VerifyWs w;
    int nparts, n_mtiles, n_vtiles;
    uint64_t seed, cycle;
    int32_t *err;
    dspark_verify_args a;  // outputs and the rest of the call (the outcome writer)
};

__device__ __forceinline__ void cp_async_stage(uint4 *dst, const __nv_bfloat16 *src, uint32_t bytes, uint64_t pol) {
    tc::cp_async16(dst, src, bytes, pol);
}

// The correction / bonus draw of request rq by one warp (all lanes; lane 0's
// result is the warp's): inverse CDF over this request's CTA totals (stot), then
// over the chosen CTA's 16-column chunk sums (csum), then over the chosen
// chunk's weights, recomputed here -- p exactly as the tile pass formed it, the
// bias dot of q on the CUDA cores (two lanes per vocabulary entry) in place of
// the tensor-core one; the two agree to a few fp32 ulps, and a target that lands
// between them takes the chunk's last positive weight.  A rejected position
// whose residual came out empty (p equal to q to rounding everywhere) draws from
// p over the whole row.  The sums were written by other CTAs of this launch:
// they are read through L2.
template <class P>
__device__ __noinline__ int draw_correction(const VerifyTcParams &p, int rq) {
    const int lane = threadIdx.x & 31;
    const int ell = p.w.ell[rq];
    if (ell < 0) return -1;
    const int fr = p.w.first_rej[rq];
    const bool res = fr < ell;
    const int n = res ? fr : ell;
    const int row = p.w.row_of[rq * (p.gamma + 1) + n];
    if (row < 0) return -1;
    const float lsep = p.w.lse_p[row] * kLog2e;
    const __nv_bfloat16 *trow = p.T + (size_t)row * p.V;
    const float u = correction_uniform(p.seed, p.cycle, n, rq);
    const float *tot = p.w.stot + (size_t)rq * kVerifyMaxParts;
    auto get_tot = [&](int i) { return __ldcg(tot + i); };
    float below = 0.f, total = 0.f;
    warp_cdf_search(p.nparts, 0.f, INFINITY, get_tot, &below, &total);
    if (res && !(total > 0.f)) {
        auto pv = [&](int v) { return ex2(fmaf(__bfloat162float(trow[v]), kLog2e, -lsep)); };
        warp_cdf_search(p.V, 0.f, INFINITY, pv, &below, &total);
        return warp_cdf_search(p.V, 0.f, u * total, pv, &below);
    }
    const float target = u * total;
    const int c = warp_cdf_search(p.nparts, 0.f, target, get_tot, &below);
    if (c < 0) return -1;
    int t_begin, ntl;
    tcp::tile_range(c, p.nparts, p.n_vtiles, t_begin, ntl);
    const int v_begin = t_begin * P::BN, v_end = min((t_begin + ntl) * P::BN, p.V);
    const int ch0 = v_begin / 16;
    float b1 = 0.f;
    const int ch = warp_cdf_search((v_end - v_begin + 15) / 16, below, target,
                                   [&](int i) { return __ldcg(p.w.csum + (size_t)(ch0 + i) * p.R + rq); }, &b1);
    if (ch < 0) return -1;
    const int vb = (ch0 + ch) * 16;
    // entry j = lane / 2 of the chunk; lanes 2j and 2j + 1 split the bias dot in halves
    const int j = lane >> 1, v = vb + j;
    const bool inv = v < p.V;
    const float pv = inv ? ex2(fmaf(__bfloat162float(trow[v]), kLog2e, -lsep)) : 0.f;
    float diff = pv;  // p - q, or p
    if (res) {
        const int half = p.r / 2;  // a multiple of 32
        const uint4 *w2 = reinterpret_cast<const uint4 *>(p.W2t + (size_t)(inv ? v : 0) * p.r + (lane & 1) * half);
        float d = 0.f;
        if (p.A) {
            const float4 *av =
                reinterpret_cast<const float4 *>(p.A + ((size_t)rq * p.gamma + n) * (size_t)p.r + (lane & 1) * half);
            for (int k = 0; k < half / 8; ++k) {
                const uint4 wr = w2[k];
                const float4 a0 = av[2 * k], a1 = av[2 * k + 1];
                const float bw[8] = {tcp::bf16_lo(wr.x), tcp::bf16_hi(wr.x), tcp::bf16_lo(wr.y), tcp::bf16_hi(wr.y),
                                     tcp::bf16_lo(wr.z), tcp::bf16_hi(wr.z), tcp::bf16_lo(wr.w), tcp::bf16_hi(wr.w)};
                const float ba[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(ba[i], bw[i], d);
            }
        } else {
            int xn = n == 0 ? p.anchor[rq] : p.x[(size_t)rq * p.gamma + n - 1];
            if (xn < 0 || xn >= p.V) xn = 0;
            const uint4 *e1 = reinterpret_cast<const uint4 *>(p.W1 + (size_t)xn * p.r + (lane & 1) * half);
            for (int k = 0; k < half / 8; ++k) {
                const uint4 wr = w2[k], er = e1[k];
                const uint32_t ww[4] = {wr.x, wr.y, wr.z, wr.w}, ee[4] = {er.x, er.y, er.z, er.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    d = fmaf(tcp::bf16_lo(ee[i]), tcp::bf16_lo(ww[i]), d);
                    d = fmaf(tcp::bf16_hi(ee[i]), tcp::bf16_hi(ww[i]), d);
                }
            }
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if (inv) {
            const __nv_bfloat16 *urow = p.U + ((size_t)rq * p.gamma + n) * (size_t)p.V;
            const float lseq = p.lse[(size_t)rq * p.gamma + n] * kLog2e;
            const float q = ex2(fmaf(d + __bfloat162float(urow[v]), kLog2e, -lseq));
            diff = pv - q;
        }
    }
    const float wv = fmaxf(diff, 0.f);
    const float wi = __shfl_sync(0xffffffffu, wv, 2 * (lane & 15));  // lane i < 16: entry i
    float b2 = 0.f;
    int e = warp_cdf_search(min(16, p.V - vb), b1, target, [&](int) { return wi; }, &b2);
    if (e < 0) {
        // the chunk's sum was positive but no recomputed weight is: its entry with
        // the largest p - q (the lowest index among equals)
        float dv = inv ? diff : -INFINITY;
        int bi = j;
#pragma unroll
        for (int off = 2; off < 32; off <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, dv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (o > dv || (o == dv && oi < bi)) {
                dv = o;
                bi = oi;
            }
        }
        e = bi;
    }
    return vb + e;
}

template <class P, bool STAGE>
__global__ void __launch_bounds__(P::kThreads, 1)
    verify_phase2_tc(const __grid_constant__ CUtensorMap tmB, const VerifyTcParams p) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_mode[P::MV], s_n[P::MV], s_row[P::MV], s_xn[P::MV];
    __shared__ float s_lsep[P::MV], s_lseq[P::MV];
    typename P::State s = P::carve(smem_raw);
    P::init(s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.n_mtiles, cv = blockIdx.x / p.n_mtiles;
    const int m0 = m_tile * P::MV;
    int t_begin, ntiles;
    tcp::tile_range(cv, p.nparts, p.n_vtiles, t_begin, ntiles);
    const int kslabs = p.r / 64;

    // per request: residual (1) or bonus (0) sample, its position and row
    if (threadIdx.x < P::MV) {
        const int rq = m0 + threadIdx.x;
        int mode = -1, n = 0, row = 0, xn = 0;
        float lsep = 0.f, lseq = 0.f;
        if (rq < p.R) {
            const int ell = p.w.ell[rq];
            if (ell >= 0) {
                const int fr = p.w.first_rej[rq];
                mode = fr < ell ? 1 : 0;
                n = fr < ell ? fr : ell;
                row = p.w.row_of[rq * (p.gamma + 1) + n];
                if (row < 0) {
                    mode = -1;
                } else {
                    lsep = p.w.lse_p[row];
                    if (mode == 1) {
                        lseq = p.lse[(size_t)rq * p.gamma + n];
                        xn = n == 0 ? p.anchor[rq] : p.x[(size_t)rq * p.gamma + n - 1];
                        if (xn < 0 || xn >= p.V) xn = 0;
                    }
                }
            } else if (cv == 0) {
                set_err(p.err, DSPARK_ERR_INVAL);  // request missing from the batch
            }
        }
        s_mode[threadIdx.x] = mode;
        s_n[threadIdx.x] = n;
        s_row[threadIdx.x] = row;
        s_xn[threadIdx.x] = xn;
        s_lsep[threadIdx.x] = lsep;
        s_lseq[threadIdx.x] = lseq;
    }
    __syncthreads();  // row metadata, barriers and TMEM ready
    P::ready(s);

    // bias operand of q_{n+1}: W_1[x_n] (x_0 = anchor) or the RNN vector A_{n+1}
    const int chunks_per_row = p.r / 8;
    for (int e = threadIdx.x; e < P::MV * chunks_per_row; e += P::kThreads) {
        const int row = e / chunks_per_row, c = e - row * chunks_per_row;
        const int rq = m0 + row;
        const bool live = s_mode[row] == 1;
        if (P::KSPLIT == 1) {
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (live) val = *reinterpret_cast<const uint4 *>(p.W1 + (size_t)s_xn[row] * p.r + c * 8);
            P::put_a(s, row, c, 0, val);
        } else {
            float xs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (live) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    p.A + ((size_t)rq * p.gamma + s_n[row]) * (size_t)p.r + c * 8);
                const float4 a0 = src[0], a1 = src[1];
                xs[0] = a0.x; xs[1] = a0.y; xs[2] = a0.z; xs[3] = a0.w;
                xs[4] = a1.x; xs[5] = a1.y; xs[6] = a1.z; xs[7] = a1.w;
            }
            uint4 hi, lo;
            tcp::split8(xs, hi, lo);
            P::put_a(s, row, c, 0, hi);
            P::put_a(s, row, c, 1, lo);
        }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();  // operand complete

    if (warp == tcp::kProducerWarp) {
        if (lane == 0) tc::prefetch_tmap(&tmB);
        __syncwarp();
        if (lane == 0) P::producer_w2(s, &tmB, t_begin * P::BN, P::BN, ntiles, kslabs, 1, p.err);
        __syncwarp();
    } else if (warp == tcp::kMmaWarp) {
        if (lane == 0) P::mma(s, ntiles, kslabs, 1, p.err);
        __syncwarp();
    } else {
        const int et = threadIdx.x;
        const int row = P::epi_row(), col0 = P::epi_col0();
        const int rq = m0 + row;
        const bool row_live = rq < p.R;
        const int mode = s_mode[row], n = s_n[row];
        const float lsep = s_lsep[row] * kLog2e, lseq = s_lseq[row] * kLog2e;
        const __nv_bfloat16 *trow = p.T + (size_t)s_row[row] * p.V;
        const __nv_bfloat16 *urow = p.U + ((size_t)(row_live ? rq : 0) * p.gamma + (mode == 1 ? n : 0)) * (size_t)p.V;
        const uint64_t pol = tc::policy_evict_first();  // target and base rows are read once
        // One draw per request: by inverse CDF over the residual max(0, p - q) at a
        // rejected position (mode 1), over p for the bonus (mode 0).  This pass
        // forms the weights of each 16-column chunk, stores the chunk's sum
        // (csum, chunk-major: a warp's 32 rows are one 128-byte line) and keeps
        // this thread's running total; the draw itself follows the M-tile's
        // synchronisation point.
        float tot = 0.f;
        // staging (STAGE): chunk i of this thread lands in stage i % 2; the copy of
        // chunk i + 1 is in flight while chunk i is processed.  Without it, plain
        // loads at the start of each chunk.
        uint4 *stage = reinterpret_cast<uint4 *>((reinterpret_cast<uintptr_t>(s.smem) + P::kBytes - 1024 + 15) &
                                                 ~static_cast<uintptr_t>(15));
        const int c_end = min((t_begin + ntiles) * P::BN, p.V);  // end of this CTA's columns
        auto stage_chunk = [&](int i, int vb) {
            uint4 *dst = stage + (size_t)(i & 1) * kStagePieces * tcp::kEpiThreads + et;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const bool in = mode >= 0 && vb + 8 * c < c_end;
                cp_async_stage(dst + c * tcp::kEpiThreads, in ? trow + vb + 8 * c : trow, in ? 16u : 0u, pol);
                const bool inu = in && mode == 1;
                cp_async_stage(dst + (2 + c) * tcp::kEpiThreads, inu ? urow + vb + 8 * c : urow, inu ? 16u : 0u,
                               pol);
            }
            tc::cp_async_commit();
        };
        if (STAGE) stage_chunk(0, t_begin * P::BN + col0);
        int ci = 0;
        P::epilogue(s, 0, t_begin * P::BN, P::BN, ntiles, p.err,
                    [&](int, int n0, int cofs, const uint32_t *acc, const unsigned char *) {
            const int vb = n0 + col0 + cofs;  // 16 columns vb .. vb + 15; V % 8 == 0
            if (STAGE) {
                // the next chunk: the rest of this warp's block, else the next tile
                const int vnext = cofs + 16 < P::CW ? vb + 16 : n0 + P::BN + col0;
                if (vnext < c_end) {
                    stage_chunk(ci + 1, vnext);
                    tc::cp_async_wait<1>();
                } else {
                    tc::cp_async_wait<0>();
                }
            }
            // the chunk of the target row (and of U_{n+1}): this thread's stage, or
            // 16-byte loads (zeros beyond the CTA's columns)
            uint4 tq[2], uq[2];
            if (STAGE) {
                const uint4 *src = stage + (size_t)(ci & 1) * kStagePieces * tcp::kEpiThreads + et;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tq[c] = src[c * tcp::kEpiThreads];
                    uq[c] = src[(2 + c) * tcp::kEpiThreads];
                }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const bool in = mode >= 0 && vb + 8 * c < c_end;
                    tq[c] = in ? tc::ld_global_hint(trow + vb + 8 * c, pol) : make_uint4(0u, 0u, 0u, 0u);
                    uq[c] = (in && mode == 1) ? tc::ld_global_hint(urow + vb + 8 * c, pol) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ++ci;
            if (mode < 0 || vb >= c_end) return;
            // weights: residual max(0, p - q) (mode 1) or p (mode 0), zero beyond V;
            // paired fp32 operations, the chunk's sum in a fixed tree
            const float2 L2e = make_float2(kLog2e, kLog2e), nlp = make_float2(-lsep, -lsep),
                         nlq = make_float2(-lseq, -lseq);
            float2 sum[8];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t tt[4] = {tq[c].x, tq[c].y, tq[c].z, tq[c].w};
                const uint32_t uu[4] = {uq[c].x, uq[c].y, uq[c].z, uq[c].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = 8 * c + 2 * i;
                    const float2 pa = fma2(make_float2(tcp::bf16_lo(tt[i]), tcp::bf16_hi(tt[i])), L2e, nlp);
                    float2 w = make_float2(ex2(pa.x), ex2(pa.y));
                    if (mode == 1) {
                        const float2 z = add2(make_float2(__uint_as_float(acc[j]), __uint_as_float(acc[j + 1])),
                                              make_float2(tcp::bf16_lo(uu[i]), tcp::bf16_hi(uu[i])));
                        const float2 qa = fma2(z, L2e, nlq);
                        const float2 r = sub2(w, make_float2(ex2(qa.x), ex2(qa.y)));
                        w = make_float2(fmaxf(r.x, 0.f), fmaxf(r.y, 0.f));
                    }
                    sum[4 * c + i] = make_float2(vb + j < p.V ? w.x : 0.f, vb + j + 1 < p.V ? w.y : 0.f);
                }
            }
#pragma unroll
            for (int wd = 4; wd > 0; wd >>= 1)
#pragma unroll
                for (int i = 0; i < wd; ++i) sum[i] = add2(sum[i], sum[i + wd]);
            const float cs = sum[0].x + sum[0].y;
            if (row_live) p.w.csum[(size_t)(vb >> 4) * p.R + rq] = cs;
            tot += cs;
        });
        // this CTA's total of each request: its warps' totals in warp order
        tc::named_bar_sync(1, tcp::kEpiThreads);  // every warp past its last accumulator
        float *red = P::merge_scratch(s);
        red[et] = tot;
        tc::named_bar_sync(1, tcp::kEpiThreads);
        if (et < P::MV && m0 + et < p.R) {
            const int wstep = P::DUAL ? 2 : 4;  // warps holding the same request
            float t2 = 0.f;
            for (int w2 = et >> 5; w2 < tcp::kEpiWarps; w2 += wstep) t2 += red[w2 * 32 + (et & 31)];
            p.w.stot[(size_t)(m0 + et) * kVerifyMaxParts + cv] = t2;
        }

        // Every CTA of the M-tile publishes, waits (bounded; the launch is cooperative,
        // so all are resident) until all have, then draws its share of the
        // requests: rows cv, cv + nparts, ..., one warp per request.
        __threadfence();
        tc::named_bar_sync(1, tcp::kEpiThreads);
        if (et == 0) {
            atomicAdd(p.w.done + m_tile, 1);
            *s.flag = tc::wait_counter_ge(p.w.done + m_tile, p.nparts, p.err) ? 1 : 0;
        }
        tc::named_bar_sync(1, tcp::kEpiThreads);
        if (*s.flag) {
            __threadfence();
            for (int i = cv, nn = 0; i < P::MV && m0 + i < p.R; i += p.nparts, ++nn) {
                if (warp != nn % tcp::kEpiWarps) continue;
                const int y = draw_correction<P>(p, m0 + i);
                if (lane == 0) {
                    const int ell = p.w.ell[m0 + i], fr = p.w.first_rej[m0 + i];
                    const bool res = ell >= 0 && fr < ell;
                    write_outcome(p.a, p.w, m0 + i, res ? y : -1, res ? -1 : y);
                }
            }
        } else {
            *s.abort_flag = 1;
        }
    }
    P::teardown(s);
}

// Pipe<requests per M-tile, vocabulary tile, W_2^T slab ring, U ring (none), operand split>.
// The 128-request configuration stages its rows (64 KB, with a shorter W_2^T ring);
// measured against plain loads it was faster there and slower for 64 requests and
// the RNN operand.  With the static row metadata, all within 227 KB.
using VerifyM64 = tcp::Pipe<64, 128, 9, 0, 1>;
using VerifyM128 = tcp::Pipe<128, 128, 5, 0, 1>;
using VerifyRnn = tcp::Pipe<128, 64, 10, 0, 2>;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class P, bool STAGE>
cudaError_t launch_cfg(const dspark_verify_args &a, VerifyWs &w, cudaStream_t s) {
    int nparts = 0, mt = 0;
    tc_grid_shape(a.R, a.V, P::MV, P::BN, &nparts, &mt);
    CUtensorMap tmB;
    if (!encode_w2t_map(&tmB, a.W2t, a.V, a.r, P::BN)) return cudaErrorInvalidValue;
    w.nparts = nparts;
    VerifyTcParams tp;
    tp.R = a.R; tp.V = a.V; tp.r = a.r; tp.gamma = a.gamma;
    tp.T = static_cast<const __nv_bfloat16 *>(a.T);
    tp.U = static_cast<const __nv_bfloat16 *>(a.U);
    tp.W1 = static_cast<const __nv_bfloat16 *>(a.W1);
    tp.W2t = static_cast<const __nv_bfloat16 *>(a.W2t);
    tp.A = a.A;
    tp.anchor = a.anchor; tp.x = a.x; tp.lse = a.lse;
    tp.w = w;
    tp.nparts = nparts; tp.n_mtiles = mt; tp.n_vtiles = (a.V + P::BN - 1) / P::BN;
    tp.seed = a.seed; tp.cycle = a.cycle; tp.err = a.err;
    tp.a = a;
    auto kern = verify_phase2_tc<P, STAGE>;
    const int smem = P::kBytes + (STAGE ? kStageBytes + 16 : 0);  // + 16: the stage starts on a 16-byte boundary
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // cooperative: the CTAs of an M-tile wait for one another before the final merge
    void *args[] = {&tmB, &tp};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(mt * nparts), dim3(P::kThreads),
                                       args, (size_t)smem, s);
}

}  // namespace

bool verify_tc_supported(const dspark_verify_args &a) {
    return tc_kernels_enabled() && a.dtype == DSPARK_BF16 && a.r % 64 == 0 && a.r >= 64 && a.r <= 256 &&
           (a.R + 63) / 64 <= kVerifyMaxMTiles &&
           a.V % 8 == 0 && aligned16(a.T) && aligned16(a.U) && aligned16(a.W1) && aligned16(a.W2t) &&
           (a.A == nullptr || aligned16(a.A)) && tc_available();
}

cudaError_t launch_verify_phase2_tc(const dspark_verify_args &a, VerifyWs &w, cudaStream_t s) {
    if (a.A) return launch_cfg<VerifyRnn, false>(a, w, s);
    if (a.R <= 64) return launch_cfg<VerifyM64, false>(a, w, s);
    return launch_cfg<VerifyM128, true>(a, w, s);
}

}  // namespace dspark
