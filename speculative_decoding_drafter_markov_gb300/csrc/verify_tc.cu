// verify_tc.cu -- verification phase 2 on the tensor cores.
//
// "DSpark explained" section 06: at the first rejected position n of request
// r the correction is drawn from norm(max(0, p_n - q_{n+1})); if every
// scheduled token passed, the bonus token is drawn from p_{l_r}.  q_{n+1}
// needs the draft logits of step n+1 again: U_{n+1} + (bias operand) W_2.
// That contraction runs on tcgen05 exactly like the draft step (shared
// pipeline in tc_pipe.cuh); the CTAs of an M-tile take vocabulary tiles from a
// shared counter (dynamic order).  The epilogue streams the target row p_n and
// the base-logit row U_{n+1} of each request from global memory, forms the
// weights (the residual, or p for the bonus) and keeps only their sums: per
// 16-column chunk and per vocabulary tile.  After the M-tile's CTAs meet, one
// warp per request draws the token by inverse CDF with the stream-2 uniform:
// tile, chunk, entry.  The sums are indexed by vocabulary position, so the
// draw does not depend on which CTA took which tile.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tc_pipe.cuh"
#include "verify_common.cuh"

namespace dspark {

namespace {

// Per-thread staging of the target and base rows in NST stages: every epilogue
// thread copies the 32 + 32 bytes of its chunks NST - 1 ahead with cp.async
// while it works on the current one.  Stage s, piece k (0-1 target, 2-3 base,
// 16 B each) of thread et sits at ((s 4 + k) kEpiThreads + et) 16: a warp's reads
// of one piece are 32 consecutive 16-byte words (no bank conflicts).
constexpr int kStagePieces = 4;
template <int NST>
constexpr int stage_bytes() {
    return NST * kStagePieces * tcp::kEpiThreads * 16;
}

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

// Row metadata of the M-tile's requests, in shared memory: the sample mode (1
// residual at a rejected position, 0 bonus, -1 none), its position n, the
// flattened target row, x_n and the two log-sum-exps.
template <int MV>
struct RowMeta {
    int mode[MV], n[MV], row[MV], xn[MV];
    float lsep[MV], lseq[MV];
};

// The correction / bonus draw of request rq (local row i of the M-tile) by one
// warp (all lanes; every lane returns the token): inverse CDF over the
// request's vocabulary-tile totals (ttot, fixed point: the tile level is exact
// integer arithmetic), then over the chosen tile's
// 16-column chunk sums (csum), then over the chosen chunk's weights,
// recomputed here -- p exactly as the tile pass formed it, the bias dot of q on
// the CUDA cores in place of the tensor-core one; the two agree to a few fp32
// ulps, and a target that lands between them takes the chunk's last positive
// weight.  A rejected position whose residual came out empty (p equal to q to
// rounding everywhere) draws from p over the whole row.  The sums were written
// by other CTAs of this launch: they are read through L2.
//
// Tile level: the sums of the runs of 32 tiles give the total and the run
// holding the target, a scan of that run's tiles the tile.
template <class P>
__device__ __noinline__ int draw_correction(const VerifyTcParams &p, const RowMeta<P::MV> &md, int i, int rq) {
    const int lane = threadIdx.x & 31;
    const int mode = md.mode[i];
    if (mode < 0) return -1;
    const bool res = mode == 1;
    const int n = md.n[i];
    const float lsep = md.lsep[i] * kLog2e;
    const __nv_bfloat16 *trow = p.T + (size_t)md.row[i] * p.V;
    const float u = correction_uniform(p.seed, p.cycle, n, rq);
    const unsigned long long *tt = p.w.ttot + rq;                            // tile t at tt[t R]
    const unsigned long long *st = p.w.ttot + (size_t)p.n_vtiles * p.R + rq;  // run s at st[s R]
    const int nt = p.n_vtiles, ns = (nt + 31) / 32;
    // the runs' sums, lane l holding runs l, l + 32, ...; the total (exact)
    constexpr int kRuns = 4;  // up to 128 runs of 32 tiles: V <= 524288 at 128-wide tiles
    unsigned long long rs[kRuns];
#pragma unroll
    for (int j = 0; j < kRuns; ++j) rs[j] = 32 * j + lane < ns ? __ldcg(st + (size_t)(32 * j + lane) * p.R) : 0ull;
    unsigned long long lt = 0ull;
#pragma unroll
    for (int j = 0; j < kRuns; ++j) lt += rs[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    const unsigned long long total = lt;  // integer sums: the same on every lane
    if (total == 0ull) {
        if (!res) return -1;
        // empty residual: p over the whole row
        float below = 0.f;
        auto pv = [&](int v) { return ex2(fmaf(__bfloat162float(trow[v]), kLog2e, -lsep)); };
        const float ptot = warp_weight_sum<8>(p.V, pv);
        return warp_cdf_search<8>(p.V, 0.f, u * ptot, pv, &below);
    }
    // the target u * total (below total); the run, then the tile, whose
    // cumulative sum first passes it: exact integer sums, so neither depends on
    // the order of the additions
    const unsigned long long target = (unsigned long long)((double)u * (double)total);
    unsigned long long carry = 0ull;
    int srun = -1;
    unsigned long long base = 0ull;
#pragma unroll
    for (int j = 0; j < kRuns; ++j) {
        if (srun < 0 && 32 * j < ns) {
            unsigned long long c = rs[j];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long o = __shfl_up_sync(0xffffffffu, c, off);
                if (lane >= off) c += o;
            }
            const unsigned long long cum_in = carry + c;
            const unsigned h = __ballot_sync(0xffffffffu, rs[j] > 0ull && cum_in > target);
            if (h) {
                const int l = __ffs(h) - 1;
                srun = 32 * j + l;
                base = __shfl_sync(0xffffffffu, cum_in - rs[j], l);
            }
            carry = __shfl_sync(0xffffffffu, cum_in, 31);
        }
    }
    if (srun < 0) return -1;  // cannot happen: target < total
    const int tb = 32 * srun;
    const unsigned long long tv64 = tb + lane < nt ? __ldcg(tt + (size_t)(tb + lane) * p.R) : 0ull;
    unsigned long long c = tv64;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) c += o;
    }
    const unsigned long long cum_in = base + c;
    const unsigned h2 = __ballot_sync(0xffffffffu, tv64 > 0ull && cum_in > target);
    const unsigned p2 = __ballot_sync(0xffffffffu, tv64 > 0ull);
    const int l2 = h2 ? __ffs(h2) - 1 : (p2 ? 31 - __clz(p2) : -1);  // the last positive: cannot happen
    if (l2 < 0) return -1;
    const int t = tb + l2;
    const unsigned long long below_t = __shfl_sync(0xffffffffu, cum_in - tv64, l2);
    if (t < 0) return -1;
    const float below = (float)((double)below_t * (1.0 / kFixScale));
    const float target_f = (float)((double)target * (1.0 / kFixScale));
    const int ch0 = t * (P::BN / 16);
    const int nch = (min(P::BN, p.V - t * P::BN) + 15) / 16;
    float b1 = 0.f;
    const int ch = warp_cdf_search(nch, below, target_f,
                                   [&](int c) { return __ldcg(p.w.csum + (size_t)(ch0 + c) * p.R + rq); }, &b1);
    if (ch < 0) return -1;
    const int vb = (ch0 + ch) * 16;
    // Entry l / 2 of the chunk on lane l (lanes 2m, 2m + 1 share one); its
    // target and base logits are fetched first.
    const int el = lane >> 1, v = vb + el;
    const bool inv = v < p.V;
    const __nv_bfloat16 *urow = p.U + ((size_t)rq * p.gamma + n) * (size_t)p.V;
    const float tv = inv ? __bfloat162float(trow[v]) : 0.f;
    const float uv = (inv && res) ? __bfloat162float(urow[v]) : 0.f;
    float diff = inv ? ex2(fmaf(tv, kLog2e, -lsep)) : 0.f;  // p - q, or p
    if (res) {
        // the bias dot of the 16 entries: lane l holds inputs 8 l .. 8 l + 7 of
        // every entry (lanes with 8 l >= r hold none); then a halving butterfly
        // leaves the dot of entry e(l) on lane l
        float bias[8];
        const bool kin = 8 * lane < p.r;
        if (p.A) {
            const float4 *av = reinterpret_cast<const float4 *>(p.A + ((size_t)rq * p.gamma + n) * (size_t)p.r);
            const float4 a0 = kin ? av[2 * lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 a1 = kin ? av[2 * lane + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
            bias[0] = a0.x; bias[1] = a0.y; bias[2] = a0.z; bias[3] = a0.w;
            bias[4] = a1.x; bias[5] = a1.y; bias[6] = a1.z; bias[7] = a1.w;
        } else {
            const uint4 er = kin ? reinterpret_cast<const uint4 *>(p.W1 + (size_t)md.xn[i] * p.r)[lane]
                                 : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ee[4] = {er.x, er.y, er.z, er.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                bias[2 * e] = tcp::bf16_lo(ee[e]);
                bias[2 * e + 1] = tcp::bf16_hi(ee[e]);
            }
        }
        float d[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint4 wr[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int ve = vb + 8 * hh + e;
                wr[e] = (kin && ve < p.V) ? reinterpret_cast<const uint4 *>(p.W2t + (size_t)ve * p.r)[lane]
                                          : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t ww[4] = {wr[e].x, wr[e].y, wr[e].z, wr[e].w};
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc = fmaf(bias[2 * c], tcp::bf16_lo(ww[c]), acc);
                    acc = fmaf(bias[2 * c + 1], tcp::bf16_hi(ww[c]), acc);
                }
                d[8 * hh + e] = acc;
            }
        }
        // halving butterfly: across lanes 16 apart the lane keeps the entries whose
        // bit 3 equals its lane bit 4 and adds its partner's share of them; then
        // bit 2 against lane bit 3 (lanes 8 apart), bit 1 / lane bit 2, bit 0 /
        // lane bit 1, so lane l ends with entry l / 2, summed over all lanes
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int h = (lane >> 4) & 1;
            const float keep = h ? d[e + 8] : d[e], send = h ? d[e] : d[e + 8];
            d[e] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = (lane >> 3) & 1;
            const float keep = h ? d[e + 4] : d[e], send = h ? d[e] : d[e + 4];
            d[e] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = (lane >> 2) & 1;
            const float keep = h ? d[e + 2] : d[e], send = h ? d[e] : d[e + 2];
            d[e] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
            const int h = (lane >> 1) & 1;
            const float keep = h ? d[1] : d[0], send = h ? d[0] : d[1];
            d[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const float dot = d[0] + __shfl_xor_sync(0xffffffffu, d[0], 1);
        if (inv) diff -= ex2(fmaf(dot + uv, kLog2e, -md.lseq[i] * kLog2e));
    }
    const float wv = fmaxf(diff, 0.f);
    const float wi = __shfl_sync(0xffffffffu, wv, 2 * (lane & 15));  // lane e < 16: entry e
    float b2 = 0.f;
    int e = warp_cdf_search(min(16, p.V - vb), b1, target_f, [&](int) { return wi; }, &b2);
    if (e < 0) {
        // the chunk's sum was positive but no recomputed weight is: its entry with
        // the largest p - q (the lowest index among equals)
        float dv = inv ? diff : -INFINITY;
        int bi = el;
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

template <class P, int NST>
__global__ void __launch_bounds__(P::kThreads, 1)
    verify_phase2_tc(const __grid_constant__ CUtensorMap tmB, const VerifyTcParams p) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ RowMeta<P::MV> md;
    __shared__ uint32_t s_ring[P::kTileRing];
    typename P::State s = P::carve(smem_raw);
    P::init(s);
    P::ring_init(s_ring);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.n_mtiles, cv = blockIdx.x / p.n_mtiles;
    const int m0 = m_tile * P::MV;
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
        md.mode[threadIdx.x] = mode;
        md.n[threadIdx.x] = n;
        md.row[threadIdx.x] = row;
        md.xn[threadIdx.x] = xn;
        md.lsep[threadIdx.x] = lsep;
        md.lseq[threadIdx.x] = lseq;
    }
    __syncthreads();  // row metadata, barriers, tile ring and TMEM ready
    P::ready(s);

    if (warp == tcp::kProducerWarp) {
        // W_2^T does not depend on the requests: its slabs stream while the operand is built
        if (lane == 0) {
            tc::prefetch_tmap(&tmB);
            P::producer_w2_dyn(s, &tmB, s_ring, p.w.tctr + m_tile, p.n_vtiles, kslabs, p.err);
        }
        __syncwarp();
    } else if (warp == tcp::kMmaWarp) {
        if (lane == 0) P::mma_dyn(s, s_ring, kslabs, p.err);
        __syncwarp();
    } else {
        const int et = threadIdx.x;
        // bias operand of q_{n+1}: W_1[x_n] (x_0 = anchor) or the RNN vector A_{n+1}
        const int chunks_per_row = p.r / 8;
        for (int e = et; e < P::MV * chunks_per_row; e += tcp::kEpiThreads) {
            const int row = e / chunks_per_row, c = e - row * chunks_per_row;
            const int rq = m0 + row;
            const bool live = md.mode[row] == 1;
            if (P::KSPLIT == 1) {
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (live) val = *reinterpret_cast<const uint4 *>(p.W1 + (size_t)md.xn[row] * p.r + c * 8);
                P::put_a(s, row, c, 0, val);
            } else {
                float xs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (live) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.A + ((size_t)rq * p.gamma + md.n[row]) * (size_t)p.r + c * 8);
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
        P::operand_written(s, et);  // the MMA issuer starts

        const int row = P::epi_row(), col0 = P::epi_col0();
        const int rq = m0 + row;
        const bool row_live = rq < p.R;
        const int mode = md.mode[row], n = md.n[row];
        const float lsep = md.lsep[row] * kLog2e, lseq = md.lseq[row] * kLog2e;
        const __nv_bfloat16 *trow = p.T + (size_t)md.row[row] * p.V;
        const __nv_bfloat16 *urow = p.U + ((size_t)(row_live ? rq : 0) * p.gamma + (mode == 1 ? n : 0)) * (size_t)p.V;
        const uint64_t pol = tc::policy_evict_first();  // target and base rows are read once
        // One draw per request: by inverse CDF over the residual max(0, p - q) at a
        // rejected position (mode 1), over p for the bonus (mode 0).  This pass
        // forms the weights of each 16-column chunk and stores the chunk's sum
        // (csum, chunk-major: a warp's 32 rows are one 128-byte line) and adds its
        // share of each tile's sum into ttot in 2^-47 fixed point, and into the sum
        // of its run of 32 tiles (integer addition, so the order of the
        // additions does not matter);
        // the draw itself follows the M-tile's synchronisation point.
        float tsum = 0.f;
        // staging (NST stages): chunk i of this thread lands in stage i % NST; the
        // copies of chunks i + 1 .. i + NST - 1 are in flight while chunk i is
        // processed (a chunk past the CTA's last tile is an empty copy group).
        // Without (NST = 0), plain loads at the start of each chunk.
        constexpr int CPT = P::CW / 16;  // a thread's chunks per tile
        uint4 *stage = reinterpret_cast<uint4 *>((reinterpret_cast<uintptr_t>(s.smem) + P::kBytes - 1024 + 15) &
                                                 ~static_cast<uintptr_t>(15));
        auto chunk_vb = [&](int c) {  // vocabulary column of this thread's chunk c, or V: none
            const int t = P::ring_read(s_ring, c / CPT, s.abort_flag, p.err);
            return t >= 0 ? t * P::BN + col0 + 16 * (c % CPT) : p.V;
        };
        auto stage_chunk = [&](int i, int vb) {
            uint4 *dst = stage + (size_t)(i % (NST > 0 ? NST : 1)) * kStagePieces * tcp::kEpiThreads + et;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const bool in = mode >= 0 && vb + 8 * c < p.V;
                cp_async_stage(dst + c * tcp::kEpiThreads, in ? trow + vb + 8 * c : trow, in ? 16u : 0u, pol);
                const bool inu = in && mode == 1;
                cp_async_stage(dst + (2 + c) * tcp::kEpiThreads, inu ? urow + vb + 8 * c : urow, inu ? 16u : 0u,
                               pol);
            }
            tc::cp_async_commit();
        };
        if (NST > 0)
            for (int c = 0; c < NST - 1; ++c) stage_chunk(c, chunk_vb(c));
        int ci = 0;
        P::epilogue_dyn(s, s_ring, p.err, [&](int k, int tile, int cofs, const uint32_t *acc) {
            const int vb = tile * P::BN + col0 + cofs;  // 16 columns vb .. vb + 15; V % 8 == 0
            if (NST > 0) {
                stage_chunk(ci + NST - 1, chunk_vb(ci + NST - 1));
                tc::cp_async_wait<(NST > 0 ? NST - 1 : 0)>();  // chunk ci has landed
            }
            // the chunk of the target row (and of U_{n+1}): this thread's stage, or
            // 16-byte loads (zeros beyond V)
            uint4 tq[2], uq[2];
            if (NST > 0) {
                const uint4 *src = stage + (size_t)(ci % (NST > 0 ? NST : 1)) * kStagePieces * tcp::kEpiThreads + et;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tq[c] = src[c * tcp::kEpiThreads];
                    uq[c] = src[(2 + c) * tcp::kEpiThreads];
                }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const bool in = mode >= 0 && vb + 8 * c < p.V;
                    tq[c] = in ? tc::ld_global_hint(trow + vb + 8 * c, pol) : make_uint4(0u, 0u, 0u, 0u);
                    uq[c] = (in && mode == 1) ? tc::ld_global_hint(urow + vb + 8 * c, pol) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ++ci;
            if (mode >= 0 && vb < p.V) {
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
                        const int jj = 8 * c + 2 * i;
                        const float2 pa = fma2(make_float2(tcp::bf16_lo(tt[i]), tcp::bf16_hi(tt[i])), L2e, nlp);
                        float2 w = make_float2(ex2(pa.x), ex2(pa.y));
                        if (mode == 1) {
                            const float2 z = add2(make_float2(__uint_as_float(acc[jj]), __uint_as_float(acc[jj + 1])),
                                                  make_float2(tcp::bf16_lo(uu[i]), tcp::bf16_hi(uu[i])));
                            const float2 qa = fma2(z, L2e, nlq);
                            const float2 r = sub2(w, make_float2(ex2(qa.x), ex2(qa.y)));
                            w = make_float2(fmaxf(r.x, 0.f), fmaxf(r.y, 0.f));
                        }
                        sum[4 * c + i] = make_float2(vb + jj < p.V ? w.x : 0.f, vb + jj + 1 < p.V ? w.y : 0.f);
                    }
                }
#pragma unroll
                for (int wd = 4; wd > 0; wd >>= 1)
#pragma unroll
                    for (int i = 0; i < wd; ++i) sum[i] = add2(sum[i], sum[i + wd]);
                const float cs = sum[0].x + sum[0].y;
                if (row_live) p.w.csum[(size_t)(vb >> 4) * p.R + rq] = cs;
                tsum += cs;
            }
            if (cofs + 16 == P::CW) {
                if (row_live && mode >= 0) {
                    const unsigned long long fx = to_fixed(tsum);
                    tc::red_add_u64(p.w.ttot + (size_t)tile * p.R + rq, fx);
                    tc::red_add_u64(p.w.ttot + (size_t)(p.n_vtiles + (tile >> 5)) * p.R + rq, fx);
                }
                tsum = 0.f;
            }
        });

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
                const int y = draw_correction<P>(p, md, i, m0 + i);
                write_outcome_warp(p.a, p.w, m0 + i, y);
            }
        } else {
            *s.abort_flag = 1;
        }
    }
    P::teardown(s);
}

// Pipe<requests per M-tile, vocabulary tile, W_2^T slab ring, U ring (none), operand split>.
// The 128-request configuration stages its rows three deep (96 KB, with a W_2^T
// ring of three slabs: the MMA is far ahead of the epilogue anyway); measured
// against plain loads staging was faster there and slower for 64 requests and the
// RNN operand, and three stages were 1-2 % faster than two with a five-slab ring.
// With the static row metadata, all within 227 KB.
using VerifyM64 = tcp::Pipe<64, 128, 9, 0, 1>;
using VerifyM128 = tcp::Pipe<128, 128, 3, 0, 1>;
using VerifyRnn = tcp::Pipe<128, 64, 10, 0, 2>;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class P, int NST>
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
    auto kern = verify_phase2_tc<P, NST>;
    const int smem = P::kBytes + (NST > 0 ? stage_bytes<NST>() + 16 : 0);  // + 16: the stage starts on a 16-byte boundary
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
           (a.R + 63) / 64 <= kVerifyMaxMTiles && verify_tc_tiles(a) <= 4096 &&
           a.V % 8 == 0 && aligned16(a.T) && aligned16(a.U) && aligned16(a.W1) && aligned16(a.W2t) &&
           (a.A == nullptr || aligned16(a.A)) && tc_available();
}

int verify_tc_tiles(const dspark_verify_args &a) {
    const int bn = a.A ? VerifyRnn::BN : a.R <= 64 ? VerifyM64::BN : VerifyM128::BN;
    return (a.V + bn - 1) / bn;
}

cudaError_t launch_verify_phase2_tc(const dspark_verify_args &a, VerifyWs &w, cudaStream_t s) {
    if (a.A) return launch_cfg<VerifyRnn, 0>(a, w, s);
    if (a.R <= 64) return launch_cfg<VerifyM64, 0>(a, w, s);
    return launch_cfg<VerifyM128, 3>(a, w, s);
}

}  // namespace dspark
