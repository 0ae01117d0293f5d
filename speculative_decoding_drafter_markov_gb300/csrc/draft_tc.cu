// draft_tc.cu -- the draft step on the 5th-generation tensor cores.
//
// DSpark digest eq. (5): B_k = W_1[x_{k-1}] W_2 (Markov head) or eq. (6)
// B_k = W_2^T tanh(W_o z_k) (RNN head), contracted on tcgen05 into TMEM and
// consumed in place by the eq. (4) epilogue: U_k add, online max / sum-exp,
// Philox Gumbel race.  No logit reaches global memory.  The pipeline (TMA ring
// of W_2^T slabs and U_k tiles, MMA warp, TMEM staging) is tc_pipeline.cuh; this
// file supplies the bias operand and the per-tile epilogue.
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
#include "tc.cuh"
#include "tc_pipeline.cuh"

namespace dspark {

namespace {

struct TcParams {
    int R, V, r, d, gamma, k;
    const __nv_bfloat16 *W1;
    const int32_t *x_prev;
    int x_stride;
    const float *A_op;  // RNN: operand of row i at A_op[i * a_stride], else null
    int a_stride;
    const __nv_bfloat16 *h;  // [R, gamma, d]
    const float *w;          // [d + r]
    const float *sts_T;      // [gamma] or null
    uint64_t seed, cycle;
    DraftPartial *part;
    int *counters;           // [n_mtiles], zero on entry, left zero on exit
    int32_t *x;
    float *logq, *lse, *c;   // [R, gamma]
    int nparts;  // vocabulary ranges (CTAs per M-tile)
    int n_mtiles;
    int n_vtiles;
    int32_t *err;
};

// eq. (7): c_k = sigma(w^T [h_k ; W_1[x_{k-1}]] / T_k) of one request, by all
// epilogue threads (16-byte chunks of h_k then of W_1[x_{k-1}]), reduced in a
// fixed order through `red` (16 floats of shared memory).
__device__ __forceinline__ void confidence_row(const TcParams &p, int grow, int et, float *red) {
    int xp = p.x_prev[(size_t)grow * p.x_stride];
    if (xp < 0 || xp >= p.V) xp = 0;
    const __nv_bfloat16 *h = p.h + ((size_t)grow * p.gamma + (p.k - 1)) * (size_t)p.d;
    const __nv_bfloat16 *e = p.W1 + (size_t)xp * p.r;
    float dot = 0.f;
    if ((p.d & 7) == 0) {
        const int hc = p.d / 8, nc = hc + p.r / 8;
        for (int ch = et; ch < nc; ch += tcp::kEpiThreads) {
            const bool in_h = ch < hc;
            const uint4 raw = *reinterpret_cast<const uint4 *>(in_h ? h + ch * 8 : e + (ch - hc) * 8);
            const float *wv = p.w + ch * 8;  // w = [w_h ; w_e] lines up with [h ; e]
            const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dot = fmaf(wv[2 * i], tcp::bf16_lo(v[i]), dot);
                dot = fmaf(wv[2 * i + 1], tcp::bf16_hi(v[i]), dot);
            }
        }
    } else {
        for (int j = et; j < p.d + p.r; j += tcp::kEpiThreads)
            dot = fmaf(p.w[j], __bfloat162float(j < p.d ? h[j] : e[j - p.d]), dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if ((et & 31) == 0) red[et >> 5] = dot;
    tc::named_bar_sync(1, tcp::kEpiThreads);
    if (et == 0) {
        float sum = 0.f;
        for (int i = 0; i < tcp::kEpiThreads / 32; ++i) sum += red[i];
        const float T_k = p.sts_T ? p.sts_T[p.k - 1] : 1.0f;
        p.c[(size_t)grow * p.gamma + (p.k - 1)] = 1.0f / (1.0f + expf(-sum / T_k));
    }
    tc::named_bar_sync(1, tcp::kEpiThreads);
}

template <class P>
__global__ void __launch_bounds__(tcp::kThreads, 1)
    draft_step_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmU,
                  const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    typename P::State s = P::carve(smem_raw);
    P::init(s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.n_mtiles, cv = blockIdx.x / p.n_mtiles;
    const int m0 = m_tile * P::MV;
    int t_begin, ntiles;
    tcp::tile_range(cv, p.nparts, p.n_vtiles, t_begin, ntiles);
    const int kslabs = p.r / 64;

    __syncthreads();  // barriers initialised, TMEM allocated
    P::ready(s);
    if (warp == tcp::kProducerWarp) {
        // W_2^T and U_k do not depend on x_{k-1}: stream from the first cycle
        if (lane == 0) {
            tc::prefetch_tmap(&tmB);
            tc::prefetch_tmap(&tmU);
        }
        __syncwarp();
        P::producer(s, &tmB, &tmU, t_begin, ntiles, kslabs, p.k - 1, m0, p.err);
        __syncwarp();
        P::teardown(s);
        return;
    }

    // bias operand of the M-tile's rows, in the swizzled K-major layout, by every
    // thread except the producer warp
    const int chunks_per_row = p.r / 8;
    constexpr int kGather = tcp::kThreads - 32;
    const int gt = threadIdx.x < tcp::kEpiThreads ? threadIdx.x : threadIdx.x - 32;
    int *s_tok = reinterpret_cast<int *>(s.staging);  // staging is free until the first tile
    if (P::KSPLIT == 1) {
        if (gt < P::MV) {  // the M-tile's tokens first: one load per row, all in flight together
            const int grow = m0 + gt;
            int xp = grow < p.R ? p.x_prev[(size_t)grow * p.x_stride] : -1;
            if (grow < p.R && (xp < 0 || xp >= p.V)) {
                set_err(p.err, DSPARK_ERR_RANGE);
                xp = 0;
            }
            s_tok[gt] = xp;
        }
        tc::named_bar_sync(2, kGather);
    }
    for (int e = gt; e < P::MV * chunks_per_row; e += kGather) {
        const int row = e / chunks_per_row, c = e - row * chunks_per_row;
        const int grow = m0 + row;
        if (P::KSPLIT == 1) {
            const int xp = s_tok[row];
            const uint4 val = xp >= 0 ? *reinterpret_cast<const uint4 *>(p.W1 + (size_t)xp * p.r + c * 8)
                                      : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(P::a_chunk(s, row, c, 0)) = val;
        } else {
            float xs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (grow < p.R) {
                const float4 *src = reinterpret_cast<const float4 *>(p.A_op + (size_t)grow * p.a_stride + c * 8);
                const float4 a0 = src[0], a1 = src[1];
                xs[0] = a0.x; xs[1] = a0.y; xs[2] = a0.z; xs[3] = a0.w;
                xs[4] = a1.x; xs[5] = a1.y; xs[6] = a1.z; xs[7] = a1.w;
            }
            uint4 hi, lo;
            tcp::split8(xs, hi, lo);
            *reinterpret_cast<uint4 *>(P::a_chunk(s, row, c, 0)) = hi;
            *reinterpret_cast<uint4 *>(P::a_chunk(s, row, c, 1)) = lo;
        }
    }
    tc::fence_proxy_async_smem();
    tc::named_bar_sync(2, kGather);  // operand complete: the MMA warp may start

    if (warp == tcp::kMmaWarp) {
        if (lane == 0) P::mma(s, ntiles, kslabs, p.err);
        __syncwarp();
    } else {
        const int et = threadIdx.x;
        const int row = et / P::TPR, gi = et % P::TPR;
        const int grow = m0 + row;
        const bool row_live = grow < p.R;
        // confidences of this CTA's share of the M-tile's rows (local rows cv,
        // cv + nparts, ...) while the first tile is in flight; the staging tile
        // is still free and holds the reduction
        for (int i = cv; i < P::MV && m0 + i < p.R; i += p.nparts) confidence_row(p, m0 + i, et, s.staging);

        const PhiloxKey key = philox_key(p.seed);
        const uint32_t c3 = philox_ctr3(p.cycle, 0);
        RowState st;
        row_init(st);
        P::epilogue(s, t_begin, ntiles, p.err, [&](int t, int n0) {
            const unsigned char *sU = P::u_tile(s, t);
            const bool full_tile = n0 + P::BN <= p.V;
#pragma unroll
            for (int j = 0; j < P::GPT; ++j) {
                if (!row_live) break;
                const int col = 4 * (gi + P::TPR * j);
                const float4 acc = *reinterpret_cast<const float4 *>(s.staging + row * P::kPitch + col);
                const uint2 uu = P::u_quad(sU, row, col);
                float z[4] = {acc.x + tcp::bf16_lo(uu.x), acc.y + tcp::bf16_hi(uu.x), acc.z + tcp::bf16_lo(uu.y),
                              acc.w + tcp::bf16_hi(uu.y)};
                const int v0 = n0 + col;
                const uint4 words =
                    philox4x32_10(make_uint4((uint32_t)(v0 >> 2), (uint32_t)p.k, (uint32_t)grow, c3), key);
                if (full_tile)
                    row_feed4<true>(st, z, v0, p.V, words);
                else
                    row_feed4<false>(st, z, v0, p.V, words);
            }
            // the row's best score so far filters all TPR threads of the row
            float thr = st.thr;
#pragma unroll
            for (int off = P::TPR / 2; off > 0; off >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, off));
            row_raise_thr(st, thr);
        });
        // merge the TPR threads of each row (consecutive lanes)
#pragma unroll
        for (int off = P::TPR / 2; off > 0; off >>= 1) {
            const float m = __shfl_xor_sync(0xffffffffu, st.m, off);
            const float S = __shfl_xor_sync(0xffffffffu, st.S, off);
            const float bb = __shfl_xor_sync(0xffffffffu, st.best, off);
            const float zb = __shfl_xor_sync(0xffffffffu, st.zbest, off);
            const int ix = __shfl_xor_sync(0xffffffffu, st.idx, off);
            row_merge(st, m, S, bb, zb, ix);
        }
        if (gi == 0 && row_live)
            p.part[(size_t)grow * p.nparts + cv] = make_partial(st.m, st.S, st.best, st.zbest, st.idx);

        // the last CTA of the M-tile to finish merges all vocabulary ranges in a
        // fixed order: lse_k, x_k and log q_k(x_k)
        __threadfence();
        tc::named_bar_sync(1, tcp::kEpiThreads);
        if (et == 0) *s.flag = atomicAdd(&p.counters[m_tile], 1) == p.nparts - 1 ? 1 : 0;
        tc::named_bar_sync(1, tcp::kEpiThreads);
        if (*s.flag) {
            __threadfence();
            RowState fin;
            row_init(fin);
            if (row_live) {
                // batches of independent 16-byte loads, merged in index order
                constexpr int kBatch = 8;
                const DraftPartial *base = p.part + (size_t)grow * p.nparts;
                for (int i0 = gi; i0 < p.nparts; i0 += P::TPR * kBatch) {
                    DraftPartial q[kBatch];
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        const int i = i0 + b * P::TPR;
                        q[b] = i < p.nparts ? load_partial_cg(base + i)
                                            : make_partial(-INFINITY, 0.f, -INFINITY, 0.f, -1);
                    }
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) row_merge(fin, q[b].m, q[b].S, q[b].best, q[b].zbest, q[b].idx);
                }
            }
#pragma unroll
            for (int off = P::TPR / 2; off > 0; off >>= 1) {
                const float m = __shfl_xor_sync(0xffffffffu, fin.m, off);
                const float S = __shfl_xor_sync(0xffffffffu, fin.S, off);
                const float bb = __shfl_xor_sync(0xffffffffu, fin.best, off);
                const float zb = __shfl_xor_sync(0xffffffffu, fin.zbest, off);
                const int ix = __shfl_xor_sync(0xffffffffu, fin.idx, off);
                row_merge(fin, m, S, bb, zb, ix);
            }
            if (gi == 0 && row_live) {
                const size_t o = (size_t)grow * p.gamma + (p.k - 1);
                const float lse = fin.m + logf(fin.S);
                int idx = fin.idx;
                if (idx < 0 || !isfinite(lse)) {
                    set_err(p.err, DSPARK_ERR_NONFINITE);
                    idx = 0;
                }
                p.x[o] = idx;
                p.lse[o] = lse;
                p.logq[o] = fin.zbest - lse;
            }
            if (et == 0) p.counters[m_tile] = 0;
        }
    }
    P::teardown(s);
}

// pipeline configurations
// Pipe<rows, vocabulary tile, W_2^T ring, U ring, operand split>
using DraftM64 = tcp::Pipe<64, 128, 2, 2, 1>;   // Markov, R <= 64 per M-tile
using DraftM128 = tcp::Pipe<128, 64, 2, 2, 1>;  // Markov, 128 rows per M-tile
using DraftRnn = tcp::Pipe<64, 64, 3, 3, 2>;    // RNN (fp32 operand split hi/lo)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class P>
cudaError_t launch_cfg(const DraftStep &p, int nparts, int n_mtiles, cudaStream_t s) {
    CUtensorMap tmB, tmU;
    if (!encode_w2t_map(&tmB, p.W2t, p.V, p.r, P::BN)) return cudaErrorInvalidValue;
    if (!encode_u_map(&tmU, p.U, p.R, p.gamma, p.V, P::MV)) return cudaErrorInvalidValue;
    TcParams tp;
    tp.R = p.R; tp.V = p.V; tp.r = p.r; tp.d = p.d; tp.gamma = p.gamma; tp.k = p.k;
    tp.h = static_cast<const __nv_bfloat16 *>(p.h); tp.w = p.w; tp.sts_T = p.sts_T;
    tp.counters = p.counters;
    tp.x = p.x_out; tp.logq = p.logq; tp.lse = p.lse; tp.c = p.c;
    tp.W1 = static_cast<const __nv_bfloat16 *>(p.W1);
    tp.x_prev = p.x_prev; tp.x_stride = p.x_stride;
    tp.A_op = p.A_op; tp.a_stride = p.a_stride;
    tp.seed = p.seed; tp.cycle = p.cycle;
    tp.part = p.part; tp.nparts = nparts;
    tp.n_mtiles = n_mtiles;
    tp.n_vtiles = (p.V + P::BN - 1) / P::BN;
    tp.err = p.err;
    auto kern = draft_step_tc<P>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kBytes);
    if (e != cudaSuccess) return e;
    kern<<<n_mtiles * nparts, tcp::kThreads, P::kBytes, s>>>(tmB, tmU, tp);
    return cudaGetLastError();
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
