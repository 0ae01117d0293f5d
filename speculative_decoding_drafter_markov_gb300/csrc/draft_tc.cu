// draft_tc.cu -- the draft step on the 5th-generation tensor cores.
//
// DSpark digest eq. (5): B_k = W_1[x_{k-1}] W_2, contracted on tcgen05 into a
// TMEM accumulator and consumed in place by the eq. (4) epilogue (U_k add,
// online max / sum-exp, Philox Gumbel race).  No logit reaches global memory.
//
// Persistent CTAs, one per SM: CTA (m, c) owns requests [m MV, (m+1) MV) and a
// contiguous range of BN-wide vocabulary tiles.  Warp roles (576 threads):
//   warps 0..15  epilogue.  Warps whose TMEM quadrant holds live rows copy the
//                accumulator tile to a padded fp32 staging tile; then all 512
//                threads each take one request row and 4 groups of 4 columns
//                (so every SM sub-partition works even when only 64 rows live).
//   warp 16      TMA producer: per tile, the W_2^T slabs (K-major, 128-byte
//                swizzle) and the U_k tile, into a STAGES-deep ring.
//   warp 17      TMEM allocator and MMA issuer: r/16 MMAs of 128 x BN x 16
//                per tile into one of two TMEM accumulators.
// The bias operand E = W_1[x_{k-1}] is gathered once per launch into shared
// memory in the MMA's swizzled K-major layout.  For MV = 64 live rows the
// M = 128 MMA reads rows 64..127 of each K-slab from the next slab (garbage
// rows whose results are never read).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dspark {

namespace {

constexpr int kEpiThreads = 512;
constexpr int kTcThreads = kEpiThreads + 64;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;

template <int MV, int BN, int STAGES>
struct Layout {
    static constexpr int kSlabA = MV * 128;            // one 64-wide K slab of E
    static constexpr int kABytes = 4 * kSlabA;         // r <= 256
    static constexpr int kSlabB = BN * 128;            // one 64-wide K slab of W_2^T
    static constexpr int kBBytes = 4 * kSlabB;
    static constexpr int kUBox = MV * 128;             // 64 columns of U_k
    static constexpr int kUBytes = (BN / 64) * kUBox;
    static constexpr int kStageBytes = kBBytes + kUBytes;
    static constexpr int kPitch = BN + 4;              // staging row, floats
    static constexpr int kStagingBytes = MV * kPitch * 4;
    static constexpr int kOffStage = kABytes;
    static constexpr int kOffStaging = kOffStage + STAGES * kStageBytes;
    static constexpr int kOffBar = kOffStaging + kStagingBytes;
    static constexpr int kNumBars = 2 * STAGES + 4;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kBytes = kOffMisc + 16 + 1024;  // + alignment slack
    static constexpr int kTmemCols = 2 * BN;
    static_assert(kBytes <= 232448, "shared memory budget");
    static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
};

struct TcParams {
    int R, V, r, gamma, k;
    const __nv_bfloat16 *W1;
    const int32_t *x_prev;
    int x_stride;
    uint64_t seed, cycle;
    DraftPartial *part;
    int nparts;     // vocabulary ranges (CTAs per M-tile)
    int n_mtiles;
    int n_vtiles;
    int32_t *err;
};

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

template <int MV, int BN, int STAGES>
__global__ void __launch_bounds__(kTcThreads, 1)
    draft_step_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmU,
                  const TcParams p) {
    using L = Layout<MV, BN, STAGES>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *sA = smem;
    float *staging = reinterpret_cast<float *>(smem + L::kOffStaging);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *full = bars;                 // TMA landed (B + U of a stage)
    uint64_t *empty = bars + STAGES;       // stage free: MMA commit + epilogue
    uint64_t *tfull = bars + 2 * STAGES;   // accumulator b ready
    uint64_t *tempty = tfull + 2;          // accumulator b drained
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
    volatile int *epi_go = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.n_mtiles, cv = blockIdx.x / p.n_mtiles;
    const int m0 = m_tile * MV;
    const int t_begin = (int)((long long)cv * p.n_vtiles / p.nparts);
    const int t_end = (int)((long long)(cv + 1) * p.n_vtiles / p.nparts);
    const int ntiles = t_end - t_begin;
    const int kslabs = p.r / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 2);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 1);
        }
        *abort_flag = 0;
        *epi_go = 1;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
        tc::tc_fence_before();
    }
    if (warp == kProducerWarp && lane == 0) {
        tc::prefetch_tmap(&tmB);
        tc::prefetch_tmap(&tmU);
    }
    // E = W_1[x_{k-1}] for the rows of this M-tile, in the swizzled K-major layout
    const int chunks_per_row = p.r / 8;  // 16-byte chunks
    for (int e = threadIdx.x; e < MV * chunks_per_row; e += kTcThreads) {
        const int row = e / chunks_per_row, c = e - row * chunks_per_row;
        const int grow = m0 + row;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (grow < p.R) {
            int xp = p.x_prev[(size_t)grow * p.x_stride];
            if (xp < 0 || xp >= p.V) {
                if (c == 0) set_err(p.err, DSPARK_ERR_RANGE);
                xp = 0;
            }
            val = *reinterpret_cast<const uint4 *>(p.W1 + (size_t)xp * p.r + c * 8);
        }
        const int slab = c >> 3, cc = c & 7;
        unsigned char *dst = sA + slab * L::kSlabA + (row >> 3) * 1024 + (row & 7) * 128 +
                             ((cc ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = val;
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % STAGES;
                const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err)) break;
                unsigned char *sB = smem + L::kOffStage + s * L::kStageBytes;
                unsigned char *sU = sB + L::kBBytes;
                const int n0 = (t_begin + t) * BN;
                tc::mbar_expect_tx(&full[s], (uint32_t)(kslabs * L::kSlabB + L::kUBytes));
                for (int j = 0; j < kslabs; ++j) tc::tma_load_2d(sB + j * L::kSlabB, &tmB, &full[s], j * 64, n0);
                for (int h = 0; h < BN / 64; ++h)
                    tc::tma_load_3d(sU + h * L::kUBox, &tmU, &full[s], n0 + h * 64, p.k - 1, m0);
                ++issued;
            }
            // never leave with copies in flight
            for (int t = issued - STAGES < 0 ? 0 : issued - STAGES; t < issued; ++t)
                tc::mbar_wait(&full[t % STAGES], (uint32_t)(t / STAGES) & 1u, abort_flag, p.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
            const uint32_t a_base = tc::smem_u32(sA);
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % STAGES, b = t & 1;
                const uint32_t ph = (uint32_t)(t / STAGES) & 1u, bph = (uint32_t)(t >> 1) & 1u;
                if (!tc::mbar_wait(&full[s], ph, abort_flag, p.err)) break;
                if (!tc::mbar_wait(&tempty[b], bph ^ 1u, abort_flag, p.err)) break;
                tc::tc_fence_after();
                const uint32_t b_base = tc::smem_u32(smem + L::kOffStage + s * L::kStageBytes);
                const uint32_t d = tmem_base + (uint32_t)(b * BN);
                for (int kk = 0; kk < p.r / 16; ++kk) {
                    const int slab = kk >> 2, off = (kk & 3) * 32;
                    tc::umma_bf16(d, tc::smem_desc_k128(a_base + slab * L::kSlabA + off),
                                  tc::smem_desc_k128(b_base + slab * L::kSlabB + off), idesc,
                                  kk > 0 ? 1u : 0u);
                }
                tc::umma_commit(&empty[s]);
                tc::umma_commit(&tfull[b]);
                ++issued;
            }
            if (issued > 0) {  // the last MMAs must finish before TMEM is freed
                const int t = issued - 1;
                tc::mbar_wait(&tfull[t & 1], (uint32_t)(t >> 1) & 1u, abort_flag, p.err);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int TPR = kEpiThreads / MV;  // threads per request row
        constexpr int GPR = BN / 4;            // 4-column groups per row and tile
        constexpr int GPT = GPR / TPR;         // groups per thread and tile
        static_assert(GPT * TPR == GPR, "epilogue mapping");
        const int et = threadIdx.x;
        const int row = et / TPR, gi = et % TPR;
        const int grow = m0 + row;
        const bool row_live = grow < p.R;
        const int q = warp & 3, wj = warp >> 2;
        const bool loader = q * 32 < MV;
        const PhiloxKey key = philox_key(p.seed);
        const uint32_t c3 = philox_ctr3(p.cycle, 0);
        RowState st;
        row_init(st);
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % STAGES, b = t & 1;
            const uint32_t ph = (uint32_t)(t / STAGES) & 1u, bph = (uint32_t)(t >> 1) & 1u;
            if (et == 0) {
                bool ok = tc::mbar_wait(&tfull[b], bph, abort_flag, p.err);
                ok = ok && tc::mbar_wait(&full[s], ph, abort_flag, p.err);
                *epi_go = ok ? 1 : 0;
            }
            tc::named_bar_sync(1, kEpiThreads);
            if (!*epi_go) break;
            tc::tc_fence_after();
            if (loader) {
                for (int ch = wj; ch < BN / 16; ch += 4) {
                    uint32_t v[16];
                    tc::tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + ch * 16), v);
                    tc::tmem_wait_ld();
                    float4 *dst = reinterpret_cast<float4 *>(staging + (q * 32 + lane) * L::kPitch + ch * 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
            tc::tc_fence_before();
            tc::named_bar_sync(1, kEpiThreads);
            if (et == 0) tc::mbar_arrive(&tempty[b]);

            const unsigned char *sU = smem + L::kOffStage + s * L::kStageBytes + L::kBBytes;
            const int n0 = (t_begin + t) * BN;
            if (row_live) {
#pragma unroll
                for (int j = 0; j < GPT; ++j) {
                    const int col = 4 * (gi + TPR * j);
                    const float4 acc = *reinterpret_cast<const float4 *>(staging + row * L::kPitch + col);
                    const int h = col >> 6, cc = col & 63;
                    const uint2 uu = *reinterpret_cast<const uint2 *>(
                        sU + h * L::kUBox + row * 128 + ((((cc >> 3) ^ (row & 7))) << 4) + ((cc & 7) << 1));
                    float z[4] = {acc.x + bf16_lo(uu.x), acc.y + bf16_hi(uu.x), acc.z + bf16_lo(uu.y),
                                  acc.w + bf16_hi(uu.y)};
                    const int v0 = n0 + col;
                    const uint4 words = philox4x32_10(
                        make_uint4((uint32_t)(v0 >> 2), (uint32_t)p.k, (uint32_t)grow, c3), key);
                    row_feed4(st, z, v0, p.V, words);
                }
            }
            tc::named_bar_sync(1, kEpiThreads);
            if (et == 0) tc::mbar_arrive(&empty[s]);
        }
        // merge the TPR threads of each row (consecutive lanes)
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) {
            const float m = __shfl_xor_sync(0xffffffffu, st.m, off);
            const float S = __shfl_xor_sync(0xffffffffu, st.S, off);
            const float bb = __shfl_xor_sync(0xffffffffu, st.best, off);
            const float zb = __shfl_xor_sync(0xffffffffu, st.zbest, off);
            const int ix = __shfl_xor_sync(0xffffffffu, st.idx, off);
            row_merge(st, m, S, bb, zb, ix);
        }
        if (gi == 0 && row_live)
            p.part[(size_t)grow * p.nparts + cv] = DraftPartial{st.m, st.S, st.best, st.zbest, st.idx};
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int MV, int BN, int STAGES>
cudaError_t launch_tc(const DraftStep &p, int nparts, int n_mtiles, cudaStream_t s) {
    using L = Layout<MV, BN, STAGES>;
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmB, tmU;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.V};
        const cuuint64_t strides[1] = {(cuuint64_t)p.r * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)BN};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.W2t), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.gamma, (cuuint64_t)p.R};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 2, (cuuint64_t)p.gamma * p.V * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)MV};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.U), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    TcParams tp;
    tp.R = p.R; tp.V = p.V; tp.r = p.r; tp.gamma = p.gamma; tp.k = p.k;
    tp.W1 = static_cast<const __nv_bfloat16 *>(p.W1);
    tp.x_prev = p.x_prev; tp.x_stride = p.x_stride;
    tp.seed = p.seed; tp.cycle = p.cycle;
    tp.part = p.part; tp.nparts = nparts;
    tp.n_mtiles = n_mtiles;
    tp.n_vtiles = (p.V + BN - 1) / BN;
    tp.err = p.err;
    auto kern = draft_step_tc<MV, BN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    kern<<<n_mtiles * nparts, kTcThreads, L::kBytes, s>>>(tmB, tmU, tp);
    return cudaGetLastError();
}

}  // namespace

bool draft_step_tc_supported(const DraftStep &p) {
    static const int force = [] {
        const char *v = getenv("DSPARK_DRAFT_KERNEL");
        if (!v) return 0;
        if (v[0] == 's') return -1;  // "simt": CUDA-core path only
        return 0;
    }();
    if (force < 0) return false;
    return p.dtype == DSPARK_BF16 && p.A_op == nullptr && p.r % 64 == 0 && p.r >= 64 && p.r <= 256 &&
           p.V % 8 == 0 && aligned16(p.U) && aligned16(p.W1) && aligned16(p.W2t) && encode_fn() != nullptr &&
           sm_count() > 0;
}

void draft_step_tc_shape(int R, int V, int *nparts, int *n_mtiles) {
    const int MV = R <= 64 ? 64 : 128;
    const int BN = MV == 64 ? 128 : 64;
    const int mt = (R + MV - 1) / MV;
    const int sms = sm_count();
    int g = sms / mt;
    if (g < 1) g = 1;
    const int nv = (V + BN - 1) / BN;
    if (g > nv) g = nv;
    *nparts = g;
    *n_mtiles = mt;
}

cudaError_t launch_draft_step_tc(const DraftStep &p, cudaStream_t s) {
    int nparts = 0, mt = 0;
    draft_step_tc_shape(p.R, p.V, &nparts, &mt);
    if (nparts != p.nparts) return cudaErrorInvalidValue;
    if (p.R <= 64) return launch_tc<64, 128, 2>(p, nparts, mt, s);
    return launch_tc<128, 64, 2>(p, nparts, mt, s);
}

}  // namespace dspark
