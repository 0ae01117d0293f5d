// gemm_tc.cu -- the RNN head's hidden-state projection on the 5th-generation
// tensor cores.
//
// DSpark digest eq. (6): z_k = [s_{k-1}; W_1[x_{k-1}]; h_k] enters one linear
// projection W = [W_g; W_c; W_o] of shape [3r, 2r + d].  The h_k columns of W
// do not depend on the recurrence, so their part of every gate pre-activation
// is formed for all (request, k) rows up front:
//     Hpre[M, 3r] = h[M, d] . W[:, 2r:]^T,   M = R gamma,
// bf16 operands, fp32 accumulation and output.  One CTA computes one 128 x 128
// output tile: warp 0 streams 64-wide K slabs of both operands by TMA (128-byte
// swizzle) through a ring of kStages slots, warp 1 owns the TMEM accumulator
// and issues tcgen05.mma (M = 128, N = 128, K = 16) per slab, committing each
// slab's MMAs to the slot's "empty" barrier; warps 2..5 read the accumulator
// (each its own TMEM lane quadrant) and store fp32 rows.  Out-of-range rows and
// K columns of a ragged tile load as zeros and their outputs are not stored.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128, kBN = 128, kStages = 4;
constexpr int kSlabA = kBM * 128;  // 128 rows x 64 bf16
constexpr int kSlabB = kBN * 128;
constexpr int kGemmThreads = 192;
constexpr int kOffBar = kStages * (kSlabA + kSlabB);
constexpr int kNumBars = 2 * kStages + 1;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kGemmSmem = kOffMisc + 16 + 1024;  // + alignment slack

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        float *C, int M, int N, int K, int ldc, int32_t *err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
    const int kslabs = (K + 63) / 64;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(tfull, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kBN);
        tc::tmem_relinquish();
        tc::tc_fence_before();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tmap(&tmA);
            tc::prefetch_tmap(&tmB);
            int issued = 0, slot = 0;
            uint32_t phase = 0;
            for (int j = 0; j < kslabs; ++j) {
                if (!tc::mbar_wait(&empty[slot], phase ^ 1u, abort_flag, err)) break;
                unsigned char *dst = smem + slot * (kSlabA + kSlabB);
                tc::mbar_expect_tx(&full[slot], (uint32_t)(kSlabA + kSlabB));
                tc::tma_load_2d(dst, &tmA, &full[slot], j * 64, m0);
                tc::tma_load_2d(dst + kSlabA, &tmB, &full[slot], j * 64, n0);
                ++issued;
                if (++slot == kStages) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            for (int g = issued - kStages < 0 ? 0 : issued - kStages; g < issued; ++g)  // nothing left in flight
                tc::mbar_wait_drain(&full[g % kStages], (uint32_t)(g / kStages) & 1u, err);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
            int slot = 0, issued = 0;
            uint32_t phase = 0;
            for (int j = 0; j < kslabs; ++j) {
                if (!tc::mbar_wait(&full[slot], phase, abort_flag, err)) break;
                tc::tc_fence_after();
                const uint32_t sa = tc::smem_u32(smem + slot * (kSlabA + kSlabB));
                const uint64_t ad = tc::smem_desc_k128(sa), bd = tc::smem_desc_k128(sa + kSlabA);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::umma_bf16(tmem, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc,
                                  (j > 0 || kk > 0) ? 1u : 0u);
                tc::umma_commit(&empty[slot]);
                ++issued;
                if (++slot == kStages) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            // the accumulator is complete (or, after an abort, the issued MMAs are
            // done) once this commit arrives; the epilogue and the TMEM release wait on it
            tc::umma_commit(tfull);
            if (issued > 0) tc::mbar_wait_drain(tfull, 0u, err);
        }
        __syncwarp();
    } else {
        // warps 2..5: TMEM lane quadrant (warp % 4) holds rows 32 q .. 32 q + 31
        const int q = warp & 3;
        int ok = 1;
        if (lane == 0) ok = tc::mbar_wait(tfull, 0u, abort_flag, err) && !*abort_flag ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
            tc::tc_fence_after();
            const int row = m0 + 32 * q + lane;
            float *crow = C + (size_t)row * ldc;
            const bool vec = (ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
#pragma unroll 1
            for (int c = 0; c < kBN / 16; ++c) {
                uint32_t acc[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * c), acc);
                tc::tmem_wait_ld();
                const int col = n0 + 16 * c;
                if (row >= M || col >= N) continue;
                if (vec && col + 16 <= N) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<float4 *>(crow + col + 4 * i) =
                            make_float4(__uint_as_float(acc[4 * i]), __uint_as_float(acc[4 * i + 1]),
                                        __uint_as_float(acc[4 * i + 2]), __uint_as_float(acc[4 * i + 3]));
                } else {
                    for (int i = 0; i < 16 && col + i < N; ++i) crow[col + i] = __uint_as_float(acc[i]);
                }
            }
        }
        tc::tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kBN);
    }
}

}  // namespace

bool hproj_tc_supported(int M, int d, int r, int dtype, const void *h, const void *W, const float *Hpre) {
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return tc_kernels_enabled() && tc_available() && dtype == DSPARK_BF16 && M > 0 && d > 0 && r > 0 &&
           d % 8 == 0 && r % 4 == 0 && (2 * r + d) % 8 == 0 && al16(h) && al16(W) && al16(Hpre);
}

cudaError_t launch_hproj_tc(int M, int d, int r, const void *h, const void *W, float *Hpre, int32_t *err,
                            cudaStream_t s) {
    const int N = 3 * r, ldw = 2 * r + d;
    CUtensorMap tmA, tmB;
    // h [M, d] and W[:, 2r:] ([3r, d] rows of stride 2r + d), both K-major
    if (!encode_kmajor_map(&tmA, h, M, d, d, kBM)) return cudaErrorInvalidValue;
    if (!encode_kmajor_map(&tmB, static_cast<const __nv_bfloat16 *>(W) + 2 * r, N, d, ldw, kBN))
        return cudaErrorInvalidValue;
    auto kern = gemm_bf16_tn_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((N + kBN - 1) / kBN, (M + kBM - 1) / kBM);
    kern<<<grid, kGemmThreads, kGemmSmem, s>>>(tmA, tmB, Hpre, M, N, d, N, err);
    return cudaGetLastError();
}

}  // namespace dspark
