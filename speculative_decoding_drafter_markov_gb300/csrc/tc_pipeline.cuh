// tc_pipeline.cuh -- the contraction pipeline shared by the tensor-core kernels.
//
// D[MV x BN tile] = A[MV rows, r] . W_2^T[BN vocabulary rows, r]^T on tcgen05,
// where A (the bias operand of each request: W_1[x] or the RNN vector A_k) is
// resident in shared memory and W_2^T streams through a STAGES-deep TMA ring.
// One CTA owns one M-tile of MV requests and a contiguous range of BN-wide
// vocabulary tiles; warp roles (576 threads):
//   warps 0..15  epilogue: warps whose TMEM quadrant holds live rows copy each
//                accumulator to a padded fp32 staging tile, then all 512 threads
//                run the caller's per-tile functor, one request row and GPT
//                groups of 4 columns per thread;
//   warp 16      TMA producer (W_2^T slabs and, optionally, a U tile per stage);
//   warp 17      TMEM allocator and MMA issuer (double-buffered accumulators).
// KSPLIT = 2 keeps an fp32 operand exact to ~2^-16 relative: A = A_hi + A_lo in
// bf16, two MMAs per K-step against the same W_2^T slab.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc.cuh"

namespace dspark {
namespace tcp {

constexpr int kEpiThreads = 512;
constexpr int kThreads = kEpiThreads + 64;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;

template <int MV_, int BN_, int SB_, int SU_, int KSPLIT_>
struct Pipe {
    static constexpr int MV = MV_, BN = BN_, SB = SB_, SU = SU_, KSPLIT = KSPLIT_;
    static constexpr bool WITH_U = SU > 0;
    static constexpr int kSlabA = MV * 128;            // one 64-wide K slab of A (bf16)
    static constexpr int kABytes = 4 * KSPLIT * kSlabA; // r <= 256
    static constexpr int kSlabB = BN * 128;            // one 64-wide K slab of W_2^T
    static constexpr int kBBytes = 4 * kSlabB;
    static constexpr int kUBox = MV * 128;             // 64 columns of U
    static constexpr int kUBytes = (BN / 64) * kUBox;
    static constexpr int kPitch = BN + 4;              // staging row (floats)
    static constexpr int kStagingBytes = MV * kPitch * 4;
    // with MV = 64 the M = 128 MMA reads 8 KB past the last A slab: B stage 0
    static constexpr int kOffB = kABytes;
    static constexpr int kOffU = kOffB + SB * kBBytes;
    static constexpr int kOffStaging = kOffU + SU * kUBytes;
    static constexpr int kOffBar = kOffStaging + kStagingBytes;
    static constexpr int kNumBars = 2 * SB + 2 * SU + 4;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kBytes = kOffMisc + 32 + 1024;  // + alignment slack
    static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int TPR = kEpiThreads / MV;  // epilogue threads per request row
    static constexpr int GPR = BN / 4;            // 4-column groups per row and tile
    static constexpr int GPT = GPR / TPR;         // groups per thread and tile
    static_assert(kBytes <= 232448, "shared memory budget");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns must be a power of two");
    static_assert(GPT * TPR == GPR, "epilogue mapping");
    static_assert(MV == 64 || MV == 128, "M-tile rows");

    struct State {
        unsigned char *smem, *sA;
        float *staging;
        uint64_t *fullB, *emptyB, *fullU, *emptyU, *tfull, *tempty;
        uint32_t *tmem_slot;
        volatile int *abort_flag, *epi_go, *flag;
        uint32_t tmem_base;
    };

    __device__ static State carve(unsigned char *raw) {
        State s;
        s.smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                                   ~static_cast<uintptr_t>(1023));
        s.sA = s.smem;
        s.staging = reinterpret_cast<float *>(s.smem + kOffStaging);
        uint64_t *bars = reinterpret_cast<uint64_t *>(s.smem + kOffBar);
        s.fullB = bars;
        s.emptyB = bars + SB;
        s.fullU = bars + 2 * SB;
        s.emptyU = bars + 2 * SB + SU;
        s.tfull = bars + 2 * SB + 2 * SU;
        s.tempty = s.tfull + 2;
        s.tmem_slot = reinterpret_cast<uint32_t *>(s.smem + kOffMisc);
        s.abort_flag = reinterpret_cast<volatile int *>(s.smem + kOffMisc + 4);
        s.epi_go = reinterpret_cast<volatile int *>(s.smem + kOffMisc + 8);  // two flags
        s.flag = reinterpret_cast<volatile int *>(s.smem + kOffMisc + 16);
        s.tmem_base = 0;
        return s;
    }

    // all threads: barrier init (thread 0) and TMEM allocation (MMA warp)
    __device__ static void init(State &s) {
        const int warp = threadIdx.x >> 5;
        if (threadIdx.x == 0) {
            for (int i = 0; i < SB; ++i) {
                tc::mbar_init(&s.fullB[i], 1);
                tc::mbar_init(&s.emptyB[i], 1);  // MMA commit
            }
            for (int i = 0; i < SU; ++i) {
                tc::mbar_init(&s.fullU[i], 1);
                tc::mbar_init(&s.emptyU[i], 1);  // epilogue
            }
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&s.tfull[b], 1);
                tc::mbar_init(&s.tempty[b], 1);
            }
            *s.abort_flag = 0;
            s.epi_go[0] = 0;
            s.epi_go[1] = 0;
            *s.flag = 0;
            tc::fence_mbar_init();
        }
        if (warp == kMmaWarp) {
            tc::tmem_alloc(s.tmem_slot, kTmemCols);
            tc::tmem_relinquish();
            tc::tc_fence_before();
        }
    }

    // after the CTA barrier that follows init
    __device__ static void ready(State &s) {
        tc::tc_fence_after();
        s.tmem_base = *s.tmem_slot;
    }

    // 16-byte chunk c (8 bf16 along K) of row `row` of split part `part` of A
    __device__ static unsigned char *a_chunk(const State &s, int row, int c, int part) {
        const int slab = (c >> 3) + 4 * part, cc = c & 7;
        return s.sA + slab * kSlabA + (row >> 3) * 1024 + (row & 7) * 128 + ((cc ^ (row & 7)) << 4);
    }

    // the U tile of tile t
    __device__ static const unsigned char *u_tile(const State &s, int t) {
        return s.smem + kOffU + (SU > 0 ? t % SU : 0) * kUBytes;
    }

    // U element (row, col) of a staged U tile (64-column boxes, 128-byte swizzle)
    __device__ static uint2 u_quad(const unsigned char *sU, int row, int col) {
        const int h = col >> 6, cc = col & 63;
        return *reinterpret_cast<const uint2 *>(sU + h * kUBox + row * 128 +
                                                ((((cc >> 3) ^ (row & 7))) << 4) + ((cc & 7) << 1));
    }

    // producer warp: lane 0 streams the W_2^T ring (freed by the MMA commits),
    // lane 1 the U ring (freed by the epilogue), so W_2^T runs ahead of the
    // epilogue by the whole B ring
    __device__ static void producer(State &s, const CUtensorMap *tmB, const CUtensorMap *tmU, int t_begin,
                                    int ntiles, int kslabs, int u_k, int m0, int32_t *err) {
        const int lane = threadIdx.x & 31;
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int st = t % SB;
                if (!tc::mbar_wait(&s.emptyB[st], ((uint32_t)(t / SB) & 1u) ^ 1u, s.abort_flag, err)) break;
                unsigned char *sB = s.smem + kOffB + st * kBBytes;
                const int n0 = (t_begin + t) * BN;
                tc::mbar_expect_tx(&s.fullB[st], (uint32_t)(kslabs * kSlabB));
                for (int j = 0; j < kslabs; ++j) tc::tma_load_2d(sB + j * kSlabB, tmB, &s.fullB[st], j * 64, n0);
                ++issued;
            }
            // never leave with copies in flight
            for (int t = issued - SB < 0 ? 0 : issued - SB; t < issued; ++t)
                tc::mbar_wait(&s.fullB[t % SB], (uint32_t)(t / SB) & 1u, s.abort_flag, err);
        } else if (lane == 1 && SU > 0) {
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int st = t % (SU > 0 ? SU : 1);
                if (!tc::mbar_wait(&s.emptyU[st], ((uint32_t)(t / SU) & 1u) ^ 1u, s.abort_flag, err)) break;
                unsigned char *sU = s.smem + kOffU + st * kUBytes;
                const int n0 = (t_begin + t) * BN;
                tc::mbar_expect_tx(&s.fullU[st], (uint32_t)kUBytes);
                for (int h = 0; h < BN / 64; ++h)
                    tc::tma_load_3d(sU + h * kUBox, tmU, &s.fullU[st], n0 + h * 64, u_k, m0);
                ++issued;
            }
            for (int t = issued - SU < 0 ? 0 : issued - SU; t < issued; ++t)
                tc::mbar_wait(&s.fullU[t % SU], (uint32_t)(t / SU) & 1u, s.abort_flag, err);
        }
    }

    // warp 17, lane 0
    __device__ static void mma(State &s, int ntiles, int kslabs, int32_t *err) {
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
        const uint32_t a_base = tc::smem_u32(s.sA);
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % SB, b = t & 1;
            if (!tc::mbar_wait(&s.fullB[st], (uint32_t)(t / SB) & 1u, s.abort_flag, err)) break;
            if (!tc::mbar_wait(&s.tempty[b], ((uint32_t)(t >> 1) & 1u) ^ 1u, s.abort_flag, err)) break;
            tc::tc_fence_after();
            const uint32_t b_base = tc::smem_u32(s.smem + kOffB + st * kBBytes);
            const uint32_t d = s.tmem_base + (uint32_t)(b * BN);
            for (int kk = 0; kk < kslabs * 4; ++kk) {
                const int slab = kk >> 2, off = (kk & 3) * 32;
                const uint64_t bd = tc::smem_desc_k128(b_base + slab * kSlabB + off);
#pragma unroll
                for (int part = 0; part < KSPLIT; ++part)
                    tc::umma_bf16(d, tc::smem_desc_k128(a_base + (slab + 4 * part) * kSlabA + off), bd, idesc,
                                  (kk > 0 || part > 0) ? 1u : 0u);
            }
            tc::umma_commit(&s.emptyB[st]);
            tc::umma_commit(&s.tfull[b]);
            ++issued;
        }
        if (issued > 0) {  // the last MMAs must finish before TMEM is freed
            const int t = issued - 1;
            tc::mbar_wait(&s.tfull[t & 1], (uint32_t)(t >> 1) & 1u, s.abort_flag, err);
        }
    }

    // thread 0 of the epilogue: wait until tile t's accumulator and U tile are ready
    __device__ static int wait_tile(State &s, int t, int32_t *err) {
        bool ok = tc::mbar_wait(&s.tfull[t & 1], (uint32_t)(t >> 1) & 1u, s.abort_flag, err);
        if (SU > 0) ok = ok && tc::mbar_wait(&s.fullU[t % SU], (uint32_t)(t / SU) & 1u, s.abort_flag, err);
        return ok ? 1 : 0;
    }

    // warps 0..15: per tile, stage the accumulator, then f(t, n0) on every thread.
    // Two epilogue barriers per tile; thread 0 waits for tile t+1 before the
    // second one and publishes the outcome in a double-buffered flag, so all
    // threads leave the loop together on a timeout.
    template <class F>
    __device__ static void epilogue(State &s, int t_begin, int ntiles, int32_t *err, F &&f) {
        const int et = threadIdx.x, warp = et >> 5, lane = et & 31;
        const int q = warp & 3, wj = warp >> 2;
        const bool loader = q * 32 < MV;
        if (et == 0) s.epi_go[0] = ntiles > 0 ? wait_tile(s, 0, err) : 0;
        tc::named_bar_sync(1, kEpiThreads);
        for (int t = 0; t < ntiles; ++t) {
            if (!s.epi_go[t & 1]) break;
            const int b = t & 1;
            tc::tc_fence_after();
            if (loader) {
                for (int ch = wj; ch < BN / 16; ch += 4) {
                    uint32_t v[16];
                    tc::tmem_ld16(s.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + ch * 16), v);
                    tc::tmem_wait_ld();
                    float4 *dst = reinterpret_cast<float4 *>(s.staging + (q * 32 + lane) * kPitch + ch * 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
            tc::tc_fence_before();
            tc::named_bar_sync(1, kEpiThreads);
            if (et == 0) tc::mbar_arrive(&s.tempty[b]);
            f(t, (t_begin + t) * BN);
            if (et == 0) s.epi_go[(t + 1) & 1] = t + 1 < ntiles ? wait_tile(s, t + 1, err) : 0;
            tc::named_bar_sync(1, kEpiThreads);
            if (SU > 0 && et == 0) tc::mbar_arrive(&s.emptyU[t % SU]);
        }
    }

    // all threads, at the very end
    __device__ static void teardown(State &s) {
        __syncthreads();
        if ((threadIdx.x >> 5) == kMmaWarp) {
            tc::tc_fence_after();
            tc::tmem_dealloc(s.tmem_base, kTmemCols);
        }
    }
};

// vocabulary tile range of CTA cv out of nparts
__device__ __forceinline__ void tile_range(int cv, int nparts, int n_vtiles, int &t_begin, int &ntiles) {
    t_begin = (int)((long long)cv * n_vtiles / nparts);
    ntiles = (int)((long long)(cv + 1) * n_vtiles / nparts) - t_begin;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// split 8 fp32 values into bf16 hi and lo parts (x = hi + lo + O(2^-16 |x|))
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * i]), h1 = __float2bfloat16_rn(x[2 * i + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(x[2 * i] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(x[2 * i + 1] - __bfloat162float(h1));
        h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

}  // namespace tcp
}  // namespace dspark
