// tc_pipe.cuh -- the contraction pipeline shared by the tensor-core kernels.
//
// D = A . W_2^T[tile]^T on tcgen05, where A (the bias operand of each request:
// W_1[x] or the RNN vector A_k, bf16, K-major, 128-byte swizzle) is resident in
// shared memory and W_2^T streams through a ring of 64-wide K slabs.  One CTA
// owns one M-tile of MV requests and a set of BN-wide vocabulary tiles (a
// contiguous range, or tiles taken one at a time from a counter the M-tile's
// CTAs share).  Warp roles (576 threads):
//   warps 0..15  epilogue: every warp reads its own block of the accumulator
//                straight from TMEM (no staging) and runs the caller's
//                functor on it; synchronisation is per warp, through mbarriers.
//   warp 16      TMA producer of the W_2^T slab ring (each slot freed by the
//                MMA commit that consumed it).
//   warp 17      TMEM allocator and MMA issuer, NACC accumulators of BN columns.
//   warp 18      (pipelines with a U ring) TMA producer of the U ring (a slot
//                freed when all 16 epilogue warps have used its tile).  Each
//                waiting role has a warp of its own: a lane blocked in an
//                mbarrier wait would otherwise hold up a sibling lane's role.
// MV = 128: quadrant q of the accumulator holds requests 32q..32q+31 and the
// four warps of a quadrant split the BN columns.  MV = 64: A holds the 64
// requests twice (rows i and 64 + i), so quadrants 0-1 and 2-3 hold the same
// requests; quadrants 0-1 take the first BN/2 columns and 2-3 the second half,
// which keeps all 16 warps busy with only 64 requests.
// KSPLIT = 2: A = A_hi + A_lo in bf16 (an fp32 operand kept to ~2^-16 relative),
// two MMAs per K-step against the same W_2^T slab.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc.cuh"

namespace dspark {
namespace tcp {

constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kUWarp = 18;

template <int MV_, int BN_, int NS_, int SU_, int KSPLIT_>
struct Pipe {
    static constexpr int MV = MV_, BN = BN_, NS = NS_, SU = SU_, KSPLIT = KSPLIT_;
    static constexpr bool DUAL = MV == 64;
    static constexpr bool WITH_U = SU > 0;
    static constexpr int kThreads = kEpiThreads + (WITH_U ? 96 : 64);  // epilogue, producer(s), MMA
    static constexpr int kArows = 128;                  // MMA rows (A duplicated when DUAL)
    static constexpr int kSlabA = kArows * 128;         // one 64-wide K slab of A
    static constexpr int kABytes = 4 * KSPLIT * kSlabA; // r <= 256
    static constexpr int kSlabB = BN * 128;             // one 64-wide K slab of W_2^T
    static constexpr int kUBox = MV * 128;              // 64 vocabulary columns of U
    // The U tile travels in UH parts of at most 128 columns, one ring slot each
    // (a 256-column tile would not fit two whole U tiles next to the operand and
    // the W_2^T ring); the epilogue warps of a part release its slot.
    static constexpr int UH = BN > 128 ? BN / 128 : 1;
    static constexpr int kUCols = BN / UH;               // columns of a part
    static constexpr int kUBytes = (kUCols / 64) * kUBox;  // bytes of a part (one slot)
    static constexpr int NACC = 512 / BN > 4 ? 4 : 512 / BN;  // TMEM accumulators
    static constexpr int kTmemCols = NACC * BN;
    static constexpr int CW = DUAL ? BN / 8 : BN / 4;  // accumulator columns per warp
    static constexpr int TPR = DUAL ? 8 : 4;           // epilogue threads per request
    static constexpr int kOffB = kABytes;
    static constexpr int kOffU = kOffB + NS * kSlabB;
    static constexpr int kOffBar = kOffU + SU * kUBytes;
    static constexpr int kNumBars = 2 * NS + 2 * SU + 2 * NACC + 2;
    static constexpr int kOffThr = kOffBar + 8 * kNumBars;  // per-request filter thresholds
    static constexpr int kOffTok = kOffThr + 8 * MV;        // per-request tokens / metadata
    static constexpr int kOffMisc = kOffTok + 4 * MV;
    static constexpr int kOffRed = kOffMisc + 64;           // 16-float reduction scratch
    static constexpr int kBytes = kOffRed + 64 + 1024;      // + alignment slack
    // scratch for the per-CTA merge after the tile loop: the operand region,
    // which no MMA reads once the last accumulator has been consumed
    static constexpr int kMergeBytes = kEpiThreads * 5 * 4;
    static_assert(kBytes <= 232448, "shared memory budget");
    static_assert(kMergeBytes <= kABytes, "merge scratch");
    static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
    static_assert(CW == 16 || CW == 32 || CW == 64, "TMEM load width");
    static_assert(UH == 1 || (kUCols % CW == 0 && (!DUAL || (BN / 2) % kUCols == 0)),
                  "a warp's columns lie in one U part");
    static_assert(MV == 64 || MV == 128, "M-tile rows");

    struct State {
        unsigned char *smem, *sA;
        uint64_t *fullB, *emptyB, *fullU, *emptyU, *tfull, *tempty;
        uint64_t *aready;  // operand of the next step written (multi-step launches)
        uint64_t *opbar;   // bulk copy of a prepared operand into the operand region landed
        unsigned long long *thr;  // per request: the best packed race winner the CTA knows
        int *tok;          // MV ints of per-request scratch
        uint32_t *tmem_slot;
        volatile int *abort_flag, *flag;
        float *red;  // 16 floats
        uint32_t tmem_base;
    };

    __device__ static State carve(unsigned char *raw) {
        State s;
        s.smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                                   ~static_cast<uintptr_t>(1023));
        s.sA = s.smem;
        uint64_t *bars = reinterpret_cast<uint64_t *>(s.smem + kOffBar);
        s.fullB = bars;
        s.emptyB = bars + NS;
        s.fullU = bars + 2 * NS;
        s.emptyU = bars + 2 * NS + SU;
        s.tfull = bars + 2 * NS + 2 * SU;
        s.tempty = s.tfull + NACC;
        s.aready = s.tempty + NACC;
        s.opbar = s.aready + 1;
        s.thr = reinterpret_cast<unsigned long long *>(s.smem + kOffThr);
        s.tok = reinterpret_cast<int *>(s.smem + kOffTok);
        s.tmem_slot = reinterpret_cast<uint32_t *>(s.smem + kOffMisc);
        s.abort_flag = reinterpret_cast<volatile int *>(s.smem + kOffMisc + 4);
        s.flag = reinterpret_cast<volatile int *>(s.smem + kOffMisc + 8);
        s.red = reinterpret_cast<float *>(s.smem + kOffRed);
        s.tmem_base = 0;
        return s;
    }

    // all threads: barrier init, thresholds (thread 0 / first MV threads) and TMEM allocation
    __device__ static void init(State &s) {
        const int warp = threadIdx.x >> 5;
        if (threadIdx.x == 0) {
            for (int i = 0; i < NS; ++i) {
                tc::mbar_init(&s.fullB[i], 1);
                tc::mbar_init(&s.emptyB[i], 1);  // the MMA commit that consumed the slab
            }
            for (int i = 0; i < SU; ++i) {
                tc::mbar_init(&s.fullU[i], 1);
                tc::mbar_init(&s.emptyU[i], kEpiWarps / UH);  // every epilogue warp of the part
            }
            for (int b = 0; b < NACC; ++b) {
                tc::mbar_init(&s.tfull[b], 1);
                tc::mbar_init(&s.tempty[b], kEpiWarps);
            }
            tc::mbar_init(s.aready, 1);
            tc::mbar_init(s.opbar, 1);
            *s.abort_flag = 0;
            *s.flag = 0;
            tc::fence_mbar_init();
        }
        if (threadIdx.x < MV) s.thr[threadIdx.x] = 0ull;
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

    // byte offset of 16-byte chunk c (8 bf16 along K) of MMA row `row` of split
    // part `part` in the operand region (K-major, 128-byte swizzle, 64-wide slabs)
    __host__ __device__ static constexpr int a_offset(int row, int c, int part) {
        return ((c >> 3) + 4 * part) * kSlabA + (row >> 3) * 1024 + (row & 7) * 128 + (((c & 7) ^ (row & 7)) << 4);
    }
    __device__ static unsigned char *a_chunk(const State &s, int row, int c, int part) {
        return s.sA + a_offset(row, c, part);
    }

    // write operand chunk c of request row `row` (both copies when DUAL)
    __device__ static void put_a(const State &s, int row, int c, int part, const uint4 &v) {
        *reinterpret_cast<uint4 *>(a_chunk(s, row, c, part)) = v;
        if (DUAL) *reinterpret_cast<uint4 *>(a_chunk(s, row + 64, c, part)) = v;
    }

    // eight columns col .. col + 7 (col a multiple of 8) of a U tile row
    __device__ static uint4 u_oct(const unsigned char *sU, int row, int col) {
        col &= kUCols - 1;  // within the part that holds it
        const int h = col >> 6, cc = col & 63;
        return *reinterpret_cast<const uint4 *>(sU + h * kUBox + row * 128 + (((cc >> 3) ^ (row & 7)) << 4));
    }

    // one quad of a U tile (64-column boxes, 128-byte swizzle)
    __device__ static uint2 u_quad(const unsigned char *sU, int row, int col) {
        col &= kUCols - 1;  // within the part that holds it
        const int h = col >> 6, cc = col & 63;
        return *reinterpret_cast<const uint2 *>(sU + h * kUBox + row * 128 +
                                                ((((cc >> 3) ^ (row & 7))) << 4) + ((cc & 7) << 1));
    }

    // epilogue thread geometry: request row within the M-tile and first column
    // (within the vocabulary tile) of this warp's accumulator block
    __device__ static int epi_row() {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        return DUAL ? lane + 32 * (warp & 1) : lane + 32 * (warp & 3);
    }
    __device__ static int epi_col0() {
        const int warp = threadIdx.x >> 5, q = warp & 3, j = warp >> 2;
        return DUAL ? (q >= 2 ? BN / 2 : 0) + j * CW : j * CW;
    }

    // warp 16, lane 0: the W_2^T slabs of `nsteps` consecutive draft steps over
    // the same tiles (W_2^T does not depend on the step, so the next step's
    // slabs stream in while the current one is merged).  Tile t of the CTA
    // starts at vocabulary column col0 + t * tstride.
    __device__ static void producer_w2(State &s, const CUtensorMap *tmB, int col0, int tstride, int ntiles,
                                       int kslabs, int nsteps, int32_t *err) {
        {
            const int total = nsteps * ntiles * kslabs;
            int issued = 0, slot = 0, t = 0, j = 0;  // ring slot, tile and K slab of load `issued`
            uint32_t phase = 0;
            for (int g = 0; g < total; ++g) {
                if (!tc::mbar_wait(&s.emptyB[slot], phase ^ 1u, s.abort_flag, err)) break;
                tc::mbar_expect_tx(&s.fullB[slot], (uint32_t)kSlabB);
                tc::tma_load_2d(s.smem + kOffB + slot * kSlabB, tmB, &s.fullB[slot], j * 64, col0 + t * tstride);
                ++issued;
                if (++slot == NS) {
                    slot = 0;
                    phase ^= 1u;
                }
                if (++j == kslabs) {
                    j = 0;
                    if (++t == ntiles) t = 0;
                }
            }
            for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)  // no copies left in flight
                tc::mbar_wait_drain(&s.fullB[g % NS], (uint32_t)(g / NS) & 1u, err);
        }
    }

    // warp 18, lane 0: the U tiles of the same steps and tiles, UH parts per
    // tile in order; U of step i is position u_k0 + i of requests m0 ..
    __device__ static void producer_u(State &s, const CUtensorMap *tmU, int col0, int tstride, int ntiles,
                                      int nsteps, int u_k0, int m0, int32_t *err) {
        if (SU > 0) {
            // U is read once: keep it from displacing W_2^T, which the next steps reuse
            const uint64_t pol = tc::policy_evict_first();
            constexpr int su = SU > 0 ? SU : 1;
            const int total = nsteps * ntiles * UH;
            int issued = 0, st = 0, step = 0, t = 0, part = 0;  // ring slot, step, tile and part of load `issued`
            uint32_t phase = 0;
            for (int g = 0; g < total; ++g) {
                if (!tc::mbar_wait(&s.emptyU[st], phase ^ 1u, s.abort_flag, err)) break;
                unsigned char *dst = s.smem + kOffU + st * kUBytes;
                const int n0 = col0 + t * tstride + part * kUCols;
                tc::mbar_expect_tx(&s.fullU[st], (uint32_t)kUBytes);
                for (int h = 0; h < kUCols / 64; ++h)
                    tc::tma_load_3d_hint(dst + h * kUBox, tmU, &s.fullU[st], n0 + h * 64, u_k0 + step, m0, pol);
                ++issued;
                if (++st == su) {
                    st = 0;
                    phase ^= 1u;
                }
                if (++part == UH) {
                    part = 0;
                    if (++t == ntiles) {
                        t = 0;
                        ++step;
                    }
                }
            }
            for (int g = issued - su < 0 ? 0 : issued - su; g < issued; ++g)
                tc::mbar_wait_drain(&s.fullU[g % su], (uint32_t)(g / su) & 1u, err);
        }
    }

    // warp 17, lane 0: `nsteps` steps of `ntiles` tiles.  The operands of the
    // first `a_ready` steps were written before the roles split; step i >= a_ready
    // starts once the epilogue has written its operand (completion i - a_ready of
    // `aready`).
    __device__ static void mma(State &s, int ntiles, int kslabs, int nsteps, int32_t *err, int a_ready = 1) {
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
        // a descriptor moves with its operand: its low field is the shared
        // address >> 4, which no address of this CTA carries out of
        const uint64_t a_desc0 = tc::smem_desc_k128(tc::smem_u32(s.sA));
        const uint64_t b_desc0 = tc::smem_desc_k128(tc::smem_u32(s.smem + kOffB));
        int issued = 0, slot = 0, b = 0;  // W_2^T ring slot and accumulator of the next MMAs
        uint32_t phase = 0, tphase = 0;
        bool ok = true;
        for (int step = 0; step < nsteps && ok; ++step) {
            if (step >= a_ready) {
                if (!tc::mbar_wait(s.aready, (uint32_t)(step - a_ready) & 1u, s.abort_flag, err)) break;
                tc::tc_fence_after();
            }
            for (int tl = 0; tl < ntiles && ok; ++tl) {
                if (!tc::mbar_wait(&s.tempty[b], tphase ^ 1u, s.abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = s.tmem_base + (uint32_t)(b * BN);
                for (int j = 0; j < kslabs; ++j) {
                    if (!tc::mbar_wait(&s.fullB[slot], phase, s.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint64_t bd = b_desc0 + (uint64_t)((slot * kSlabB) >> 4);
                    const uint64_t ad = a_desc0 + (uint64_t)((j * kSlabA) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int part = 0; part < KSPLIT; ++part)
                            tc::umma_bf16(d, ad + (uint64_t)((4 * part * kSlabA + kk * 32) >> 4),
                                          bd + (uint64_t)((kk * 32) >> 4), idesc,
                                          (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
                    tc::umma_commit(&s.emptyB[slot]);
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc::umma_commit(&s.tfull[b]);
                ++issued;
                if (++b == NACC) {
                    b = 0;
                    tphase ^= 1u;
                }
            }
        }
        if (issued > 0) {  // the last MMAs must finish before TMEM is freed
            const int t = issued - 1;
            tc::mbar_wait_drain(&s.tfull[t % NACC], (uint32_t)(t / NACC) & 1u, err);
        }
    }

    // ---- dynamic tile order ------------------------------------------------
    // The CTAs of one M-tile take vocabulary tiles from a shared counter, so a
    // CTA that streams faster takes more tiles and all finish together.  The
    // producer takes the tiles and announces them to the MMA issuer and the
    // epilogue through a ring of kTileRing words in shared memory: the word of
    // the CTA's k-th tile is (k << 16) | (tile + 1), and tile + 1 == 0 marks
    // the end.  The producer runs at most NACC + NS / kslabs + 1 tiles ahead of the slowest
    // epilogue warp (its slab waits depend on the MMA, which waits for free
    // accumulators), far less than the ring.
    static constexpr int kTileRing = 32;

    __device__ static uint32_t ring_word(int k, int tile) { return ((uint32_t)(k & 0xFFFF) << 16) | (uint32_t)(tile + 1); }

    // ring words start as 0xFFFFFFFF, a tag no tile number below 65535 carries
    __device__ static void ring_init(volatile uint32_t *ring) {
        if (threadIdx.x < kTileRing) ring[threadIdx.x] = 0xFFFFFFFFu;
    }

    // the tile of local index k (-1: no more tiles, or an aborted launch); a
    // bounded wait for the producer's word
    __device__ static int ring_read(const volatile uint32_t *ring, int k, volatile int *abort_flag, int32_t *err) {
        const uint32_t tag = (uint32_t)(k & 0xFFFF);
        uint32_t w = ring[k % kTileRing];
        if ((w >> 16) == tag) return (int)(w & 0xFFFFu) - 1;
        const uint64_t t0 = tc::globaltimer_ns();
        for (;;) {
            __nanosleep(32);
            w = ring[k % kTileRing];
            if ((w >> 16) == tag) return (int)(w & 0xFFFFu) - 1;
            if (*abort_flag) return -1;
            if (tc::globaltimer_ns() - t0 > tc::kWaitLimitNs) {
                *abort_flag = 1;
                set_err(err, DSPARK_ERR_TIMEOUT);
                return -1;
            }
        }
    }

    // warp 16, lane 0: take tiles from *ctr (n_vtiles in all) and stream their
    // W_2^T slabs; the next tile is taken while the current one's slabs are issued
    __device__ static void producer_w2_dyn(State &s, const CUtensorMap *tmB, volatile uint32_t *ring, int *ctr,
                                           int n_vtiles, int kslabs, int32_t *err) {
        int issued = 0, slot = 0;
        uint32_t phase = 0;
        int tile = atomicAdd(ctr, 1);
        for (int k = 0;; ++k) {
            if (tile >= n_vtiles) {
                // the end, at this index and the next three (the epilogue also asks
                // for tiles ahead of its current one, to stage their chunks)
                for (int j = 0; j < 4; ++j) ring[(k + j) % kTileRing] = ring_word(k + j, -1);
                break;
            }
            ring[k % kTileRing] = ring_word(k, tile);
            const int next = atomicAdd(ctr, 1);
            bool ok = true;
            for (int j = 0; j < kslabs; ++j) {
                if (!tc::mbar_wait(&s.emptyB[slot], phase ^ 1u, s.abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc::mbar_expect_tx(&s.fullB[slot], (uint32_t)kSlabB);
                tc::tma_load_2d(s.smem + kOffB + slot * kSlabB, tmB, &s.fullB[slot], j * 64, tile * BN);
                ++issued;
                if (++slot == NS) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;  // the abort flag is up: the other roles stop on their own
            tile = next;
        }
        for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)  // no copies left in flight
            tc::mbar_wait_drain(&s.fullB[g % NS], (uint32_t)(g / NS) & 1u, err);
    }

    // warp 17, lane 0: the tiles the producer announces, after the operand is
    // written (the first completion of `aready`)
    __device__ static void mma_dyn(State &s, const volatile uint32_t *ring, int kslabs, int32_t *err) {
        static_assert(SU == 0, "dynamic tiles stream no U ring");
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
        const uint64_t a_desc0 = tc::smem_desc_k128(tc::smem_u32(s.sA));
        const uint64_t b_desc0 = tc::smem_desc_k128(tc::smem_u32(s.smem + kOffB));
        int issued = 0, slot = 0, b = 0;
        uint32_t phase = 0, tphase = 0;
        bool ok = tc::mbar_wait(s.aready, 0u, s.abort_flag, err);
        if (ok) tc::tc_fence_after();
        for (int k = 0; ok; ++k) {
            if (ring_read(ring, k, s.abort_flag, err) < 0) break;
            if (!tc::mbar_wait(&s.tempty[b], tphase ^ 1u, s.abort_flag, err)) break;
            tc::tc_fence_after();
            const uint32_t d = s.tmem_base + (uint32_t)(b * BN);
            for (int j = 0; j < kslabs; ++j) {
                if (!tc::mbar_wait(&s.fullB[slot], phase, s.abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint64_t bd = b_desc0 + (uint64_t)((slot * kSlabB) >> 4);
                const uint64_t ad = a_desc0 + (uint64_t)((j * kSlabA) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int part = 0; part < KSPLIT; ++part)
                        tc::umma_bf16(d, ad + (uint64_t)((4 * part * kSlabA + kk * 32) >> 4),
                                      bd + (uint64_t)((kk * 32) >> 4), idesc,
                                      (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
                tc::umma_commit(&s.emptyB[slot]);
                if (++slot == NS) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc::umma_commit(&s.tfull[b]);
            ++issued;
            if (++b == NACC) {
                b = 0;
                tphase ^= 1u;
            }
        }
        if (issued > 0) {
            const int t = issued - 1;
            tc::mbar_wait_drain(&s.tfull[t % NACC], (uint32_t)(t / NACC) & 1u, err);
        }
    }

    // warps 0..15: as epilogue(), over the announced tiles; f(k, tile, cofs, acc)
    // with k the CTA's tile count so far and tile the vocabulary tile
    template <class F>
    __device__ static void epilogue_dyn(State &s, const volatile uint32_t *ring, int32_t *err, F &&f) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const uint32_t taddr0 = s.tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)epi_col0();
        for (int k = 0;; ++k) {
            const int b = k % NACC;
            int tile = -1;
            if (lane == 0) {
                tile = ring_read(ring, k, s.abort_flag, err);
                if (tile >= 0 && !tc::mbar_wait(&s.tfull[b], (uint32_t)(k / NACC) & 1u, s.abort_flag, err)) tile = -1;
            }
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            tc::tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < CW / 16; ++h) {
                uint32_t acc[16];
                tc::tmem_ld16(taddr0 + (uint32_t)(b * BN + 16 * h), acc);
                tc::tmem_wait_ld();
                if (h == CW / 16 - 1) {
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&s.tempty[b]);
                }
                f(k, tile, 16 * h, acc);
            }
        }
    }

    // epilogue side of the operand hand-off: called by all epilogue threads after
    // they wrote the next step's operand with generic stores
    __device__ static void operand_written(State &s, int et) {
        tc::fence_proxy_async_smem();
        tc::named_bar_sync(1, kEpiThreads);
        if (et == 0) tc::mbar_arrive(s.aready);
    }

    // warps 0..15: per tile, load this warp's CW accumulator columns of its 32
    // rows 16 at a time and call f(t, n0, cofs, acc, sU) on each chunk (t: tile
    // within this call; n0 = col0 + t tstride: first vocabulary entry of the
    // tile; cofs: the chunk's offset within the warp's CW columns; acc: its 16
    // values; sU: the ring slot of the U part that holds this warp's columns, or null).  The accumulator is released once its
    // last chunk has been read.  Barrier phases continue from tile number tg0
    // (the tiles of earlier steps of the launch).  Per-warp flow, no CTA barrier.
    template <class F>
    __device__ static void epilogue(State &s, int tg0, int col0, int tstride, int ntiles, int32_t *err, F &&f) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const uint32_t taddr0 = s.tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)epi_col0();
        constexpr int su = SU > 0 ? SU : 1;
        for (int t = 0; t < ntiles; ++t) {
            const int tg = tg0 + t, b = tg % NACC;
            const int ug = tg * UH + epi_col0() / kUCols;  // this warp's U part in the ring order
            int ok = 1;
            if (lane == 0) {
                ok = tc::mbar_wait(&s.tfull[b], (uint32_t)(tg / NACC) & 1u, s.abort_flag, err) ? 1 : 0;
                if (ok && SU > 0)
                    ok = tc::mbar_wait(&s.fullU[ug % su], (uint32_t)(ug / su) & 1u, s.abort_flag, err) ? 1 : 0;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (SU > 0) __syncwarp();  // the other lanes read the U tile lane 0 waited for
            tc::tc_fence_after();
            const unsigned char *sU = SU > 0 ? s.smem + kOffU + (ug % su) * kUBytes : nullptr;
#pragma unroll 1
            for (int h = 0; h < CW / 16; ++h) {
                uint32_t acc[16];
                tc::tmem_ld16(taddr0 + (uint32_t)(b * BN + 16 * h), acc);
                tc::tmem_wait_ld();
                if (h == CW / 16 - 1) {
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&s.tempty[b]);
                }
                f(t, col0 + t * tstride, 16 * h, acc, sU);
            }
            __syncwarp();
            if (SU > 0 && lane == 0) tc::mbar_arrive(&s.emptyU[ug % su]);
        }
    }

    // raise row r's shared threshold to the packed winner w (pack_winner)
    __device__ static void publish_thr(State &s, int r, unsigned long long w) {
        atomicMax(&s.thr[r], w);
    }
    __device__ static unsigned long long read_thr(const State &s, int r) {
        return *reinterpret_cast<volatile unsigned long long *>(&s.thr[r]);
    }

    // per-CTA merge scratch in the operand region (valid once every epilogue
    // warp has consumed its last accumulator, until the next operand is written)
    __device__ static float *merge_scratch(const State &s) {
        return reinterpret_cast<float *>(s.sA);
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

// vocabulary column range [c0, c1) of CTA cv out of nparts: equal shares with
// boundaries on multiples of 8 (a TMA box's first column must sit on a 16-byte
// boundary); tiles of BN columns start at c0, the last one cut at c1
__device__ __forceinline__ void col_range(int cv, int nparts, int V, int &c0, int &c1) {
    c0 = (int)(((long long)cv * V / nparts) & ~7ll);
    c1 = cv + 1 == nparts ? V : (int)(((long long)(cv + 1) * V / nparts) & ~7ll);
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
