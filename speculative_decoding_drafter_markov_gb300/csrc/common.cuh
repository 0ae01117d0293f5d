// common.cuh -- device building blocks shared by the DSpark kernels.
//
// * Philox-4x32-10 (Salmon et al., SC'11) and the word -> uniform map.
// * The running state of one row's fused epilogue: the sum of exponentials for
//   the exact softmax normaliser of eq. (4) of the DSpark digest, and its
//   two-level draw: 16-entry vocabulary blocks raced by the Gumbel-max rule on
//   their masses in "exponential race" form, argmax_b ln S_b - ln E_b with
//   E_b = -ln u_b (which equals argmax_b ln S_b - ln(-ln u_b)), then the
//   winning block's entry by inverse CDF.
// * Error reporting into the caller's device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- errors
__device__ __forceinline__ void set_err(int32_t *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- fast exp2
// MUFU ex2 (relative error ~2^-22); ex2(-inf) = +0, ex2(+inf) = +inf.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- paired fp32
// Two independent fp32 operations in one instruction (the f32x2 forms of
// sm_100-family GPUs); each lane rounds exactly like the scalar operation.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// ---------------------------------------------------------------- Philox
struct PhiloxKey {
    uint32_t k0, k1;
};

__device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
    return PhiloxKey{(uint32_t)seed, (uint32_t)(seed >> 32)};
}

// counter word 3: low 30 bits of the cycle, then the 2-bit stream id
__device__ __forceinline__ uint32_t philox_ctr3(uint64_t cycle, uint32_t stream) {
    return (uint32_t)(cycle << 2) | stream;
}

// The 32x32 -> 64-bit products are written as 64-bit multiplies (one wide
// integer multiply each); the round keys k + i W depend only on the seed.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t k0 = key.k0 + (uint32_t)round * 0x9E3779B9u;
        const uint32_t k1 = key.k1 + (uint32_t)round * 0xBB67AE85u;
        const uint64_t p0 = (uint64_t)c.x * 0xD2511F53ull;
        const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57ull;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                       (uint32_t)p0);
    }
    return c;
}

// The 20 round keys of one seed, k + i W for i = 0..9.  The tensor-core kernels
// get them in their launch parameters (computed on the host), so each round's
// key xor takes its operand straight from the parameter bank: a Philox call is
// then two wide multiplies and two three-way xors per round.
struct PhiloxRoundKeys {
    uint32_t k0[10], k1[10];
};

__host__ __device__ inline PhiloxRoundKeys philox_round_keys(uint64_t seed) {
    PhiloxRoundKeys rk;
    for (int i = 0; i < 10; ++i) {
        rk.k0[i] = (uint32_t)seed + (uint32_t)i * 0x9E3779B9u;
        rk.k1[i] = (uint32_t)(seed >> 32) + (uint32_t)i * 0xBB67AE85u;
    }
    return rk;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxRoundKeys &rk) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)c.x * 0xD2511F53ull;
        const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57ull;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk.k0[round], (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ rk.k1[round], (uint32_t)p0);
    }
    return c;
}

// Philox-4x32-10 of counters (w0, w1, req, w3) for a fixed (w1, req), as the
// draft forms them (w1 = step, req = request, w0 = vocabulary quad): the half of
// round 1 and the multiply of round 2 that depend only on (w1, req) are formed
// once per (step, request), so a call starts with one multiply in each of its
// first two rounds.  The words equal philox4x32_10((w0, w1, req, w3), key).
struct PhiloxRow {
    uint32_t n0, n1, h2, l2;
};
__device__ __forceinline__ PhiloxRow philox_row(uint32_t w1, uint32_t req, const PhiloxRoundKeys &rk) {
    const uint64_t p1 = (uint64_t)req * 0xCD9E8D57ull;
    PhiloxRow r;
    r.n0 = (uint32_t)(p1 >> 32) ^ w1 ^ rk.k0[0];
    r.n1 = (uint32_t)p1;
    const uint64_t p0 = (uint64_t)r.n0 * 0xD2511F53ull;
    r.h2 = (uint32_t)(p0 >> 32);
    r.l2 = (uint32_t)p0;
    return r;
}
__device__ __forceinline__ uint4 philox4x32_10(uint32_t w0, uint32_t w3, const PhiloxRow &pr, const PhiloxRoundKeys &rk) {
    const uint64_t q0 = (uint64_t)w0 * 0xD2511F53ull;
    const uint32_t n2 = (uint32_t)(q0 >> 32) ^ w3 ^ rk.k1[0], n3 = (uint32_t)q0;
    const uint64_t q1 = (uint64_t)n2 * 0xCD9E8D57ull;
    uint4 c = make_uint4((uint32_t)(q1 >> 32) ^ pr.n1 ^ rk.k0[1], (uint32_t)q1, pr.h2 ^ n3 ^ rk.k1[1], pr.l2);
#pragma unroll
    for (int round = 2; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)c.x * 0xD2511F53ull;
        const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57ull;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk.k0[round], (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ rk.k1[round], (uint32_t)p0);
    }
    return c;
}

__device__ __forceinline__ uint32_t word_lane(const uint4 &w, int lane) {
    return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

// u = ((w >> 9) + 1/2) 2^-23, exact in fp32
__device__ __forceinline__ float uniform_of(uint32_t w) {
    return __uint2float_rn(w >> 9) * (1.0f / 8388608.0f) + (1.0f / 16777216.0f);
}

// t = 1 - u, also exact: the lattice {(k + 1/2) 2^-23} is symmetric about 1/2.
// Built from the bits: 1 + k' 2^-23 with k' = 2^23 - 1 - (w >> 9), minus
// (1 - 2^-24); the subtraction is exact (Sterbenz).
__device__ __forceinline__ float one_minus_uniform(uint32_t w) {
    const uint32_t bits = ((~w) >> 9) | 0x3F800000u;
    return __uint_as_float(bits) - (1.0f - 1.0f / 16777216.0f);
}

// MUFU log2 (absolute error about 2^-22.6)
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ln E for the unit exponential variate E = -ln u = -ln(1 - t) behind the race.
// For t < 2^-7, E = t + t^2/2 + t^3/3 + t^4/4 (truncation below 2^-28 relative);
// otherwise E = -ln(2) log2(u) with u = 1 - t exact, whose absolute error
// 2^-22.6 is at most 1.4e-5 relative because |log2 u| >= 2^-7 / ln 2.  The final
// logarithm adds about 1e-7, so race scores carry an error below 2e-5.
__device__ __forceinline__ float log_exp_variate(float t) {
    float E;
    if (t < 0.0078125f)
        E = t * fmaf(t, fmaf(t, fmaf(t, 0.25f, 0.33333334f), 0.5f), 1.0f);
    else
        E = -kLn2 * lg2(1.0f - t);
    return kLn2 * lg2(E);
}

// ---------------------------------------------------------------- epilogue state
// One row's running fused-epilogue state: the sum of exponentials for the
// exact normaliser of eq. (4), and the two-level draw of x_k -- vocabulary
// blocks of 16 entries raced by the Gumbel-max rule on their masses
// (score ln S_b - ln E_b, E_b = -ln u_b), the winning block's entry drawn by
// inverse CDF with its second uniform.
struct RowState {
    float m;      // reference of the sum (the max of z, or below it; exp(z - m) stays finite)
    float mL;     // m * log2(e)
    float S;      // sum exp(z - m)
    float best;   // best block score of this thread's blocks
    float zbest;  // z of the entry drawn in that block
    int idx;      // its vocabulary index (-1: none yet)
};

__device__ __forceinline__ void row_init(RowState &s) {
    s.m = -INFINITY;
    s.mL = -INFINITY;
    s.S = 0.f;
    s.best = -INFINITY;
    s.zbest = 0.f;
    s.idx = -1;
}

// The sum of exponentials runs against a reference m that only has to keep
// the terms finite: it is the first block's maximum and moves up only when a
// block's sum leaves [0, 2^64] (a term far above m, or a non-finite logit), so
// a block needs no max and no rescale.  Any reference gives the same
// lse = m + ln S and the same block scores m + ln S_b.
__device__ __forceinline__ void row_set_reference(RowState &s, const float (&z)[16]) {
    float mx[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) mx[j] = z[j];
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
    const float M = fmaxf(s.m, mx[0]);
    s.S = M == -INFINITY ? 0.f : s.S * ex2((s.m - M) * kLog2e);
    s.m = M;
    s.mL = M * kLog2e;
}

// The block's terms e_j = exp(z_j - m) and their sums over aligned runs of 2,
// 4 and 8 entries (pr[i] = e_2i + e_2i+1, qd[i] = pr[2i] + pr[2i+1],
// oc[i] = qd[2i] + qd[2i+1]); returns oc[0] + oc[1].  Arguments and sums two at
// a time (each lane rounds like the scalar operation).
__device__ __forceinline__ float block_exp_sums(const RowState &s, const float (&z)[16], float (&e)[16],
                                                float (&pr)[8], float (&qd)[4], float (&oc)[2]) {
    const float2 L = make_float2(kLog2e, kLog2e), nm = make_float2(-s.mL, -s.mL);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 arg = fma2(make_float2(z[2 * i], z[2 * i + 1]), L, nm);
        e[2 * i] = ex2(arg.x);
        e[2 * i + 1] = ex2(arg.y);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = add2(make_float2(e[4 * i], e[4 * i + 2]), make_float2(e[4 * i + 1], e[4 * i + 3]));
        pr[2 * i] = t.x;
        pr[2 * i + 1] = t.y;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 t = add2(make_float2(pr[4 * i], pr[4 * i + 2]), make_float2(pr[4 * i + 1], pr[4 * i + 3]));
        qd[2 * i] = t.x;
        qd[2 * i + 1] = t.y;
    }
    const float2 t = add2(make_float2(qd[0], qd[2]), make_float2(qd[1], qd[3]));
    oc[0] = t.x;
    oc[1] = t.y;
    return oc[0] + oc[1];
}

template <int N>
__device__ __forceinline__ float select_of(const float (&v)[N], int i) {
    // v[i] by a tree of selects on the bits of i (registers only)
    float w[N];
#pragma unroll
    for (int j = 0; j < N; ++j) w[j] = v[j];
#pragma unroll
    for (int h = N / 2, bit = N / 2; h > 0; h >>= 1, bit >>= 1)
#pragma unroll
        for (int j = 0; j < h; ++j) w[j] = (i & bit) ? w[j + h] : w[j];
    return w[0];
}

// Level 2 of the draw inside one block: the first entry whose running sum of
// e exceeds the target t = u' S_b, found by descending the aligned sums (go to
// the right half when t reaches the left half's sum, less that sum).  A half
// of zero mass is never entered, so the entry has e_j > 0 whatever the
// roundings.  Returns j in 0..15.
__device__ __forceinline__ int block_entry(float t, const float (&e)[16], const float (&pr)[8],
                                           const float (&qd)[4], const float (&oc)[2]) {
    const bool r1 = t >= oc[0] && oc[1] > 0.f;
    t = r1 ? t - oc[0] : t;
    const float qL = r1 ? qd[2] : qd[0], qR = r1 ? qd[3] : qd[1];
    const bool r2 = t >= qL && qR > 0.f;
    t = r2 ? t - qL : t;
    const int qi = (r1 ? 2 : 0) | (r2 ? 1 : 0);
    float pl[4], pg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pl[i] = pr[2 * i];
        pg[i] = pr[2 * i + 1];
    }
    const float pL = select_of(pl, qi), pR = select_of(pg, qi);
    const bool r3 = t >= pL && pR > 0.f;
    t = r3 ? t - pL : t;
    const int pi = 2 * qi + (r3 ? 1 : 0);
    float el[8], eg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        el[i] = e[2 * i];
        eg[i] = e[2 * i + 1];
    }
    const float eL = select_of(el, pi), eR = select_of(eg, pi);
    const bool r4 = t >= eL && eR > 0.f;
    return 2 * pi + (r4 ? 1 : 0);
}

// A race winner as one 64-bit word whose unsigned order is the merge order
// (higher score, then lower index): order-preserving score bits on top, the
// complemented index below.  Zero means "no candidate".
__device__ __forceinline__ unsigned long long pack_winner(float best, int idx) {
    const uint32_t b = __float_as_uint(best);
    const uint32_t ob = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ob << 32) | (uint32_t)~(uint32_t)idx;
}

// Feed one block of 16 consecutive vocabulary entries vb .. vb + 15 of a row
// (vb a multiple of 16; entries at or beyond V carry z = -inf) with the
// block's race word wr and entry word we.  The block's terms join the sum of
// exponentials; its race score is formed and, when it beats `thr` (a packed
// winner of the same row: this thread's best or a better one found elsewhere;
// a block below it cannot win the row), the entry is drawn and the block
// becomes this thread's best.  Returns whether it did.
__device__ __forceinline__ bool block_feed16(RowState &s, const float (&z)[16], int vb, uint32_t wr, uint32_t we,
                                             unsigned long long thr) {
    if (s.m == -INFINITY) row_set_reference(s, z);  // the row's first block in this thread
    float e[16], pr[8], qd[4], oc[2];
    float S = block_exp_sums(s, z, e, pr, qd, oc);
    if (!(S <= 18446744073709551616.f)) {  // 2^64: move the reference up to this block's maximum
        row_set_reference(s, z);
        S = block_exp_sums(s, z, e, pr, qd, oc);
    }
    s.S += S;
    if (!(S > 0.f)) return false;  // no mass at this reference (entries beyond V, or far below m)
    const float score = s.m + kLn2 * lg2(S) - log_exp_variate(one_minus_uniform(wr));
    if (pack_winner(score, vb) <= thr) return false;
    const int j = block_entry(uniform_of(we) * S, e, pr, qd, oc);
    s.best = score;
    s.idx = vb + j;
    s.zbest = select_of(z, j);
    return true;
}

__device__ __forceinline__ int winner_index(unsigned long long w) { return (int)~(uint32_t)w; }
__device__ __forceinline__ float winner_score(unsigned long long w) {
    if (w == 0ull) return -INFINITY;
    const uint32_t ob = (uint32_t)(w >> 32);
    return __uint_as_float((ob & 0x80000000u) ? (ob & 0x7FFFFFFFu) : ~ob);
}

// Combine two states (b into a).  Ties of the race go to the lower index.
__device__ __forceinline__ void row_merge(RowState &a, float m, float S, float best, float zbest,
                                          int idx) {
    const float M = fmaxf(a.m, m);
    if (M == -INFINITY) {
        a.S = 0.f;
    } else {
        a.S = a.S * ex2((a.m - M) * kLog2e) + S * ex2((m - M) * kLog2e);
    }
    a.m = M;
    a.mL = M * kLog2e;
    if (idx >= 0 && (a.idx < 0 || best > a.best || (best == a.best && idx < a.idx))) {
        a.best = best;
        a.zbest = zbest;
        a.idx = idx;
    }
}

// Partial result of one (row, vocabulary slice) of a draft step (32 bytes, so
// a merge reads it with two 16-byte loads).
struct __align__(16) DraftPartial {
    float m, S, best, zbest;
    int idx, pad0, pad1, pad2;
};

__device__ __forceinline__ DraftPartial make_partial(float m, float S, float best, float zbest, int idx) {
    return DraftPartial{m, S, best, zbest, idx, 0, 0, 0};
}

// L2 read of a partial written by another CTA of the same launch
__device__ __forceinline__ DraftPartial load_partial_cg(const DraftPartial *q) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(q));
    const int4 b = __ldcg(reinterpret_cast<const int4 *>(q) + 1);
    return DraftPartial{a.x, a.y, a.z, a.w, b.x, 0, 0, 0};
}

// Partial result of one (row, vocabulary slice) of verification phase 2 on the
// CUDA cores: the sums of the residual weights max(0, p - q) and of p.
struct VerifyPartial {
    float sum_res, sum_p;
};

}  // namespace dspark
