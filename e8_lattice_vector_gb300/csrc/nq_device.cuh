// nq_device.cuh -- device building blocks of the E8 KV-cache codec (sm_103a).
//
// Arithmetic contract: every floating-point operation that decides a code is
// written with an explicit IEEE intrinsic (__fadd_rn, __fmul_rn, __fmaf_rn ...)
// and the library is built with --fmad=false, so the compiler fuses nothing on
// its own.  The op order is the one the method's steps define:
//   RoPE removal   x_i' = fma(x_i, c, x_j*s),  x_j' = fma(x_j, c, -(x_i*s))
//   Hadamard       butterflies (a + b, a - b); compression runs the stages
//                  h = 1, ..., Dp/8, Dp/2, Dp/4, decompression h = 1, ..., Dp/2
//   scaling        u = y * inv,  inv = 1 / (sc * Dp)
//   E8 distances   d = fma(e_j, e_j, d) over j = 0..7, plus 1 - 2*score for a
//                  parity fix-up, as fma(-2, score, 1) added to d (the fast
//                  path reaches the same coset choice from an estimate whose
//                  sign provably agrees outside a narrow band; see e8_fast).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace nq {

constexpr unsigned kFull = 0xffffffffu;
// 1.5 * 2^23: for |x| < 2^22, (x + kMagic) rounds x to the nearest integer
// with ties to even (kMagic is even) and keeps that integer in the low
// mantissa bits; (x + kMagic) - kMagic is then rint(x) exactly.
constexpr float kMagic = 12582912.0f;

template <int BITS>
struct Code {
    static constexpr int L = 1 << BITS;
    static constexpr unsigned MASK = L - 1;
    static constexpr int BLOCK_BITS = 8 * BITS;
    static constexpr float HI0 = float(L / 2 - 1);   // integer-coset box edge
    static constexpr float H = float(L - 1) * 0.5f;  // half-coset box edge
    static constexpr unsigned OFF0 = L / 2 - 1;      // code of integer 0
    // high bit of each of the 8 fields of a block code (SWAR mod-2^b ops)
    static constexpr unsigned FIELD_HI =
        (1u << (BITS - 1)) * (1u | (1u << BITS) | (1u << 2 * BITS) | (1u << 3 * BITS) |
                              (1u << 4 * BITS) | (1u << 5 * BITS) | (1u << 6 * BITS) |
                              (1u << 7 * BITS));
};

// Field-wise (a - b) mod 2^b and (a + b) mod 2^b of 8 packed b-bit fields.
// Two-bit fields take a bit-level form: the low bit is a0 ^ b0, and the high
// bit a1 ^ b1 ^ k with k the borrow (~a0 & b0) or carry (a0 & b0) of the low
// bit, shifted into its own field only (three logic and shift operations
// instead of the masked integer add's five).  Wider fields mask the high bit
// of each field so that a carry or borrow stays inside it.
template <int BITS>
__device__ __forceinline__ unsigned swar_sub(unsigned a, unsigned b) {
    constexpr unsigned H = Code<BITS>::FIELD_HI;
    if constexpr (BITS == 2)
        return a ^ b ^ ((~a & b & (H >> 1)) << 1);
    else
        return ((a | H) - (b & ~H)) ^ ((a ^ ~b) & H);
}
template <int BITS>
__device__ __forceinline__ unsigned swar_add(unsigned a, unsigned b) {
    constexpr unsigned H = Code<BITS>::FIELD_HI;
    if constexpr (BITS == 2)
        return a ^ b ^ ((a & b & (H >> 1)) << 1);
    else
        return ((a & ~H) + (b & ~H)) ^ ((a ^ b) & H);
}

// Strict-E8 joint enumeration of a block in exactly 8b bits.  In both cosets
// of strict E8 the field sum m_0 + ... + m_7 is even (the coordinate sum is
// even and the offsets add a multiple of 8 * (L - 1) / 2 that is even), so the
// low bit of m_7 follows from the other fields and its place holds the coset
// bit: fields 0..6 as they are, m_7 >> 1 in the next b - 1 bits, the coset in
// the top bit.
template <int BITS>
__device__ __forceinline__ unsigned joint_pack(unsigned code, unsigned coset) {
    constexpr int SH = 7 * BITS;
    const unsigned m7 = (code >> SH) & Code<BITS>::MASK;
    return (code & ((1u << SH) - 1u)) | ((m7 >> 1) << SH) | (coset << (8 * BITS - 1));
}
template <int BITS>
__device__ __forceinline__ unsigned joint_split(unsigned joint, unsigned& coset) {
    constexpr int SH = 7 * BITS;
    constexpr unsigned LOW7 = (Code<BITS>::FIELD_HI >> (BITS - 1)) & ((1u << SH) - 1u);  // bit j*b, j < 7
    coset = (joint >> (8 * BITS - 1)) & 1u;
    const unsigned parity = __popc(joint & LOW7) & 1u;
    const unsigned hi = (joint >> SH) & ((1u << (BITS - 1)) - 1u);
    return (joint & ((1u << SH) - 1u)) | (((hi << 1) | parity) << SH);
}

// Field-wise (a + b) mod 4 of the 16 two-bit fields of a packed word (the
// bit-level form of swar_add<2>).
__device__ __forceinline__ unsigned swar_add_word2(unsigned a, unsigned b) {
    constexpr unsigned LO = 0x55555555u;  // low bit of every field
    return a ^ b ^ ((a & b & LO) << 1);
}

// ------------------------------------------------------------------ Hadamard

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    unsigned long long pa, pb, r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1,%2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pa), "l"(pb));
    float2 d;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(r));
    return d;
}

// One butterfly stage (a, b) -> (a + b, a - b) over pairs (i, i + h).  The
// packed f32x2 instructions pair slots (i, i + P): for h != P the butterflies
// (i, i+h) and (i+P, i+P+h) share one packed add and one subtract (each half
// is an ordinary IEEE round-to-nearest operation, so the results are those of
// the scalar butterflies); the stage h == P runs scalar.  P = 1 pairs
// neighbouring slots, P = 4 the two halves of an 8-block (the pairing the
// compression side's E8 search wants).
template <int N, int P = 1>
__device__ __forceinline__ void fwht_stage(float (&y)[N], int h) {
    if (h == P) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if ((i & P) == 0) {
                const float a = y[i], b = y[i + P];
                y[i] = __fadd_rn(a, b);
                y[i + P] = __fsub_rn(a, b);
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if ((i & P) == 0 && (i & h) == 0) {
            const float2 a = make_float2(y[i], y[i + P]);
            const float2 b = make_float2(y[i + h], y[i + h + P]);
            const float2 s = __fadd2_rn(a, b);
            const float2 d = fsub2(a, b);
            y[i] = s.x;
            y[i + P] = s.y;
            y[i + h] = d.x;
            y[i + h + P] = d.y;
        }
    }
}

// Unnormalised Walsh-Hadamard transform in the textbook stage order h = 1, 2,
// ..., N/2 (the decompression direction).
template <int N>
__device__ __forceinline__ void fwht(float (&y)[N]) {
#pragma unroll
    for (int h = 1; h < N; h *= 2) fwht_stage<N>(y, h);
}

// Butterfly stage on slot pairs (l, l + Q) with a per-thread sign:
// (P, Q) -> (P + sgn*Q, P - sgn*Q).  fma(x, +-1, y) is exactly y +- x, so with
// sgn = +1 this is the plain butterfly and with sgn = -1 it is the butterfly
// with its two outputs exchanged.  Packed pairs as in fwht_stage.
template <int N, int P = 1>
__device__ __forceinline__ void stage_signed(float (&y)[N], float sgn) {
    constexpr int Q = N / 2;
#pragma unroll
    for (int l = 0; l < Q; ++l) {
        if ((l & P) == 0) {
            const float2 p = make_float2(y[l], y[l + P]);
            const float2 q = make_float2(y[l + Q], y[l + Q + P]);
            const float2 a = __ffma2_rn(q, make_float2(sgn, sgn), p);
            const float2 b = __ffma2_rn(q, make_float2(-sgn, -sgn), p);
            y[l] = a.x;
            y[l + P] = a.y;
            y[l + Q] = b.x;
            y[l + Q + P] = b.y;
        }
    }
}

// Exchange stage between the two threads of a row: each sends slots
// [N/2, N) to its partner and makes (own + recv, own - recv) from slots
// [0, N/2) and the received values.  Packed pairs as in fwht_stage.
template <int N, int P = 1>
__device__ __forceinline__ void stage_exchange(float (&y)[N]) {
    constexpr int Q = N / 2;
    float r[Q];
#pragma unroll
    for (int l = 0; l < Q; ++l) r[l] = __shfl_xor_sync(kFull, y[l + Q], 1);
#pragma unroll
    for (int l = 0; l < Q; ++l) {
        if ((l & P) == 0) {
            const float2 a = make_float2(y[l], y[l + P]);
            const float2 b = make_float2(r[l], r[l + P]);
            const float2 s = __fadd2_rn(a, b);
            const float2 d = fsub2(a, b);
            y[l] = s.x;
            y[l + P] = s.y;
            y[l + Q] = d.x;
            y[l + Q + P] = d.y;
        }
    }
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// ------------------------------------------------------------------- scale

// Smallest binary16 v with v * step >= amax (step = Dp * (2^b - 1) / 2), as
// bits.  Candidate: amax * (1 / step) rounded to fp16 -- within two fp32 ulps
// of amax / step, so at most one fp16 step away from the answer -- then one
// step up or down decided by the exact products v * step (fp16 times a small
// integer or half-integer is exact in fp32).
__device__ __forceinline__ unsigned short group_scale(float amax, float step, float inv_step) {
    if (!(amax > 0.0f)) return 0;
    float q = __fmul_rn(amax, inv_step);
    unsigned short v = __half_as_ushort(__float2half_rn(q));
    if (__fmul_rn(__half2float(__ushort_as_half(v)), step) < amax) {
        ++v;
    } else if (v > 0 && __fmul_rn(__half2float(__ushort_as_half((unsigned short)(v - 1))), step) >= amax) {
        --v;
    }
    return v;
}

// ------------------------------------------------------------- E8 decoder

// General decoder for one coset: rounding clamped into [-hi, hi] (hi = +inf
// for the unbounded lattice), optional even-sum fix-up on the coordinate of
// largest score (|e| for a step toward u, -|e| for a step away from it, first
// index on ties).  Writes the point, returns the squared distance.
__device__ __forceinline__ float coset_general(const float (&u)[8], bool half, bool parity,
                                               float hi, float (&r)[8]) {
    float e[8];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float v = half ? __fsub_rn(ceilf(u[j]), 0.5f) : rintf(u[j]);
        v = fminf(fmaxf(v, -hi), hi);
        r[j] = v;
        e[j] = __fsub_rn(u[j], v);
        sum += __float2int_rn(half ? __fsub_rn(v, 0.5f) : v);
    }
    float d = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) d = __fmaf_rn(e[j], e[j], d);
    if (parity && (sum & 1)) {
        int k = 0;
        float best = 0.0f, best_dir = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float dir = (e[j] >= 0.0f) ? 1.0f : -1.0f;
            float score = fabsf(e[j]);
            float moved = __fadd_rn(r[j], dir);
            if (moved > hi || moved < -hi) {
                dir = -dir;
                score = -score;
            }
            if (j == 0 || score > best) {
                k = j;
                best = score;
                best_dir = dir;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j == k) r[j] = __fadd_rn(r[j], best_dir);
        d = __fadd_rn(d, __fmaf_rn(-2.0f, best, 1.0f));
    }
    return d;
}

// Nearest codebook point, general path.  Returns the coset (0 / 1).
__device__ __forceinline__ int e8_general(const float (&u)[8], bool strict, float hi0, float h,
                                          float (&r)[8]) {
    float r0[8], r1[8];
    float d0 = coset_general(u, false, true, hi0, r0);
    float d1 = coset_general(u, true, strict, h, r1);
    bool c = d1 < d0;
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = c ? r1[j] : r0[j];
    return c ? 1 : 0;
}

// Fast path, valid when every |u_j| < (2^b - 1)/2 (then no rounding leaves the
// box and the half-integer fix-up never needs to turn around).  Computes the
// same codes as the general path:
//   e~0 = rint(u) - u  (exact, never -0); the half-integer point is
//   rint(u) + 1/2 if e~0 < 0 else rint(u) - 1/2 (= ceil(u) - 1/2), so its
//   residual is e~1 = e~0 - copysign(1/2, e~0); the integer score is
//   min(|e~0|, hi0 - |u|) (a step that would leave the box turns around).
//
// Coset choice.  Per coordinate |e~1| = 1/2 - |e~0| exactly, so
// e~0^2 - e~1^2 = |e~0| - 1/4 and, with the fix-up costs 1 - 2*score,
//   D = d0' - d1' = sum_j |e~0_j| - 2 + odd0 (1 - 2 smax0) - odd1 (1 - 2 smax1)
// in exact arithmetic.  The general path (the method's own procedure) sums the
// squared residuals in fp32; each of its two distances is within 1.3e-6 of the
// exact value (eight roundings of numbers below 3, one rounding of e~1), and
// the estimate of D formed here is within 1.2e-6 of the exact D.  So wherever
// |estimate| > 2^-16 the sign of the estimate is the sign of the general
// path's comparison; inside that band the function returns false and the
// caller runs the general path.
//
// The codes are accumulated as exact integer-valued floats on the FMA pipe
// (sum of r_j * L^j over half-blocks of 4 coordinates, < 2^16), the parities
// by xor of the magic-rounded bit patterns.  Coordinates j and j + 4 share
// packed f32x2 instructions (each half an ordinary IEEE operation), so the
// two lanes of an accumulator are the two half-blocks and every sum comes out
// of the packed operations whole.  A block whose chosen coset needs a fix-up
// with a tie for the maximal score or a maximal score <= 2^-100 (every
// coordinate nearly an integer or past the box edge) is not handled here
// either.
//
// POINT: instead of the code, write the chosen lattice point itself into u
// (r0 - hb cs + m ind cs per coordinate: exact multiples of 1/2), for a caller
// that dequantizes at once (the one-pass round trip); the code accumulators
// are then not formed.  The point is the one the code names.
template <int BITS, bool STRICT, bool POINT, typename U>
__device__ __forceinline__ bool e8_fast_core(U& u, unsigned& code, unsigned& coset) {
    using C = Code<BITS>;
    constexpr float L = float(C::L);
    constexpr float Lp[4] = {1.0f, L, L * L, L * L * L};
    constexpr float SUML = 1.0f + L + L * L + L * L * L;
    constexpr float TWO23 = 8388608.0f;
    constexpr float BAND = 1.52587890625e-05f;  // 2^-16
    const float2 M2 = make_float2(kMagic, kMagic);
    // clv_j = cs_j L^(j mod 4) with cs_j = copysign(1/2, e~0_j): the sign bit
    // of e~0_j on the power of two L^(j mod 4) / 2 (one logic op, exact); the
    // weights restart at each half-block, whose code is a field of its own
    float eb1[8], s0[8], clv[8];  // eb1: |e~1| (strict)
    // S = sum |e~0_j| in two accumulators; the strict decoder sums
    // -2 cs_j e~0_j = -|e~0_j| instead (it needs -2 cs_j for |e~1| anyway), an
    // exact rescaling of each term
    float2 S = make_float2(0.0f, 0.0f);
    // A = 2^23 + (L/2 - 1) SUML + sum r0_j L^j: 2^23 plus the integer code
    // B = sum cs_j L^j - SUML / 2, so that A - B = 2^23 plus the half code
    // (lane x: coordinates 0-3, lane y: coordinates 4-7)
    constexpr float A0 = TWO23 + float(C::OFF0) * SUML;
    constexpr float B0 = -0.5f * SUML;
    float2 A = make_float2(A0, A0);
    float2 B = make_float2(B0, B0);
    unsigned x0 = 0, xs = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 uu = make_float2(u[j], u[j + 4]);
        const float2 t = __fadd2_rn(uu, M2);
        const float2 r0 = fsub2(t, M2);
        const float2 e0 = fsub2(r0, uu);
        const float2 cl = make_float2(copysignf(0.5f * Lp[j], e0.x), copysignf(0.5f * Lp[j], e0.y));
        clv[j] = cl.x;
        clv[j + 4] = cl.y;
        if constexpr (!POINT) {
            A = __ffma2_rn(r0, make_float2(Lp[j], Lp[j]), A);
            B = __fadd2_rn(B, cl);
        }
        s0[j] = fminf(fabsf(e0.x), __fsub_rn(C::HI0, fabsf(uu.x)));
        s0[j + 4] = fminf(fabsf(e0.y), __fsub_rn(C::HI0, fabsf(uu.y)));
        x0 ^= __float_as_uint(t.x) ^ __float_as_uint(t.y);
        if (STRICT) {
            // -2 copysign(1/2, e~0) = -2 cl / L^j (exact; no sign operations)
            const float2 m2cs = __fmul2_rn(cl, make_float2(-2.0f / Lp[j], -2.0f / Lp[j]));
            S = __ffma2_rn(m2cs, e0, S);  // -|e~0| per coordinate (exact products)
            // |e~1| = |e~0 - cs| = 1/2 - |e~0|, rounded once: the magnitude of e~0 - cs
            const float2 a1 = __ffma2_rn(m2cs, e0, make_float2(0.5f, 0.5f));
            eb1[j] = a1.x;
            eb1[j + 4] = a1.y;
            xs ^= __float_as_uint(e0.x) ^ __float_as_uint(e0.y);
        } else {
            S.x = __fadd_rn(S.x, fabsf(e0.x));
            S.y = __fadd_rn(S.y, fabsf(e0.y));
        }
    }
    const float smax0 = fmax3(fmax3(s0[0], s0[1], s0[2]), fmax3(s0[3], s0[4], s0[5]), fmaxf(s0[6], s0[7]));
    float smax1 = 0.0f;
    if (STRICT)
        smax1 = fmax3(fmax3(eb1[0], eb1[1], eb1[2]), fmax3(eb1[3], eb1[4], eb1[5]), fmaxf(eb1[6], eb1[7]));
    const bool odd0 = (x0 & 1u) != 0;
    const bool odd1 = STRICT && (((x0 ^ (xs >> 31)) & 1u) != 0);  // + number of e~0 < 0
    float D = STRICT ? __fsub_rn(-2.0f, __fadd_rn(S.x, S.y)) : __fsub_rn(__fadd_rn(S.x, S.y), 2.0f);  // sum |e~0| - 2
    if (odd0) D = __fadd_rn(D, __fmaf_rn(-2.0f, smax0, 1.0f));
    if (odd1) D = __fsub_rn(D, __fmaf_rn(-2.0f, smax1, 1.0f));
    bool ok = fabsf(D) > BAND;
    const bool half = D > 0.0f;

    // fix-up of the chosen coset: move its first maximal-score coordinate k one
    // step toward u, i.e. add -2*cs_k*L^k to the integer code (u above rint(u)
    // moves up) or +2*cs_k*L^k to the half-integer code.  k is found on the FMA
    // pipe: i_j = sat(1 - (smax - s_j) * 2^127) is 1 at a maximum and 0
    // elsewhere (with smax > 2^-100, distinct scores differ by at least 2^-123),
    // and G = sum_j i_j cs_j L^j picks cs_k L^k (G.x over coordinates 0-3, G.y
    // over 4-7).  A tie goes to the general path.  Computed for every block (no
    // branch), applied if needed.
    const bool fix = half ? odd1 : odd0;
    const float smax = STRICT ? (half ? smax1 : smax0) : smax0;  // relaxed: a fix-up means the integer coset
    // POINT: the fix-up step m and the half-integer shift hb, needed in the loop
    float mpt = 0.0f, hbpt = 0.0f;
    if constexpr (POINT) {
        mpt = fix ? (half ? 2.0f : -2.0f) : 0.0f;
        hbpt = half ? 1.0f : 0.0f;
    }
    float2 G = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 sj = (STRICT && half) ? make_float2(eb1[j], eb1[j + 4])
                                           : make_float2(s0[j], s0[j + 4]);
        const float2 dlt = fsub2(make_float2(smax, smax), sj);
        float2 ind;
        asm("fma.rn.sat.f32 %0, %1, 0fFF000000, 0f3F800000;" : "=f"(ind.x) : "f"(dlt.x));
        asm("fma.rn.sat.f32 %0, %1, 0fFF000000, 0f3F800000;" : "=f"(ind.y) : "f"(dlt.y));
        G = __ffma2_rn(ind, make_float2(clv[j], clv[j + 4]), G);
        if constexpr (POINT) {  // r0 again (magic rounding), cs = cl / L^j, then r0 + cs (m ind - hb)
            const float2 uu = make_float2(u[j], u[j + 4]);
            const float2 r0 = fsub2(__fadd2_rn(uu, M2), M2);
            const float2 csj = __fmul2_rn(make_float2(clv[j], clv[j + 4]), make_float2(1.0f / Lp[j], 1.0f / Lp[j]));
            const float2 w = __ffma2_rn(ind, make_float2(mpt, mpt), make_float2(-hbpt, -hbpt));
            const float2 pt = __ffma2_rn(csj, w, r0);
            u[j] = pt.x;
            u[j + 4] = pt.y;
        }
    }
    // A unique maximum leaves one term +-L^k / 2, a power of two, in exactly one
    // half-block; ties leave sums of distinct +-L^j / 2 (L >= 4), which are
    // never powers of two (L^b times an odd number of magnitude >= 3), or terms
    // in both halves.  For b <= 3 the upper half is weighted by L^4, making the
    // eight terms distinct powers +-L^j / 2, j = 0..7, whose sum is exact (at
    // most 7b + 1 <= 22 significant bits): one power-of-two test covers both
    // cases.  For b = 4 that sum could round, so the halves are tested apart.
    bool unique;
    if constexpr (BITS <= 3) {
        constexpr float L4 = L * L * L * L;
        unique = (__float_as_uint(__fmaf_rn(G.y, L4, G.x)) & 0x7fffffu) == 0u;
    } else {
        const bool one = (G.x == 0.0f) != (G.y == 0.0f);
        unique = one && (__float_as_uint(__fadd_rn(G.x, G.y)) & 0x7fffffu) == 0u;
    }
    ok = ok && (!fix || (smax > 7.88860905e-31f && unique));  // 2^-100
    if constexpr (!POINT) {
        const float m = fix ? (half ? 2.0f : -2.0f) : 0.0f;
        const float hb = half ? 1.0f : 0.0f;

        // integer codes m0 = r0 + (L/2 - 1), half-integer codes m1 = r1 + (L - 1)/2,
        // per half-block an exact integer below 2^16 in the low bits of 2^23 + m
        // (every intermediate is a multiple of 1/2 below 2^24, so all of this is exact)
        // (two fused steps, each exact: every intermediate is an integer-valued float below 2^24)
        const float2 f = __ffma2_rn(G, make_float2(m, m), __ffma2_rn(B, make_float2(-hb, -hb), A));
        const unsigned fx = __float_as_uint(f.x), fy = __float_as_uint(f.y);
        if constexpr (BITS == 2)  // 8-bit half codes, the bits above them zero: one byte permutation
            code = __byte_perm(fx, fy, 0x1140);
        else if constexpr (BITS == 4)  // 16-bit half codes
            code = __byte_perm(fx, fy, 0x5410);
        else
            code = (fx & 0xffffu) | ((fy & 0xffffu) << (4 * BITS));
    }
    coset = half ? 1u : 0u;
    return ok;
}

template <int BITS, bool STRICT>
__device__ __forceinline__ bool e8_fast(const float (&u)[8], unsigned& code, unsigned& coset) {
    return e8_fast_core<BITS, STRICT, false>(u, code, coset);
}

// The fast path's lattice point in place of u (coordinates, not codes).
template <int BITS, bool STRICT>
__device__ __forceinline__ bool e8_fast_point(float (&u)[8], unsigned& coset) {
    unsigned unused;
    return e8_fast_core<BITS, STRICT, true>(u, unused, coset);
}

// Block code of a general-path point.
template <int BITS>
__device__ __forceinline__ unsigned pack_point(const float (&r)[8], int coset);

// The general path as an out-of-line call (it is rare: only rows whose scaled
// maximum reaches the box edge exactly take it), arguments and result in
// registers.  Returns (block code, coset).
template <int BITS, bool STRICT>
__device__ __noinline__ uint2 e8_slow(float4 lo, float4 hi) {
    using C = Code<BITS>;
    const float u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float r[8];
    const int c = e8_general(u, STRICT, C::HI0, C::H, r);
    return make_uint2(pack_point<BITS>(r, c), unsigned(c));
}

template <int BITS>
__device__ __forceinline__ unsigned pack_point(const float (&r)[8], int coset) {
    using C = Code<BITS>;
    const float off = coset ? C::H : C::HI0;
    unsigned code = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) code |= (unsigned)__float2int_rn(__fadd_rn(r[j], off)) << (j * BITS);
    return code;
}

// Block code -> the 8 unscaled coordinates y_j = (m_j - offset) * sc, exact:
// 2^22 + m_j is built from its bits (the fp32 spacing at 2^22 is 1/2, so the
// field goes in shifted left by one), 2^22 + offset is exact for the integer
// and the half-integer offsets alike, their difference is m_j - offset, and
// that small half-integer times the fp16 scale is exact too.  Pairs of
// coordinates share packed f32x2 instructions.
template <int BITS>
__device__ __forceinline__ void unscale_block(unsigned code, unsigned coset, float sc, float* y) {
    using C = Code<BITS>;
    const float k = coset ? 4194304.0f + C::H : 4194304.0f + C::HI0;
    const float2 k2 = make_float2(k, k), s2 = make_float2(sc, sc);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const unsigned a = j ? (code >> (j * BITS - 1)) : (code << 1);
        const unsigned b = code >> ((j + 1) * BITS - 1);
        const float2 t = make_float2(__uint_as_float((a & (C::MASK << 1)) | 0x4A800000u),
                                     __uint_as_float((b & (C::MASK << 1)) | 0x4A800000u));
        const float2 v = __fmul2_rn(fsub2(t, k2), s2);
        y[j] = v.x;
        y[j + 1] = v.y;
    }
}

// ------------------------------------------------------------ fp16 <-> fp32

__device__ __forceinline__ void h8_to_f(const uint4& v, float* y) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float2 f = __half22float2(h[q]);
        y[2 * q] = f.x;
        y[2 * q + 1] = f.y;
    }
}

// Round to fp16 (nearest even), saturating at +-65504: a finite input never
// comes back as an infinity.
__device__ __forceinline__ unsigned f2_to_h2_sat(float lo, float hi) {
    unsigned r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 f_to_h8(const float* y) {
    return make_uint4(f2_to_h2_sat(y[0], y[1]), f2_to_h2_sat(y[2], y[3]), f2_to_h2_sat(y[4], y[5]),
                      f2_to_h2_sat(y[6], y[7]));
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------- tile staging (smem)

// A tile is 32 consecutive tokens of one slice; one warp owns it, lane r owns
// row r.  fp16 rows are staged in shared memory as two 4 KB boxes of
// 32 rows x 128 bytes (head_dim columns 0-63 and 64-127); inside a box the
// 16-byte chunk c of row r sits at chunk position c ^ (r & 7).  That is the
// TMA 128-byte swizzle, so a row read or write by one lane per row is free of
// bank conflicts, and a tensor store can move the tile out unchanged.
constexpr int kTileRows = 32;
constexpr int kTileBytes = 8192;

__device__ __forceinline__ uint32_t swz(int r, int q) {
    return uint32_t(((q >> 3) << 12) + (r << 7) + (((q & 7) ^ (r & 7)) << 4));
}

// The same layout for a 16-row tile (boxes of 16 rows x 128 bytes = 2 KB).
constexpr int kPairRows = 16;
constexpr int kPairTileBytes = 4096;
__device__ __forceinline__ uint32_t swz16(int r, int q) {
    return uint32_t(((q >> 3) << 11) + (r << 7) + (((q & 7) ^ (r & 7)) << 4));
}

// Two threads per row (lanes 2r and 2r+1 share row r): thread hf owns the
// coordinates hf*Q + l (slot l < Q) and DP/2 + hf*Q + (l - Q) (slot l >= Q),
// Q = DP/4, so the RoPE partners (i, i + DP/2) sit in slots (l, l + Q).
template <int DP>
struct PairMap {
    static constexpr int HALF = DP / 2;  // coordinates per thread
    static constexpr int Q = DP / 4;
    static constexpr int NBT = HALF / 8;  // 8-blocks (and 16-byte fp16 chunks) per thread
    // global 16-byte chunk (8 coordinates) of the thread's slot chunk c
    __device__ static __forceinline__ int chunk(int hf, int c) {
        return c < Q / 8 ? hf * (Q / 8) + c : DP / 16 + hf * (Q / 8) + (c - Q / 8);
    }
};

// Shared-memory address of the thread's slot chunk c of row r in a 16-row
// tile, swz16(r, PairMap<DP>::chunk(hf, c)), split into the lane's part
// (row offset, and the swizzle bits of hf * DP/32 and r) and the chunk's own
// immediate: the chunk bits of slot chunk c are disjoint from hf * DP/32.
template <int DP>
struct PairTileAddr {
    uint32_t base, x0;
    __device__ __forceinline__ PairTileAddr(uint32_t stage, int r, int hf)
        : base(stage + (uint32_t(r) << 7)), x0(uint32_t((hf * (DP / 32)) ^ (r & 7)) << 4) {}
    __device__ __forceinline__ uint32_t operator()(int c) const {
        const int cp = c < DP / 32 ? c : c + DP / 16 - DP / 32;  // chunk(hf, c) - hf * DP/32
        return base + (uint32_t(cp >> 3) << 11) + (x0 ^ (uint32_t(cp & 7) << 4));
    }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared async copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ unsigned lds32(uint32_t a) {
    unsigned v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts32(uint32_t a, unsigned v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts16(uint32_t a, unsigned v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, const uint4& v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Slots of an S-deep ring for loop step i: cur = i mod S (the tile computed
// now), pre = (i + S - 1) mod S (the tile being prefetched), kept by
// wrapping increments instead of a modulo per step.
template <int S>
struct RingSlots {
    int cur = 0, pre = S - 1;
    __device__ __forceinline__ void advance() {
        cur = cur + 1 == S ? 0 : cur + 1;
        pre = pre + 1 == S ? 0 : pre + 1;
    }
};

// Work items: (slice, chunk of `chunk` tokens), item = slice * nchunks + c; a
// warp walks its items' tiles of ROWS tokens in order, items first, first +
// step, ...  Two copies of the walk run one pipeline depth apart (the one that
// prefetches and the one that computes).  The divisions happen once, in the
// constructor: moving to the next item adds step = dslice * nchunks + dc as a
// (slice, c) pair with one carry; the walk ends when slice reaches slices.
template <int ROWS>
struct TileWalkT {
    static constexpr bool kGroups = false;  // single tiles, no delta groups
    int64_t slice, slices, dslice;
    int nchunks, chunk, tokens, c, dc, t0;
    __device__ TileWalkT(int64_t first, int64_t step, int64_t slices_, int tokens_, int chunk_)
        : slices(slices_), chunk(chunk_), tokens(tokens_) {
        nchunks = (tokens_ + chunk_ - 1) / chunk_;
        slice = slices_;  // no work when there are no chunks
        dslice = 0;
        c = dc = 0;
        if (nchunks > 0) {
            slice = first / nchunks;
            c = int(first - slice * nchunks);
            dslice = step / nchunks;
            dc = int(step - dslice * nchunks);
        }
        t0 = c * chunk;
    }
    __device__ __forceinline__ bool valid() const { return slice < slices; }
    __device__ __forceinline__ int t_begin() const { return c * chunk; }
    __device__ __forceinline__ int t_end() const { return min(c * chunk + chunk, tokens); }
    __device__ __forceinline__ void next() {
        t0 += ROWS;
        if (t0 >= t_end()) {
            slice += dslice;
            c += dc;
            if (c >= nchunks) {
                c -= nchunks;
                ++slice;
            }
            t0 = c * chunk;
        }
    }
};
using TileWalk = TileWalkT<kTileRows>;

// Compression work items: (slice, segment of `seg` tokens), item = slice *
// nseg + c, walked like TileWalkT.  With a temporal delta whose chains restart
// every `dchunk` tokens (0: no delta), a segment that begins inside a chain
// needs the raw codes of the token before its first row: the walk then starts
// one tile early, at t_begin - ROWS, with a halo tile that is encoded but not
// stored.  `rem` is t0 modulo dchunk, kept by additions (one division per
// segment): row 0 of a tile with rem == 0 starts a chain.  dchunk and seg are
// multiples of 32 (ROWS divides both).
template <int ROWS>
struct SegWalk {
    int64_t slice, slices, dslice;
    int nseg, seg, tokens, c, dc, t0, dchunk, rem;
    __device__ SegWalk(int64_t first, int64_t step, int64_t slices_, int tokens_, int seg_, int dchunk_)
        : slices(slices_), seg(seg_), tokens(tokens_), dchunk(dchunk_) {
        nseg = (tokens_ + seg_ - 1) / seg_;
        slice = slices_;  // no work when there are no segments
        dslice = 0;
        c = dc = 0;
        if (nseg > 0) {
            slice = first / nseg;
            c = int(first - slice * nseg);
            dslice = step / nseg;
            dc = int(step - dslice * nseg);
        }
        enter();
    }
    __device__ __forceinline__ void enter() {  // the first tile of segment c
        t0 = c * seg;
        rem = dchunk > 0 ? t0 % dchunk : 0;
        if (rem != 0) {
            t0 -= ROWS;
            rem -= ROWS;
        }
    }
    __device__ __forceinline__ bool valid() const { return slice < slices; }
    __device__ __forceinline__ int t_begin() const { return c * seg; }
    __device__ __forceinline__ int t_end() const { return min(c * seg + seg, tokens); }
    __device__ __forceinline__ bool halo() const { return t0 < c * seg; }
    __device__ __forceinline__ bool chain_start() const { return rem == 0; }
    __device__ __forceinline__ void next() {
        t0 += ROWS;
        rem += ROWS;
        if (rem == dchunk) rem = 0;
        if (t0 >= t_end()) {
            slice += dslice;
            c += dc;
            if (c >= nseg) {
                c -= nseg;
                ++slice;
            }
            enter();
        }
    }
};

// ----------------------------------------------------------- row records

// Block codes <-> the row's idx bytes (coordinate i's field at bit i*b).
// NB = number of 8-blocks in the row (Dp / 8).  Words are little-endian.
template <int BITS, int NB>
struct RowPack {
    static constexpr int WORDS = NB * BITS / 4;  // 32-bit words per row
    __device__ static __forceinline__ void pack(const unsigned (&blk)[NB], unsigned (&w)[WORDS]) {
        if constexpr (BITS == 2) {
#pragma unroll
            for (int i = 0; i < WORDS; ++i) w[i] = blk[2 * i] | (blk[2 * i + 1] << 16);
        } else if constexpr (BITS == 4) {
#pragma unroll
            for (int i = 0; i < WORDS; ++i) w[i] = blk[i];
        } else {  // 24-bit blocks: 4 blocks -> 3 words
#pragma unroll
            for (int g = 0; g < NB / 4; ++g) {
                unsigned b0 = blk[4 * g], b1 = blk[4 * g + 1], b2 = blk[4 * g + 2], b3 = blk[4 * g + 3];
                w[3 * g] = b0 | (b1 << 24);
                w[3 * g + 1] = (b1 >> 8) | (b2 << 16);
                w[3 * g + 2] = (b2 >> 16) | (b3 << 8);
            }
        }
    }
    __device__ static __forceinline__ void unpack(const unsigned (&w)[WORDS], unsigned (&blk)[NB]) {
        if constexpr (BITS == 2) {
#pragma unroll
            for (int i = 0; i < WORDS; ++i) {
                blk[2 * i] = w[i] & 0xffffu;
                blk[2 * i + 1] = w[i] >> 16;
            }
        } else if constexpr (BITS == 4) {
#pragma unroll
            for (int i = 0; i < WORDS; ++i) blk[i] = w[i];
        } else {
#pragma unroll
            for (int g = 0; g < NB / 4; ++g) {
                unsigned w0 = w[3 * g], w1 = w[3 * g + 1], w2 = w[3 * g + 2];
                blk[4 * g] = w0 & 0xffffffu;
                blk[4 * g + 1] = (w0 >> 24) | ((w1 & 0xffffu) << 8);
                blk[4 * g + 2] = (w1 >> 16) | ((w2 & 0xffu) << 16);
                blk[4 * g + 3] = w2 >> 8;
            }
        }
    }
};

}  // namespace nq
