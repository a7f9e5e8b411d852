// nq_decode.cuh -- the decoding steps shared by the decompression and the
// round-trip kernels: block codes -> unscaled coordinates -> inverse Hadamard
// transform (textbook stage order), the RoPE re-apply, and the fp16 rows' way
// out (swizzled shared-memory tile, TMA tensor store), for the one-thread-per-
// row layout (32-row tiles) and the two-threads-per-row layout (16-row tiles).
#pragma once

#include "nq_internal.h"

namespace nq {

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// One record row -> unscaled, inverse-transformed coordinates (before the
// RoPE re-apply).  `stage` holds the 32-row record tile of the lane's warp.

// Block codes of a one-thread row -> x = H (r * sc), the first D entries
// meaningful.  cw: coset word (bit k = block k); scf: the 32-subgroup scales.
template <int D, int BITS>
__device__ __forceinline__ void row_decode_codes(const unsigned (&blk)[PaddedDim<D>::value / 8], unsigned cw,
                                                 const float (&scf)[PaddedDim<D>::value / 32],
                                                 float (&y)[PaddedDim<D>::value]) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    // unpack, unscale: y = (code - offset) * scale  (exact)
#pragma unroll
    for (int k = 0; k < NB; ++k) unscale_block<BITS>(blk[k], (cw >> k) & 1u, scf[k / 4], &y[8 * k]);
    // inverse Hadamard: x = H (r * sc)
    fwht<DP>(y);
}

// Rotate the pairs (2q, 2q + D/2) and (2q + 1, 2q + 1 + D/2) by +angle;
// cs = (cos, sin) of both pairs.
template <int D, int N>
__device__ __forceinline__ void rope_apply_pairs(float (&y)[N], int q, float4 cs) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int j = 2 * q + p;
        const float c = p ? cs.z : cs.x, s = p ? cs.w : cs.y;
        const float a = y[j], b = y[j + D / 2];
        y[j] = __fmaf_rn(a, c, -__fmul_rn(b, s));
        y[j + D / 2] = __fmaf_rn(b, c, __fmul_rn(a, s));
    }
}

// fp16 rows -> swizzled shared-memory tile -> TMA tensor store of 32 rows
// (the map clips rows past the slice end and columns past head_dim).  PENDING
// = stores of the warp's other output tiles that may still be reading.
template <int D, int PENDING, int N>
__device__ __forceinline__ void store_rows(const float (&y)[N], uint32_t ob, int lane, const CUtensorMap* map,
                                           int t0, int slice) {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(PENDING) : "memory");  // ob is free
    __syncwarp();
#pragma unroll
    for (int q = 0; q < D / 8; ++q) sts128(ob + swz(lane, q), f_to_h8(&y[8 * q]));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, ob, 0, t0, slice);
        if (D > 64) tma_store_3d(map, ob + 4096, 64, t0, slice);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// The inverse rotation of the thread's unscaled slots (two-thread layout), the
// stages as pair_decode_codes below describes them.
template <int D>
__device__ __forceinline__ void pair_inverse_rotation(float (&y)[D / 2], float sgn) {
    using PM = PairMap<D>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
#pragma unroll
    for (int h = 1; h < Q; h *= 2) fwht_stage<HALF>(y, h);
    stage_signed<HALF>(y, sgn);
    stage_exchange<HALF>(y);
}

// The thread's half of a two-thread row: block codes (its NBT blocks, coset
// bits cwl with bit k = block k, scales of its 32-subgroups) -> coordinates
// in PairMap slots.  The inverse transform (textbook order) runs its bits
// below DP/4 in-thread, bit DP/4 in-thread with a sign that leaves the odd
// thread's slot halves exchanged, and bit DP/2 as one symmetric shuffle
// exchange; the odd thread's upper slots come out negated.
template <int D, int BITS>
__device__ __forceinline__ void pair_decode_codes(const unsigned (&blk)[D / 16], unsigned cwl,
                                                  const float (&scf)[D / 64], float sgn, float (&y)[D / 2]) {
    constexpr int NBT = PairMap<D>::NBT;
#pragma unroll
    for (int k = 0; k < NBT; ++k) unscale_block<BITS>(blk[k], (cwl >> k) & 1u, scf[(8 * k) / 32], &y[8 * k]);
    pair_inverse_rotation<D>(y, sgn);
}

// RoPE re-apply of slot pairs (2qq, 2qq + Q) and (2qq + 1, 2qq + 1 + Q) (the
// pairs (i, i + D/2) of the row); cs = (cos, sin) of both pairs.  The odd
// thread's upper slots are negated, so its sin changes sign.
template <int D>
__device__ __forceinline__ void pair_rope_apply(float (&y)[D / 2], int qq, float4 cs, float sgn) {
    constexpr int Q = PairMap<D>::Q;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int l = 2 * qq + p;
        const float c = p ? cs.z : cs.x;
        const float s = __fmul_rn(p ? cs.w : cs.y, sgn);
        const float a = y[l], b = y[l + Q];
        y[l] = __fmaf_rn(a, c, -__fmul_rn(b, s));
        y[l + Q] = __fmaf_rn(b, c, __fmul_rn(a, s));
    }
}

// RoPE re-apply on a two-thread row of head_dim 96 (padded to 128), whose
// pairs (i, i + 48) are not slot pairs.  In PairMap<128> thread 0 holds
// global chunks 0-3 and 8-11, thread 1 chunks 4-7 and the zero padding 12-15;
// chunk g pairs with g + 6 (g < 6).  Thread 0's pairs (2, 8) and (3, 9) are
// local; the others cross threads, so four symmetric exchanges of one
// 8-coordinate chunk bring every partner: (0|6), (1|7), (10|4), (11|5) as
// (thread 0 sends | thread 1 sends).  cs: the token's table column.
__device__ __forceinline__ void pair96_rope_apply(float (&y)[64], int hf, const float4* cs, int tokens) {
    // slot chunk sent in exchange e by thread 0 / thread 1, and the own slot chunk it completes
    constexpr int SEND0[4] = {0, 1, 6, 7}, SEND1[4] = {2, 3, 0, 1};
    float part[4][8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float v = hf ? y[8 * SEND1[e] + j] : y[8 * SEND0[e] + j];
            part[e][j] = __shfl_xor_sync(kFull, v, 1);
        }
    }
    // thread 0's local pairs use the values before rotation
    float loc[2][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        loc[0][j] = y[8 * 2 + j];  // chunk 2 (partner of chunk 8, slot 4)
        loc[1][j] = y[8 * 3 + j];  // chunk 3 (partner of chunk 9, slot 5)
    }
    // rotate member `own` (lower: a of (a, b), else b) of the 8 pairs starting at pair index p0
    auto rot = [&](float* own, const float* other, int p0, bool lower) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const float4 v = __ldg(cs + int64_t(p0 / 2 + qq) * tokens);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float c = p ? v.z : v.x, sn = p ? v.w : v.y;
                const int j = 2 * qq + p;
                const float o = own[j], x = other[j];
                own[j] = lower ? __fmaf_rn(o, c, -__fmul_rn(x, sn)) : __fmaf_rn(o, c, __fmul_rn(x, sn));
            }
        }
    };
    if (hf == 0) {
        float c4[8], c5[8];  // chunks 8 and 9 before rotation
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c4[j] = y[8 * 4 + j];
            c5[j] = y[8 * 5 + j];
        }
        rot(&y[0], part[0], 0, true);        // chunk 0 with chunk 6
        rot(&y[8], part[1], 8, true);        // chunk 1 with chunk 7
        rot(&y[16], c4, 16, true);           // chunk 2 with chunk 8
        rot(&y[24], c5, 24, true);           // chunk 3 with chunk 9
        rot(&y[32], loc[0], 16, false);      // chunk 8 with chunk 2
        rot(&y[40], loc[1], 24, false);      // chunk 9 with chunk 3
        rot(&y[48], part[2], 32, false);     // chunk 10 with chunk 4
        rot(&y[56], part[3], 40, false);     // chunk 11 with chunk 5
    } else {
        rot(&y[0], part[2], 32, true);       // chunk 4 with chunk 10
        rot(&y[8], part[3], 40, true);       // chunk 5 with chunk 11
        rot(&y[16], part[0], 0, false);      // chunk 6 with chunk 0
        rot(&y[24], part[1], 8, false);      // chunk 7 with chunk 1
    }
}

// fp16 rows of a 16-row tile -> swizzled shared-memory tile -> TMA tensor
// store (the odd thread's negated slots get their sign bits flipped back).
// PENDING = stores of the warp's other output tiles that may still be reading.
template <int D, int PENDING>
__device__ __forceinline__ void pair_store_rows(const float (&y)[D / 2], uint32_t ob, int r, int hf, int lane,
                                                const CUtensorMap* map, int t0, int slice) {
    using PM = PairMap<D>;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    const unsigned negbits = hf ? 0x80008000u : 0u;
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(PENDING) : "memory");  // ob is free
    __syncwarp();
    const PairTileAddr<D> ta(ob, r, hf);
#pragma unroll
    for (int c = 0; c < NBT; ++c) {
        uint4 v = f_to_h8(&y[8 * c]);
        if (8 * c >= Q) {
            v.x ^= negbits;
            v.y ^= negbits;
            v.z ^= negbits;
            v.w ^= negbits;
        }
        sts128(ta(c), v);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, ob, 0, t0, slice);
        if (D > 64) tma_store_3d(map, ob + 2048, 64, t0, slice);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

}  // namespace nq
