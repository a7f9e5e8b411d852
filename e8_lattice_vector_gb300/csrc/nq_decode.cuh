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

// The thread's half of a two-thread row: block codes (its NBT blocks, coset
// bits cwl with bit k = block k, scales of its 32-subgroups) -> coordinates
// in PairMap slots.  The inverse transform (textbook order) runs its bits
// below DP/4 in-thread, bit DP/4 in-thread with a sign that leaves the odd
// thread's slot halves exchanged, and bit DP/2 as one symmetric shuffle
// exchange; the odd thread's upper slots come out negated.
template <int D, int BITS>
__device__ __forceinline__ void pair_decode_codes(const unsigned (&blk)[D / 16], unsigned cwl,
                                                  const float (&scf)[D / 64], float sgn, float (&y)[D / 2]) {
    using PM = PairMap<D>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
#pragma unroll
    for (int k = 0; k < NBT; ++k) unscale_block<BITS>(blk[k], (cwl >> k) & 1u, scf[(8 * k) / 32], &y[8 * k]);
#pragma unroll
    for (int h = 1; h < Q; h *= 2) fwht_stage<HALF>(y, h);
    stage_signed<HALF>(y, sgn);
    stage_exchange<HALF>(y);
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
#pragma unroll
    for (int c = 0; c < NBT; ++c) {
        uint4 v = f_to_h8(&y[8 * c]);
        if (8 * c >= Q) {
            v.x ^= negbits;
            v.y ^= negbits;
            v.z ^= negbits;
            v.w ^= negbits;
        }
        sts128(ob + swz16(r, PM::chunk(hf, c)), v);
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
