// nq_encode.cuh -- the encoding steps shared by the compression and the
// round-trip kernels (two threads per row): tile loads, the RoPE removal, and
// per row the zero-padded Hadamard rotation, the group scales and the E8 block
// codes.
#pragma once

#include "nq_internal.h"

namespace nq {

// Scaled coordinates u = y * inv of 8-block k of the thread's coordinates
// (packed pairs j, j + 4, as the E8 search and the transform use them).
template <int N>
__device__ __forceinline__ void row_block_u(const float (&y)[N], float inv, int k, float (&u)[8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 p = __fmul2_rn(make_float2(y[8 * k + j], y[8 * k + j + 4]), make_float2(inv, inv));
        u[j] = p.x;
        u[j + 4] = p.y;
    }
}

// With the two-thread layout: slots at or above Q hold the odd thread's
// negated coordinates, so their reciprocal scale carries the thread's sign.
template <int Q, int N, int NS>
__device__ __forceinline__ void pair_block_u(const float (&y)[N], const float (&inv)[NS], float sgn, int k,
                                             float (&u)[8]) {
    const float ik = (8 * k >= Q) ? __fmul_rn(inv[(8 * k) / 32], sgn) : inv[(8 * k) / 32];
    row_block_u(y, ik, k, u);
}

// Copy the fp16 rows of a 16-row tile into a stage (rows past the slice are
// zeros).
template <int D>
__device__ __forceinline__ void load_pair_tile(const __half* __restrict__ x, int64_t slice, int t0, int tokens,
                                               uint32_t stage, int lane) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    const int nvalid = min(kPairRows, tokens - t0);
    const __half* base = x + (slice * tokens + min(t0, tokens - 1)) * int64_t(D);
    if constexpr (CPR == 8 || CPR == 16) {
        if (nvalid == kPairRows) {  // full tile (warp-uniform): no bounds, swizzle by parts
            // copy i of the lane is chunk g = lane + 32 i: row r = r0 + (32 / CPR) i,
            // column c = lane % CPR; (r & 7) = r0 + (32 / CPR) (i % (8 CPR / 32))
            // with disjoint bits, so the swizzle term is x0 ^ that step.
            constexpr int RS = 32 / CPR;   // rows per copy step
            constexpr int PER = 8 / RS;    // steps until (r & 7) repeats
            const int c = lane % CPR, r0 = lane / CPR;
            const uint32_t d0 = stage + ((c >> 3) << 11) + (r0 << 7);
            const uint32_t x0 = uint32_t((c & 7) ^ r0) << 4;
#pragma unroll
            for (int i = 0; i < CPR / 2; ++i)
                cp_async16(d0 + ((RS * i) << 7) + (x0 ^ (uint32_t(RS * (i % PER)) << 4)), base + 8 * (lane + 32 * i), 16);
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < CPR / 2; ++i) {  // 16 rows * CPR chunks / 32 lanes
        const int g = lane + 32 * i;
        const int r = g / CPR;
        const int c = g - r * CPR;
        const bool ok = r < nvalid;
        cp_async16(stage + swz16(r, c), ok ? base + 8 * g : base, ok ? 16 : 0);
    }
}

// Rotation and group scales of the thread's half of a row (two-thread
// layout): the fp16 scale bits sc and reciprocals inv of its 32-subgroups;
// returns whether every scaled coordinate is inside the box (the fast
// decoder's condition).
template <int D, int BITS>
__device__ __forceinline__ bool pair_rotate_scale(float (&y)[D / 2], float sgn, int group,
                                                  unsigned short (&sc)[D / 64], float (&inv)[D / 64]) {
    constexpr int DP = D;
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NSUB = HALF / 32;  // 32-coordinate subgroups per thread
    using C = Code<BITS>;
    constexpr float STEP = float(DP) * C::H;
    const int span = group / 32;  // 32-coordinate subgroups per scale group

    // ---- Hadamard rotation, compression order: bits below DP/4 in-thread,
    //      bit DP/2 in-thread (signed), bit DP/4 by exchange
#pragma unroll
    for (int h = 1; h < Q; h *= 2) fwht_stage<HALF, 4>(y, h);
    stage_signed<HALF, 4>(y, sgn);
    stage_exchange<HALF, 4>(y);

    // ---- group absmax -> fp16 scale -> reciprocal (per 32-subgroup)
    float amax[NSUB];
#pragma unroll
    for (int s = 0; s < NSUB; ++s) {
        float m = 0.0f;
#pragma unroll
        for (int j = 32 * s; j < 32 * s + 32; j += 2) m = fmax3(m, fabsf(y[j]), fabsf(y[j + 1]));
        amax[s] = m;
    }
    if (NSUB == 2 && span >= 2) amax[0] = amax[1] = fmaxf(amax[0], amax[1]);
    if (span > NSUB) {
        const float o = __shfl_xor_sync(kFull, amax[0], 1);
#pragma unroll
        for (int s = 0; s < NSUB; ++s) amax[s] = fmaxf(amax[s], o);
    }
    bool fast = true;
    if (NSUB == 2 && span >= 2) {  // one scale group covers both subgroups: one scale, one reciprocal
        const unsigned short v = group_scale(amax[0], STEP, 1.0f / STEP);
        const float iv = v ? __frcp_rn(__fmul_rn(__half2float(__ushort_as_half(v)), float(DP))) : 0.0f;
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
            sc[s] = v;
            inv[s] = iv;
        }
        fast = __fmul_rn(amax[0], iv) < C::H;
    } else {
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
            sc[s] = group_scale(amax[s], STEP, 1.0f / STEP);
            const float scf = __half2float(__ushort_as_half(sc[s]));
            inv[s] = sc[s] ? __frcp_rn(__fmul_rn(scf, float(DP))) : 0.0f;
            fast = fast && (__fmul_rn(amax[s], inv[s]) < C::H);
        }
    }

    return fast;
}

// Rotation, group scales and E8 codes of the thread's half of a row
// (two-thread layout): block codes blk (the thread's NBT blocks), their coset
// bits cwl (bit k = block k) and the fp16 scale bits of its 32-subgroups.
template <int D, int BITS, bool STRICT>
__device__ __forceinline__ void pair_encode_codes(float (&y)[D / 2], int hf, float sgn, int group,
                                                  unsigned (&blk)[D / 16], unsigned& cwl,
                                                  unsigned short (&sc)[D / 64]) {
    using PM = PairMap<D>;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    float inv[D / 64];
    const bool fast = pair_rotate_scale<D, BITS>(y, sgn, group, sc, inv);

    // ---- E8 nearest point per 8-block -> block codes
    // Fast path for every block without a branch, then the general path for
    // the blocks it declined (rare), so consecutive blocks can overlap.
    unsigned declined = 0;
    cwl = 0;
#pragma unroll
    for (int k = 0; k < NBT; ++k) {
        float u[8];
        pair_block_u<Q>(y, inv, sgn, k, u);
        unsigned c;
        const bool ok = e8_fast<BITS, STRICT>(u, blk[k], c);
        cwl |= c << k;
        declined |= unsigned(!ok) << k;
    }
    if (!fast) declined = (1u << NBT) - 1u;
    if (__any_sync(kFull, declined != 0u)) {  // warp-uniform: most tiles of most warps skip this
#pragma unroll
        for (int k = 0; k < NBT; ++k) {
            if (!((declined >> k) & 1u)) continue;
            float u[8];
            pair_block_u<Q>(y, inv, sgn, k, u);
            const uint2 res = e8_slow<BITS, STRICT>(make_float4(u[0], u[1], u[2], u[3]),
                                                    make_float4(u[4], u[5], u[6], u[7]));
            blk[k] = res.x;
            cwl = (cwl & ~(1u << k)) | (res.y << k);
        }
    }
}

// ------------------------------------ keys: the RoPE table shared by a block
//
// A block of WARPS warps processes the same 16-token tile of WARPS consecutive
// slices (warp w: slice WARPS*g + w).  The tile's RoPE table rows (head_dim/4
// planes x 16 tokens x 16 bytes) are staged once per block, next to the
// warps' fp16 tiles, in a STAGES-deep ring filled by cp.async; one block
// barrier per tile orders the refills.  Each key row then reads 512 bytes of
// table from shared memory instead of L2.
template <int D, int WARPS, int STAGES>
struct RopeRing {
    static constexpr int THREADS = WARPS * 32;
    static constexpr int TABLE = D * 4 * kPairRows;  // head_dim/4 planes x 16 tokens x 16 B
    static constexpr int BYTES = TABLE + WARPS * kPairTileBytes;
    static constexpr int SMEM = STAGES * BYTES + 1024;
};

// table position of (plane q, tile row rr): the odd thread's planes (q >= D/8)
// are shifted by 4 rows so the two threads of a row hit different banks
template <int D>
__device__ __forceinline__ uint32_t rope_slot(int q, int rr) {
    return uint32_t((q * kPairRows + (rr ^ (q >= D / 8 ? 4 : 0))) * 16);
}

// The block's table entry of (plane q, tile row rr) as (cos, sin, cos, sin).
template <int D>
__device__ __forceinline__ float4 rope_tile_entry(uint32_t stage, int q, int rr) {
    const uint4 raw = lds128(stage + rope_slot<D>(q, rr));
    return make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                       __uint_as_float(raw.w));
}

// RoPE removal of one member of two consecutive pairs given the raw partner
// values: own = (x_i, x_i+1) of the lower members (lower) or (x_j, x_j+1) of
// the upper ones, partner = the other members; cs = (cos, sin) of both pairs.
__device__ __forceinline__ void rope_remove_member(float* own, const float* partner, float4 cs, bool lower) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const float c = p ? cs.z : cs.x, sn = p ? cs.w : cs.y;
        const float ps = __fmul_rn(partner[p], sn);
        own[p] = __fmaf_rn(own[p], c, lower ? ps : -ps);
    }
}

// RoPE removal on a two-thread row whose pairs (i, i + D/2) are not slot
// pairs (head_dim 96 in PairMap<128>): every own coordinate below D is
// rotated against its partner's raw value, read from the fp16 tile in shared
// memory (chunk g pairs with g + D/16).  cs: the token's table column.
template <int D, int N>
__device__ __forceinline__ void pair_rope_remove_from_tile(float (&y)[N], int hf, uint32_t stage, int r,
                                                           const float4* cs, int tokens) {
    using PM = PairMap<2 * N>;
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
        const int gc = PM::chunk(hf, c);
        if (gc < D / 8) {
            const bool lower = gc < D / 16;  // member i of the pair (else i + D/2)
            float xp[8];
            h8_to_f(lds128(stage + swz16(r, lower ? gc + D / 16 : gc - D / 16)), xp);
            const int q0 = 4 * (lower ? gc : gc - D / 16);  // table plane of the chunk's first pair
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
                rope_remove_member(&y[8 * c + 2 * qq], &xp[2 * qq], __ldg(cs + int64_t(q0 + qq) * tokens), lower);
        }
    }
}

// The same on a two-thread row before the rotation: the pairs (i, i + D/2)
// are slots (l, l + Q), l = 2qq and 2qq + 1.
template <int D>
__device__ __forceinline__ void pair_rope_remove(float (&y)[D / 2], int qq, float4 cs) {
    constexpr int Q = PairMap<D>::Q;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int l = 2 * qq + p;
        const float c = p ? cs.z : cs.x, sn = p ? cs.w : cs.y;
        const float a = y[l], b = y[l + Q];
        y[l] = __fmaf_rn(a, c, __fmul_rn(b, sn));
        y[l + Q] = __fmaf_rn(b, c, -__fmul_rn(a, sn));
    }
}

}  // namespace nq
