// nq_chain.cuh -- the temporal delta's running sums for decompression in
// parallel, with no waiting between warps.
//
// A record tile's rows are delta-coded against their predecessors along the
// slice.  The decompressors walk the tiles of a chain in runs ("groups") of up
// to 32 consecutive tiles, a warp per group, carrying the running sum
// (field-wise modulo 2^b; coset words by exclusive or) from tile to tile in
// registers.  A group that does not start its chain (chains longer than 32
// tiles, up to the method's single chain per slice) needs the sum of every
// stored row of its chain before it.  Two light passes give it that before the
// decoder runs:
//   1. group totals: a block per group sums its tiles' rows (column sums);
//   2. chain scan: a warp per chain scans its groups' totals into, per group,
//      the sum of the chain's groups before it.
// The states live in the caller's workspace: one slot of slot_words words per
// group and pass, holding the idx row words (packed as in a record row) and a
// coset word.
#pragma once

#include "nq_internal.h"

namespace nq {

template <int BITS>
struct DeltaUnit;
template <>
struct DeltaUnit<2> {  // one word, 16 fields
    static constexpr int U = 1, NV = 1;
    __device__ static void load(uint32_t a, unsigned (&v)[NV]) { v[0] = lds32(a); }
    __device__ static void store(uint32_t a, const unsigned (&v)[NV]) { sts32(a, v[0]); }
    __device__ static unsigned add(unsigned a, unsigned b) { return swar_add_word2(a, b); }
};
template <>
struct DeltaUnit<4> {  // one word = one block of 8 fields
    static constexpr int U = 1, NV = 1;
    __device__ static void load(uint32_t a, unsigned (&v)[NV]) { v[0] = lds32(a); }
    __device__ static void store(uint32_t a, const unsigned (&v)[NV]) { sts32(a, v[0]); }
    __device__ static unsigned add(unsigned a, unsigned b) { return swar_add<4>(a, b); }
};
template <>
struct DeltaUnit<3> {  // three words = four 24-bit blocks (fields straddle the words)
    static constexpr int U = 3, NV = 4;
    __device__ static void load(uint32_t a, unsigned (&v)[NV]) {
        const unsigned w0 = lds32(a), w1 = lds32(a + 4), w2 = lds32(a + 8);
        v[0] = w0 & 0xffffffu;
        v[1] = (w0 >> 24) | ((w1 & 0xffffu) << 8);
        v[2] = (w1 >> 16) | ((w2 & 0xffu) << 16);
        v[3] = w2 >> 8;
    }
    __device__ static void store(uint32_t a, const unsigned (&v)[NV]) {
        sts32(a, v[0] | (v[1] << 24));
        sts32(a + 4, (v[1] >> 8) | (v[2] << 16));
        sts32(a + 8, (v[2] >> 16) | (v[3] << 8));
    }
    __device__ static unsigned add(unsigned a, unsigned b) { return swar_add<3>(a, b); }
};

// Load one column unit of a state slot (its U packed words) as NV field
// groups, and store it back.
template <int BITS>
__device__ __forceinline__ void unit_load(const uint32_t* src, unsigned (&v)[DeltaUnit<BITS>::NV]) {
    if constexpr (BITS == 3) {
        const unsigned w0 = src[0], w1 = src[1], w2 = src[2];
        v[0] = w0 & 0xffffffu;
        v[1] = (w0 >> 24) | ((w1 & 0xffffu) << 8);
        v[2] = (w1 >> 16) | ((w2 & 0xffu) << 16);
        v[3] = w2 >> 8;
    } else {
        v[0] = src[0];
    }
}
template <int BITS>
__device__ __forceinline__ void unit_store(uint32_t* dst, const unsigned (&v)[DeltaUnit<BITS>::NV]) {
    if constexpr (BITS == 3) {
        dst[0] = v[0] | (v[1] << 24);
        dst[1] = (v[1] >> 8) | (v[2] << 16);
        dst[2] = (v[2] >> 16) | (v[3] << 8);
    } else {
        dst[0] = v[0];
    }
}

// Group work items of a delta-coded tensor: G = (unit * cps + c) * gpc + q is
// group q of chain c of a unit (a slice, or a block's group of slices), tiles
// [j0, j1); walked grid-stride, empty groups (past a short last chain)
// skipped.  One division per group.
template <int R>
struct GroupWalk {
    static constexpr bool kGroups = true;
    ChainGeom geo;
    uint64_t G, step, total, slice;  // slice: the unit (a slice, or a block's group of slices)
    uint32_t c, q, j0, j1, j;
    int t0;
    __device__ GroupWalk(uint64_t first, uint64_t step_, uint64_t units, const ChainGeom& g)
        : geo(g), G(first), step(step_), total(units * g.cps * g.gpc) {
        enter();
    }
    __device__ __forceinline__ void enter() {
        const uint64_t per = uint64_t(geo.cps) * geo.gpc;
        for (; G < total; G += step) {
            slice = G / per;
            const uint32_t rest = uint32_t(G - slice * per);
            c = rest / geo.gpc;
            q = rest - c * geo.gpc;
            j0 = c * geo.tpc + 32u * q;
            j1 = min(min(j0 + 32u, (c + 1u) * geo.tpc), geo.tiles);
            if (j0 < j1) break;
        }
        j = j0;
        t0 = int(j) * R;
    }
    __device__ __forceinline__ bool valid() const { return G < total; }
    __device__ __forceinline__ bool group_start() const { return j == j0; }
    // the group's index in the slice-level numbering, for slice s of the unit
    __device__ __forceinline__ uint64_t slice_group(uint64_t s) const { return (s * geo.cps + c) * geo.gpc + q; }
    __device__ __forceinline__ void next() {
        ++j;
        t0 += R;
        if (j >= j1) {
            G += step;
            enter();
        }
    }
};

// Pass 1: group totals (every group but the last of its chain: no starting
// sum includes that one).  A block of kGroupWarps warps per group: warp w sums
// tiles j0 + w, j0 + w + kGroupWarps, ... of the group (lane (u, sg) takes
// column unit u of the rows of segment sg of each tile, the split of the
// decoder's tile scan, and reduces over the segments with xor shuffles); the
// warps' partial sums meet in shared memory.  Spreading a group over the
// block keeps every warp's loads in flight at once (a warp walking all 32
// tiles of a group waited on memory tile after tile when the groups were
// few).
constexpr int kGroupWarps = 8;

template <int BITS, int RB, int R>
__global__ void __launch_bounds__(kGroupWarps * 32)
    delta_group_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset, int64_t slices,
                       int tpad, ChainGeom geo, uint32_t* __restrict__ gsum, int slot_words) {
    using DU = DeltaUnit<BITS>;
    constexpr int NV = DU::NV;
    constexpr int NU = RB / (4 * DU::U);
    constexpr int SEGS = 32 / NU;
    constexpr int RPS = R / SEGS;
    constexpr int CW = RB / 4;
    static_assert(NU * SEGS == 32 && RPS * SEGS == R, "tile split");
    __shared__ unsigned part[kGroupWarps][NU][NV];
    __shared__ unsigned part_c[kGroupWarps];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int u = lane % NU, sg = lane / NU;
    const uint64_t per = uint64_t(geo.cps) * geo.gpc;
    const uint64_t total = uint64_t(slices) * per;
    for (uint64_t G = blockIdx.x; G < total; G += gridDim.x) {
        const uint64_t slice = G / per;
        const uint32_t rest = uint32_t(G - slice * per);
        const uint32_t c = rest / geo.gpc;
        const uint32_t q = rest - c * geo.gpc;
        const uint32_t j0 = c * geo.tpc + 32u * q;
        const uint32_t j1 = min(min(j0 + 32u, (c + 1u) * geo.tpc), geo.tiles);
        // past a short last chain, or the last group of its chain, whose total no
        // starting sum needs (the same in the whole block)
        if (j0 >= j1 || j1 == min((c + 1u) * geo.tpc, geo.tiles)) continue;
        unsigned run[NV], run_c = 0u;
#pragma unroll
        for (int n = 0; n < NV; ++n) run[n] = 0u;
#pragma unroll 4
        for (uint32_t j = j0 + wid; j < j1; j += kGroupWarps) {
            const int64_t row0 = int64_t(slice) * tpad + int64_t(j) * R;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(idx + (row0 + sg * RPS) * RB) + DU::U * u;
#pragma unroll
            for (int i = 0; i < RPS; ++i) {
                unsigned v[NV];
                unit_load<BITS>(src + i * (RB / 4), v);
#pragma unroll
                for (int n = 0; n < NV; ++n) run[n] = DU::add(run[n], v[n]);
            }
            if (coset != nullptr && lane < R) run_c ^= unsigned(coset[row0 + lane]);
        }
#pragma unroll
        for (int d = NU; d < 32; d *= 2)
#pragma unroll
            for (int n = 0; n < NV; ++n) run[n] = DU::add(run[n], __shfl_xor_sync(kFull, run[n], d));
        if (coset != nullptr) {
#pragma unroll
            for (int d = 1; d < 32; d *= 2) run_c ^= __shfl_xor_sync(kFull, run_c, d);
        }
        if (sg == 0)
#pragma unroll
            for (int n = 0; n < NV; ++n) part[wid][u][n] = run[n];
        if (lane == 0) part_c[wid] = run_c;
        __syncthreads();
        if (wid == 0) {
            uint32_t* p = gsum + size_t(G) * slot_words;
            if (lane < NU) {
                unsigned t[NV];
#pragma unroll
                for (int n = 0; n < NV; ++n) t[n] = part[0][lane][n];
#pragma unroll
                for (int w = 1; w < kGroupWarps; ++w)
#pragma unroll
                    for (int n = 0; n < NV; ++n) t[n] = DU::add(t[n], part[w][lane][n]);
                unit_store<BITS>(p + DU::U * lane, t);
            }
            if (coset != nullptr && lane == 0) {
                unsigned t = 0u;
#pragma unroll
                for (int w = 0; w < kGroupWarps; ++w) t ^= part_c[w];
                p[CW] = t;
            }
        }
        __syncthreads();  // the partial sums are read before the next group's
    }
}

// Pass 2: chain scan of the group totals.  A warp per chain, 32 groups at a
// time: lane l takes group 32 k + l, an inclusive warp scan per column unit,
// then the exclusive sums plus the chain's running total are written.
template <int BITS, int RB>
__global__ void __launch_bounds__(256)
    delta_chain_kernel(int64_t slices, ChainGeom geo, const uint32_t* __restrict__ gsum,
                       uint32_t* __restrict__ gexcl, int slot_words, bool has_coset) {
    using DU = DeltaUnit<BITS>;
    constexpr int NV = DU::NV;
    constexpr int NU = RB / (4 * DU::U);
    constexpr int CW = RB / 4;
    const int lane = threadIdx.x & 31;
    const uint64_t chains = uint64_t(slices) * geo.cps;
    const uint64_t nwarps = (uint64_t(gridDim.x) * blockDim.x) >> 5;
    for (uint64_t ch = (uint64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; ch < chains; ch += nwarps) {
        const uint32_t slice = uint32_t(ch / geo.cps);
        const uint32_t c = uint32_t(ch - uint64_t(slice) * geo.cps);
        const uint32_t jn = min(geo.tpc, geo.tiles - c * geo.tpc);  // tiles of this chain
        const uint32_t ng = (jn + 31u) / 32u;                           // its groups
        unsigned carry[NU][NV], carry_c = 0u;
#pragma unroll
        for (int x = 0; x < NU; ++x)
#pragma unroll
            for (int n = 0; n < NV; ++n) carry[x][n] = 0u;
        for (uint32_t q0 = 0; q0 < ng; q0 += 32u) {
            const uint32_t q = q0 + lane;
            const bool ok = q < ng;
            const bool has_total = q + 1u < ng;  // the chain's last group has none (nothing needs it)
            const uint32_t* src = gsum + size_t(ch * geo.gpc + (has_total ? q : 0u)) * slot_words;
            unsigned v[NU][NV], vc = 0u;
#pragma unroll
            for (int x = 0; x < NU; ++x) {
                unit_load<BITS>(src + DU::U * x, v[x]);
                if (!has_total)
#pragma unroll
                    for (int n = 0; n < NV; ++n) v[x][n] = 0u;
            }
            if (has_coset && has_total) vc = src[CW];
#pragma unroll
            for (int d = 1; d < 32; d *= 2) {
#pragma unroll
                for (int x = 0; x < NU; ++x)
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        const unsigned t = __shfl_up_sync(kFull, v[x][n], d);
                        if (lane >= d) v[x][n] = DU::add(v[x][n], t);
                    }
                const unsigned tc = __shfl_up_sync(kFull, vc, d);
                if (lane >= d) vc ^= tc;
            }
            uint32_t* dst = gexcl + size_t(ch * geo.gpc + (ok ? q : 0u)) * slot_words;
#pragma unroll
            for (int x = 0; x < NU; ++x) {
                unsigned e[NV];
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    e[n] = __shfl_up_sync(kFull, v[x][n], 1);
                    if (lane == 0) e[n] = 0u;
                    e[n] = DU::add(e[n], carry[x][n]);
                }
                if (ok) unit_store<BITS>(dst + DU::U * x, e);
            }
            unsigned ec = __shfl_up_sync(kFull, vc, 1);
            if (lane == 0) ec = 0u;
            if (has_coset && ok) dst[CW] = ec ^ carry_c;
#pragma unroll
            for (int x = 0; x < NU; ++x)
#pragma unroll
                for (int n = 0; n < NV; ++n) carry[x][n] = DU::add(carry[x][n], __shfl_sync(kFull, v[x][n], 31));
            carry_c ^= __shfl_sync(kFull, vc, 31);
        }
    }
}

// The starting sum of a group (slice-level index G) for the lane's column unit
// u (NV field groups into carry[0..NV)) and its coset word; carry_c is the
// full coset word.
template <int BITS, int RB>
__device__ __forceinline__ void load_group_carry(const ChainState& cs, uint64_t G, int u, unsigned* carry,
                                                 unsigned& carry_c, bool has_coset) {
    using DU = DeltaUnit<BITS>;
    constexpr int CW = RB / 4;
    const uint32_t* p = cs.gexcl + size_t(G) * cs.slot_words;
    unit_load<BITS>(p + DU::U * u, *reinterpret_cast<unsigned(*)[DU::NV]>(carry));
    carry_c = has_coset ? p[CW] : 0u;
}

// The same for the column layout of the three-bit 32-row decoders (one block
// code per lane): the 24-bit code of block column c, bytes 3c..3c+2 of the
// slot's packed row (the byte above it is the next code's; the sums ignore it).
__device__ __forceinline__ void load_group_carry24(const ChainState& cs, uint64_t G, int c, unsigned& carry,
                                                   unsigned& carry_c, bool has_coset) {
    constexpr int CW = 48 / 4;
    const uint32_t* p = cs.gexcl + size_t(G) * cs.slot_words;
    const int w = (3 * c) >> 2;  // c = 15: the second word is the coset word (in the slot)
    carry = __byte_perm(p[w], p[w + 1], 0x3210u + 0x1111u * ((3u * uint32_t(c)) & 3u));
    carry_c = has_coset ? p[CW] : 0u;
}

}  // namespace nq
