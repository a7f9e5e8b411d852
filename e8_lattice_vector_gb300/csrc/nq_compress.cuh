// nq_compress.cuh -- fused compression kernels: fp16 row -> RoPE removal (keys)
// -> zero-padded Hadamard -> group scale -> E8 nearest point -> b-bit codes ->
// temporal delta -> idx / coset / scale sections.
//
// Layout of the work: two threads per token row (lanes 2r and 2r+1 of a warp
// share row r of a 16-token tile of one (layer, batch, head) slice), so a
// thread holds 64 of the padded row's 128 coordinates (32 of 64) and the
// kernels fit 128 registers.  Tiles stream through a 3-stage shared-memory
// ring per warp, filled by coalesced 16-byte cp.async copies two tiles ahead;
// keys of head_dim 64 / 128 instead run in blocks of warps that share the
// tile's RoPE table rows in shared memory.  The previous token's codes for
// the delta come from the lanes two below.  Warps take work items (slice,
// chunk of delta_chunk tokens, or 16 tokens without delta) round-robin.
#pragma once

#include <type_traits>

#include "nq_encode.cuh"

namespace nq {

// ------------------------------------------------------- two threads per row
//
// Lanes 2r and 2r+1 share token row r of a 16-row tile (PairMap of the padded
// dimension; head_dim 96 adds zero chunks 12..15): each thread holds 64 (or
// 32) coordinates, so the kernel fits 128 registers and two blocks per SM.  The Hadamard transform runs in the
// compression stage order; its stage on bit DP/2 is in-thread with a sign
// that leaves the odd thread's slot halves exchanged, so the last stage
// (bit DP/4) is one symmetric shuffle exchange.  Afterwards thread hf holds
// coordinates [hf*DP/2, (hf+1)*DP/2) in natural order, the odd thread's upper
// quarter negated, which is folded into the sign of its reciprocal scale.
constexpr int kPairStages = 3;
constexpr int kPairCompressSmem = kWarpsPerBlock * kPairStages * kPairTileBytes;

// The walk of a launch without a temporal delta: every 16-token tile is a work
// item, no tile starts a chain and none is a halo.  (A launch with a delta
// walks segments of a chain, each after a one-tile halo: SegWalk.)  The two
// are separate instantiations so the plain path carries none of the chain
// bookkeeping.
struct PlainWalk : TileWalkT<kPairRows> {
    __device__ PlainWalk(int64_t first, int64_t step, int64_t slices, int tokens, int seg, int)
        : TileWalkT<kPairRows>(first, step, slices, tokens, seg) {}
    __device__ __forceinline__ bool chain_start() const { return false; }
    __device__ __forceinline__ bool halo() const { return false; }
};
template <bool DELTA>
using CompressWalk = typename std::conditional<DELTA, SegWalk<kPairRows>, PlainWalk>::type;

// The walk runs over the padded token range (tokens rounded up to 32) so that
// every record row, padding included, is written; rows at or past `tokens`
// are zero-filled.
template <int NBYTES>
__device__ __forceinline__ void store_words(uint8_t* dst, const unsigned* w) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int q = 0; q < NBYTES / 16; ++q)
            st_stream(reinterpret_cast<uint4*>(dst) + q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
    } else if constexpr (NBYTES % 8 == 0) {
#pragma unroll
        for (int q = 0; q < NBYTES / 8; ++q) reinterpret_cast<uint2*>(dst)[q] = make_uint2(w[2 * q], w[2 * q + 1]);
    } else {
#pragma unroll
        for (int q = 0; q < NBYTES / 4; ++q) reinterpret_cast<unsigned*>(dst)[q] = w[q];
    }
}

// The per-row work after the RoPE removal, shared by both two-thread
// kernels: the block codes (rotation, group scale, E8 search), the temporal
// delta, and the store of record row rrow.  y: the thread's coordinates in
// PairMap slots.  chain_start: row 0 of the tile begins a delta chain (it is
// stored raw); otherwise row 0's predecessor is the previous tile's last row,
// whose raw codes are in carry.  store: false for a halo tile (codes and
// carry only).
template <int D, int BITS, int MODE>
__device__ __forceinline__ void pair_encode_row(float (&y)[D / 2], int hf, int r, float sgn, bool active,
                                                bool delta, bool chain_start, bool store, int64_t rrow, int group,
                                                unsigned (&carry)[D / 16], unsigned& carry_c,
                                                uint8_t* __restrict__ idx, uint16_t* __restrict__ coset,
                                                __half* __restrict__ scales) {
    constexpr int DP = D;
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int NBT = PM::NBT;
    constexpr int NSUB = HALF / 32;  // 32-coordinate subgroups per thread
    using RP = RowPack<BITS, NBT>;
    constexpr int RB = DP * BITS / 8;  // idx bytes per row
    constexpr int RBT = RB / 2;        // idx bytes per thread
    // group is 32, 64 or 128: span = 2^gsh 32-coordinate subgroups per scale
    // group, nsc = DP / group scales per row (shifts, not divisions)
    const int gsh = group == 32 ? 0 : (group == 64 ? 1 : 2);
    const int nsc = DP >> (5 + gsh);

    unsigned short sc[NSUB];
    unsigned blk[NBT];
    unsigned cwl;
    pair_encode_codes<D, BITS, MODE != 0>(y, hf, sgn, group, blk, cwl, sc);
    if constexpr (MODE == 2) {  // strict joint format: the coset bit goes into the block code
#pragma unroll
        for (int k = 0; k < NBT; ++k) blk[k] = joint_pack<BITS>(blk[k], (cwl >> k) & 1u);
    }
    unsigned cw = cwl << (hf * NBT);
    cw |= __shfl_xor_sync(kFull, cw, 1);

    // ---- temporal delta against the previous token (row r - 1: lane - 2)
    if (delta) {
        const bool raw = r == 0 && chain_start;
#pragma unroll
        for (int k = 0; k < NBT; ++k) {
            unsigned prev = __shfl_up_sync(kFull, blk[k], 2);
            const unsigned last = __shfl_sync(kFull, blk[k], 30 + hf);
            if (r == 0) prev = carry[k];
            if (!raw) blk[k] = swar_sub<BITS>(blk[k], prev);
            carry[k] = last;  // raw codes of the tile's last token
        }
        unsigned pc = __shfl_up_sync(kFull, cw, 2);
        const unsigned lastc = __shfl_sync(kFull, cw, 30);
        if (r == 0) pc = carry_c;
        if (!raw) cw ^= pc;
        carry_c = lastc;
    }
    if (!store) return;  // a halo tile: only the carry was wanted

    // ---- store (padding rows past the slice get zeros)
    if (!active) {
#pragma unroll
        for (int k = 0; k < NBT; ++k) blk[k] = 0;
        cw = 0;
#pragma unroll
        for (int s = 0; s < NSUB; ++s) sc[s] = 0;
    }
    unsigned w[RP::WORDS];
    RP::pack(blk, w);
    store_words<RBT>(idx + rrow * RB + hf * RBT, w);
    if (MODE != 2 && hf == 0) coset[rrow] = uint16_t(cw);
#pragma unroll
    for (int s = 0; s < NSUB; ++s) {
        const int gs = hf * NSUB + s;  // global 32-subgroup
        if ((gs & ((1 << gsh) - 1)) == 0) scales[rrow * nsc + (gs >> gsh)] = __ushort_as_half(sc[s]);
    }
}

template <int D, int BITS, int MODE, bool DELTA>
__global__ void __launch_bounds__(kThreads, 2)
    compress_pair_kernel(const __half* __restrict__ x, const float4* __restrict__ rope, int64_t slices,
                         int tokens, int tpad, int group, int seg, int dchunk, uint8_t* __restrict__ idx,
                         uint16_t* __restrict__ coset, __half* __restrict__ scales) {
    constexpr int DP = PaddedDim<D>::value;  // head_dim 96 runs zero-padded to 128
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    using Walk = CompressWalk<DELTA>;
    constexpr bool delta = DELTA;

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int hf = lane & 1;
    const int r = lane >> 1;
    const float sgn = hf ? -1.0f : 1.0f;
    const uint32_t ring = smem_u32(smem) + (threadIdx.x >> 5) * (kPairStages * kPairTileBytes);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;

    Walk cur(warp, nwarps, slices, tpad, seg, dchunk);
    Walk pre = cur;
#pragma unroll
    for (int s = 0; s < kPairStages - 1; ++s) {
        if (pre.valid()) {
            load_pair_tile<D>(x, pre.slice, pre.t0, tokens, ring + s * kPairTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
    }

    unsigned carry[NBT];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NBT; ++k) carry[k] = 0;

    RingSlots<kPairStages> rs;

    for (int i = 0; cur.valid(); ++i) {
        if (pre.valid()) {
            load_pair_tile<D>(x, pre.slice, pre.t0, tokens, ring + rs.pre * kPairTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
        cp_async_wait<kPairStages - 1>();
        __syncwarp();
        const uint32_t stage = ring + rs.cur * kPairTileBytes;
        rs.advance();
        const int t = cur.t0 + r;
        const bool active = t < tokens;

        // ---- the thread's 64 (32) coordinates of row r (zeros past head_dim)
        float y[HALF];
        const PairTileAddr<DP> ta(stage, r, hf);
#pragma unroll
        for (int c = 0; c < NBT; ++c) {
            const int gc = PM::chunk(hf, c);
            if (D == DP || gc < D / 8) {
                h8_to_f(lds128(ta(c)), &y[8 * c]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) y[8 * c + j] = 0.0f;
            }
        }

        // ---- RoPE removal on keys
        if (rope != nullptr) {
            const float4* cs = rope + (active ? t : 0);
            if constexpr (D == DP) {  // pairs (i, i + D/2) are slots (l, l + Q)
#pragma unroll
                for (int qq = 0; qq < Q / 2; ++qq)
                    pair_rope_remove<D>(y, qq, __ldg(cs + int64_t(hf * (Q / 2) + qq) * tokens));
            } else {  // pairs (i, i + D/2) are not slot pairs: partners come from the tile
                pair_rope_remove_from_tile<D>(y, hf, stage, r, cs, tokens);
            }
        }
        __syncwarp();  // every lane has read its coordinates: the stage may be refilled

        pair_encode_row<DP, BITS, MODE>(y, hf, r, sgn, active, delta, cur.chain_start(), !cur.halo(),
                                         cur.slice * tpad + t, group, carry, carry_c, idx, coset, scales);
        cur.next();
    }
    cp_async_wait<0>();
}

// Keys: blocks of 8 warps sharing the RoPE table tile, a 2-deep ring, two
// blocks per SM (16 warps; a barrier waits for 8 of them).
constexpr int kCompressRopeWarps = 8;
constexpr int kCompressRopeThreads = kCompressRopeWarps * 32;
constexpr int kCompressRopeStages = 2;

template <int D, int BITS, int MODE, bool DELTA>
__global__ void __launch_bounds__(kCompressRopeThreads, 2)
    compress_pair_rope_kernel(const __half* __restrict__ x, const float4* __restrict__ rope, int64_t slices,
                              int tokens, int tpad, int group, int seg, int dchunk, uint8_t* __restrict__ idx,
                              uint16_t* __restrict__ coset, __half* __restrict__ scales) {
    constexpr int DP = D;
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    using RS = RopeRing<D, kCompressRopeWarps, kCompressRopeStages>;
    using Walk = CompressWalk<DELTA>;
    constexpr bool delta = DELTA;

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hf = lane & 1;
    const int r = lane >> 1;
    const float sgn = hf ? -1.0f : 1.0f;
    const int64_t ngroups = (slices + kCompressRopeWarps - 1) / kCompressRopeWarps;

    // the walk runs over slice groups; the warp's slice is 16 * group + wib
    Walk cur(blockIdx.x, gridDim.x, ngroups, tpad, seg, dchunk);
    Walk pre = cur;

    auto load_stage = [&](const Walk& w, uint32_t stage) {
        // the table tile: thread t copies token row t % 16 of planes t / 16 + 16 j
        constexpr int QS = kCompressRopeThreads / kPairRows;  // plane step
        static_assert((D / 4) % QS == 0, "table copies per thread");
        const int rr = threadIdx.x % kPairRows, q0 = threadIdx.x / kPairRows;
        const int tok = w.t0 + rr;
        const bool ok = tok < tokens;
        const float4* src = rope + int64_t(q0) * tokens + (ok ? tok : 0);
#pragma unroll
        for (int j = 0; j < (D / 4) / QS; ++j)
            cp_async16(stage + rope_slot<D>(q0 + QS * j, rr), src + int64_t(QS * j) * tokens, ok ? 16 : 0);
        const int64_t sl = w.slice * kCompressRopeWarps + wib;
        if (sl < slices) load_pair_tile<D>(x, sl, w.t0, tokens, stage + RS::TABLE + wib * kPairTileBytes, lane);
    };

#pragma unroll
    for (int s = 0; s < kCompressRopeStages - 1; ++s) {
        if (pre.valid()) {
            load_stage(pre, sbase + s * RS::BYTES);
            pre.next();
        }
        cp_async_commit();
    }

    unsigned carry[NBT];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NBT; ++k) carry[k] = 0;

    RingSlots<kCompressRopeStages> rs;

    for (int i = 0; cur.valid(); ++i) {
        cp_async_wait<kCompressRopeStages - 2>();  // this thread's copies of tile i are done
        __syncthreads();                    // everyone's are; everyone is done with tile i - 1
        if (pre.valid()) {
            load_stage(pre, sbase + rs.pre * RS::BYTES);
            pre.next();
        }
        cp_async_commit();
        const uint32_t stage = sbase + rs.cur * RS::BYTES;
        rs.advance();
        const int64_t slice = cur.slice * kCompressRopeWarps + wib;
        if (slice < slices) {  // warp-uniform
            const int t = cur.t0 + r;
            const bool active = t < tokens;
            float y[HALF];
            const uint32_t tile = stage + RS::TABLE + wib * kPairTileBytes;
            const PairTileAddr<DP> ta(tile, r, hf);
#pragma unroll
            for (int c = 0; c < NBT; ++c) h8_to_f(lds128(ta(c)), &y[8 * c]);
            // RoPE removal with the block's table tile: pairs (i, i + D/2) are slots (l, l + Q)
#pragma unroll
            for (int qq = 0; qq < Q / 2; ++qq) pair_rope_remove<D>(y, qq, rope_tile_entry<D>(stage, hf * (Q / 2) + qq, r));
            pair_encode_row<D, BITS, MODE>(y, hf, r, sgn, active, delta, cur.chain_start(), !cur.halo(),
                                             slice * tpad + t, group, carry, carry_c, idx, coset, scales);
        }
        cur.next();
    }
    cp_async_wait<0>();
}

// Segment length of the compression work items.  Without a delta every tile
// is an item.  With a delta, chains restart every delta_chunk tokens; a chunk
// of at most kMaxSeg tokens is one item, and a longer chain (the method's own
// single chain per slice when delta_chunk >= tokens) is cut into segments of
// at most kMaxSeg tokens, each preceded by one halo tile, halved down to
// kMinSeg while there are fewer than 4 items per resident warp.
constexpr int kMaxSeg = 1024;
constexpr int kMinSeg = 256;

static int compress_segment(const LaunchArgs& a, int64_t units, int64_t resident_warps) {
    if (a.delta_chunk <= 0) return kPairRows;
    if (a.delta_chunk <= kMaxSeg) return a.delta_chunk;
    int seg = kMaxSeg;
    while (seg > kMinSeg && units * ((a.tpad + seg - 1) / seg) < 4 * resident_warps) seg /= 2;
    return seg;
}

template <int D, int BITS, int MODE, bool DELTA>
static int launch_pair(const LaunchArgs& a, const __half* x, const float4* rope, uint8_t* idx,
                       uint16_t* coset, __half* scales) {
    auto kern = compress_pair_kernel<D, BITS, MODE, DELTA>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), kPairCompressSmem)) return NQ_ERR_CUDA;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern), kPairCompressSmem);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int seg = compress_segment(a, a.slices, int64_t(cap) * kWarpsPerBlock);
    const int64_t items = a.slices * ((a.tpad + seg - 1) / seg);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, kPairCompressSmem, a.stream>>>(x, rope, a.slices, a.tokens, a.tpad, a.group, seg,
                                                          a.delta_chunk, idx, coset, scales);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D, int BITS, int MODE, bool DELTA>
static int launch_pair_rope(const LaunchArgs& a, const __half* x, const float4* rope, uint8_t* idx,
                            uint16_t* coset, __half* scales) {
    auto kern = compress_pair_rope_kernel<D, BITS, MODE, DELTA>;
    constexpr int smem = RopeRing<D, kCompressRopeWarps, kCompressRopeStages>::SMEM;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem)) return NQ_ERR_CUDA;
    const int cap = grid_capacity_threads(reinterpret_cast<const void*>(kern), smem, kCompressRopeThreads);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int64_t groups = (a.slices + kCompressRopeWarps - 1) / kCompressRopeWarps;
    const int seg = compress_segment(a, groups, cap);  // items are block-wide
    const int64_t items = groups * ((a.tpad + seg - 1) / seg);
    if (items == 0) return NQ_OK;
    const int grid = int(std::min<int64_t>(items, cap));
    kern<<<grid, kCompressRopeThreads, smem, a.stream>>>(x, rope, a.slices, a.tokens, a.tpad, a.group, seg,
                                                 a.delta_chunk, idx, coset, scales);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D, int BITS, int MODE, bool DELTA>
static int launch_pair_any(const LaunchArgs& a, const __half* x, const float4* rope, uint8_t* idx,
                           uint16_t* coset, __half* scales) {
    return rope ? launch_pair_rope<D, BITS, MODE, DELTA>(a, x, rope, idx, coset, scales)
                : launch_pair<D, BITS, MODE, DELTA>(a, x, rope, idx, coset, scales);
}

template <int D, bool DELTA>
static int dispatch_bits(const LaunchArgs& a, int bits, int mode, const __half* x,
                         const float4* rope, uint8_t* idx, uint16_t* coset, __half* scales) {
#define NQ_MODE(B, M)                                                                           \
    if constexpr (D == 96)                                                                      \
        return launch_pair<D, B, M, DELTA>(a, x, rope, idx, coset, scales);                    \
    else                                                                                        \
        return launch_pair_any<D, B, M, DELTA>(a, x, rope, idx, coset, scales);
#define NQ_CASE(B)                                                                              \
    case B:                                                                                     \
        if (mode == 2) {                                                                        \
            NQ_MODE(B, 2)                                                                       \
        } else if (mode == 1) {                                                                 \
            NQ_MODE(B, 1)                                                                       \
        } else {                                                                                \
            NQ_MODE(B, 0)                                                                       \
        }
    switch (bits) {
        NQ_CASE(2)
        NQ_CASE(3)
        NQ_CASE(4)
        default:
            return NQ_ERR_UNSUPPORTED;
    }
#undef NQ_CASE
#undef NQ_MODE
}

// The launch of one tensor, with or without the temporal delta: the two
// instantiations live in translation units of their own (nq_compress.cu and
// nq_compress_delta.cu) so they compile in parallel.
template <bool DELTA>
int launch_compress_tensor_as(const LaunchArgs& a, int head_dim, int bits, int mode, const void* x,
                              const float* rope, uint8_t* idx, uint16_t* coset, uint16_t* scales) {
    const __half* xh = static_cast<const __half*>(x);
    const float4* r = reinterpret_cast<const float4*>(rope);
    __half* sh = reinterpret_cast<__half*>(scales);
    switch (head_dim) {
        case 64:
            return dispatch_bits<64, DELTA>(a, bits, mode, xh, r, idx, coset, sh);
        case 96:
            return dispatch_bits<96, DELTA>(a, bits, mode, xh, r, idx, coset, sh);
        case 128:
            return dispatch_bits<128, DELTA>(a, bits, mode, xh, r, idx, coset, sh);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

int launch_compress_tensor_delta(const LaunchArgs& a, int head_dim, int bits, int mode, const void* x,
                                 const float* rope, uint8_t* idx, uint16_t* coset, uint16_t* scales);

}  // namespace nq
