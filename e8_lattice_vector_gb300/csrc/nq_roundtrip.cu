// nq_roundtrip.cu -- the round trip in one pass: fp16 rows -> RoPE removal
// (keys) -> Hadamard -> group scale -> E8 nearest point -> scaled point ->
// inverse Hadamard -> RoPE re-apply -> fp16 rows, with no compressed
// intermediate in memory and no codes formed.  The reconstruction equals
// decompress(compress(x)) bit for bit: the lattice points and scales are the
// ones the compressor encodes (the temporal delta is lossless and has no
// effect here), a point's coordinate is exactly the decompressor's
// (code - offset), and the rest of the decode is the decompressor's.
//
// The streaming is the compressor's: fp16 tiles arrive in a shared-memory
// ring by cp.async; each reconstructed tile is written back into the ring
// slot its input came from (same swizzled layout the TMA tensor store reads)
// and leaves by TMA.  A slot is refilled only after the store from it has
// finished reading.  Tiles are read before they are written and never read
// again, so the output may alias the input (an in-place round trip).
#include "nq_decode.cuh"
#include "nq_encode.cuh"

namespace nq {

constexpr int kRtStages = 3;
// keys: blocks of 8 warps share the table tile, two blocks per SM, a 2-deep
// ring: the slot a store reads from is refilled at the next tile, after the
// warp has waited for that store's read and the block barrier
constexpr int kRtRopeWarps = 8;
constexpr int kRtRopeThreads = kRtRopeWarps * 32;
constexpr int kRtRopeStages = 2;
constexpr int kRtPairSmem = kWarpsPerBlock * kRtStages * kPairTileBytes + 1024;

// ------------------------------------------------------ two threads per row

// Encode + decode of the thread's half of row r (PairMap slots, RoPE removed).
// No codes are formed: the fast decoder hands over each block's lattice point,
// which is scaled straight back into the block's slots (the very product the
// decompressor forms from the code: (code - offset) is the point's coordinate
// exactly).  A block the fast decoder declines goes through the general path
// at once and its code is unscaled as in decompression.
template <int D, int BITS, bool STRICT>
__device__ __forceinline__ void pair_round_trip(float (&y)[D / 2], int hf, float sgn, int group) {
    constexpr int Q = PairMap<D>::Q;
    constexpr int NBT = PairMap<D>::NBT;
    constexpr int NSUB = D / 64;
    unsigned short sc[NSUB];
    float inv[NSUB];
    const bool fast = pair_rotate_scale<D, BITS>(y, sgn, group, sc, inv);
    float scf[NSUB];
#pragma unroll
    for (int s = 0; s < NSUB; ++s) scf[s] = __half2float(__ushort_as_half(sc[s]));
#pragma unroll
    for (int k = 0; k < NBT; ++k) {
        float u[8];
        pair_block_u<Q>(y, inv, sgn, k, u);
        unsigned c;
        const bool ok = e8_fast_point<BITS, STRICT>(u, c);
        const float s = scf[(8 * k) / 32];
        if (fast && ok) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 v = __fmul2_rn(make_float2(u[j], u[j + 4]), make_float2(s, s));
                y[8 * k + j] = v.x;
                y[8 * k + j + 4] = v.y;
            }
        } else {
            pair_block_u<Q>(y, inv, sgn, k, u);
            const uint2 res = e8_slow<BITS, STRICT>(make_float4(u[0], u[1], u[2], u[3]),
                                                    make_float4(u[4], u[5], u[6], u[7]));
            unscale_block<BITS>(res.x, res.y, s, &y[8 * k]);
        }
    }
    pair_inverse_rotation<D>(y, sgn);
}

// Values, keys without RoPE, and keys of head_dim 96 (RoPE from the global
// table, partners from the tile and by exchange): a warp per 16-token tile.
template <int D, int BITS, bool STRICT, bool ROPE>
__global__ void __launch_bounds__(kThreads, 2)
    roundtrip_pair_kernel(const __half* __restrict__ x, const float4* __restrict__ rope,
                          const __grid_constant__ CUtensorMap out_map, int64_t slices, int tokens, int group) {
    constexpr int DP = PaddedDim<D>::value;
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    using Walk = TileWalkT<kPairRows>;

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int hf = lane & 1;
    const int r = lane >> 1;
    const float sgn = hf ? -1.0f : 1.0f;
    const uint32_t ring =
        ((smem_u32(smem) + 1023u) & ~1023u) + (threadIdx.x >> 5) * (kRtStages * kPairTileBytes);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;

    Walk cur(warp, nwarps, slices, tokens, kPairRows);
    Walk pre = cur;
#pragma unroll
    for (int s = 0; s < kRtStages - 1; ++s) {
        if (pre.valid()) {
            load_pair_tile<D>(x, pre.slice, pre.t0, tokens, ring + s * kPairTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
    }

    RingSlots<kRtStages> rs;
    for (int i = 0; cur.valid(); ++i) {
        cp_async_wait<kRtStages - 2>();
        __syncwarp();
        const uint32_t stage = ring + rs.cur * kPairTileBytes;
        const int t = cur.t0 + r;
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
        const float4* cs = ROPE ? rope + (t < tokens ? t : 0) : nullptr;
        if constexpr (ROPE) {
            if constexpr (D == DP) {
#pragma unroll
                for (int qq = 0; qq < Q / 2; ++qq)
                    pair_rope_remove<D>(y, qq, __ldg(cs + int64_t(hf * (Q / 2) + qq) * tokens));
            } else {
                pair_rope_remove_from_tile<D>(y, hf, stage, r, cs, tokens);
            }
        }
        // the slot of tile i - 1 is refilled next: its store must have read it
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        if (pre.valid()) {
            load_pair_tile<D>(x, pre.slice, pre.t0, tokens, ring + rs.pre * kPairTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
        rs.advance();

        pair_round_trip<DP, BITS, STRICT>(y, hf, sgn, group);
        if constexpr (ROPE) {
            if constexpr (D == DP) {
#pragma unroll
                for (int qq = 0; qq < Q / 2; ++qq)
                    pair_rope_apply<D>(y, qq, __ldg(cs + int64_t(hf * (Q / 2) + qq) * tokens), sgn);
            } else {
                pair96_rope_apply(y, hf, cs, tokens);
            }
        }
        pair_store_rows<DP, 0>(y, stage, r, hf, lane, &out_map, cur.t0, int(cur.slice));
        cur.next();
    }
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Keys with RoPE: the warps of a block share the tile's table rows (8 slices
// at the same tokens), as in the compressor; one block barrier per tile.
template <int D, int BITS, bool STRICT>
__global__ void __launch_bounds__(kRtRopeThreads, 2)
    roundtrip_pair_rope_kernel(const __half* __restrict__ x, const float4* __restrict__ rope,
                               const __grid_constant__ CUtensorMap out_map, int64_t slices, int tokens,
                               int group) {
    using PM = PairMap<D>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    using RS = RopeRing<D, kRtRopeWarps, kRtRopeStages>;
    using Walk = TileWalkT<kPairRows>;

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hf = lane & 1;
    const int r = lane >> 1;
    const float sgn = hf ? -1.0f : 1.0f;
    const int64_t ngroups = (slices + kRtRopeWarps - 1) / kRtRopeWarps;

    Walk cur(blockIdx.x, gridDim.x, ngroups, tokens, kPairRows);
    Walk pre = cur;

    auto load_stage = [&](const Walk& w, uint32_t stage) {
        // the table tile: thread t copies token row t % 16 of planes t / 16 + QS j
        constexpr int QS = kRtRopeThreads / kPairRows;  // plane step
        const int rr = threadIdx.x % kPairRows, q0 = threadIdx.x / kPairRows;
        const int tok = w.t0 + rr;
        const bool ok = tok < tokens;
        const float4* src = rope + int64_t(q0) * tokens + (ok ? tok : 0);
#pragma unroll
        for (int j = 0; j < (D / 4 + QS - 1) / QS; ++j)
            if ((D / 4) % QS == 0 || q0 + QS * j < D / 4)
                cp_async16(stage + rope_slot<D>(q0 + QS * j, rr), src + int64_t(QS * j) * tokens, ok ? 16 : 0);
        const int64_t sl = w.slice * kRtRopeWarps + wib;
        if (sl < slices) load_pair_tile<D>(x, sl, w.t0, tokens, stage + RS::TABLE + wib * kPairTileBytes, lane);
    };

#pragma unroll
    for (int s = 0; s < kRtRopeStages - 1; ++s) {
        if (pre.valid()) {
            load_stage(pre, sbase + s * RS::BYTES);
            pre.next();
        }
        cp_async_commit();
    }

    RingSlots<kRtRopeStages> rs;
    for (int i = 0; cur.valid(); ++i) {
        cp_async_wait<kRtRopeStages - 2>();  // this thread's copies of tile i are done
        // the ring slot about to be refilled held tile i - 1: this warp's store
        // from it must have finished reading before the barrier releases the refill
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncthreads();
        if (pre.valid()) {
            load_stage(pre, sbase + rs.pre * RS::BYTES);
            pre.next();
        }
        cp_async_commit();
        const uint32_t stage = sbase + rs.cur * RS::BYTES;
        rs.advance();
        const int64_t slice = cur.slice * kRtRopeWarps + wib;
        if (slice < slices) {  // warp-uniform
            const uint32_t tile = stage + RS::TABLE + wib * kPairTileBytes;
            float y[HALF];
            const PairTileAddr<D> ta(tile, r, hf);
#pragma unroll
            for (int c = 0; c < NBT; ++c) h8_to_f(lds128(ta(c)), &y[8 * c]);
#pragma unroll
            for (int qq = 0; qq < Q / 2; ++qq) pair_rope_remove<D>(y, qq, rope_tile_entry<D>(stage, hf * (Q / 2) + qq, r));
            pair_round_trip<D, BITS, STRICT>(y, hf, sgn, group);
#pragma unroll
            for (int qq = 0; qq < Q / 2; ++qq)
                pair_rope_apply<D>(y, qq, rope_tile_entry<D>(stage, hf * (Q / 2) + qq, r), sgn);
            __syncwarp();  // every lane has read its input from the tile
            pair_store_rows<D, 0>(y, tile, r, hf, lane, &out_map, cur.t0, int(slice));
        }
        cur.next();
    }
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------- launch

template <typename K>
static int grid_for(K kern, int smem, int threads, int64_t items) {
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem)) return -1;
    const int cap = grid_capacity_threads(reinterpret_cast<const void*>(kern), smem, threads);
    if (cap <= 0) return -1;
    return int(std::min<int64_t>(items, cap));
}

template <int D, int BITS, bool STRICT>
static int launch_rt(const LaunchArgs& a, const __half* x, const float4* rope, const CUtensorMap& map) {
    const int64_t tiles16 = (a.tokens + kPairRows - 1) / kPairRows;
    if constexpr (D != 96) {
        if (rope != nullptr) {
            auto kern = roundtrip_pair_rope_kernel<D, BITS, STRICT>;
            constexpr int smem = RopeRing<D, kRtRopeWarps, kRtRopeStages>::SMEM;
            const int64_t items = (a.slices + kRtRopeWarps - 1) / kRtRopeWarps * tiles16;
            const int grid = grid_for(kern, smem, kRtRopeThreads, items);
            if (grid < 0) return NQ_ERR_CUDA;
            kern<<<grid, kRtRopeThreads, smem, a.stream>>>(x, rope, map, a.slices, a.tokens, a.group);
            return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
        }
    }
    auto kern = rope != nullptr ? roundtrip_pair_kernel<D, BITS, STRICT, true>
                                : roundtrip_pair_kernel<D, BITS, STRICT, false>;
    const int64_t items = a.slices * tiles16;
    const int grid = grid_for(kern, kRtPairSmem, kThreads, (items + kWarpsPerBlock - 1) / kWarpsPerBlock);
    if (grid < 0) return NQ_ERR_CUDA;
    kern<<<grid, kThreads, kRtPairSmem, a.stream>>>(x, rope, map, a.slices, a.tokens, a.group);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D>
static int dispatch_bits(const LaunchArgs& a, int bits, bool strict, const __half* x, const float4* rope,
                         const CUtensorMap& map) {
    switch (bits * 2 + (strict ? 1 : 0)) {
        case 4: return launch_rt<D, 2, false>(a, x, rope, map);
        case 5: return launch_rt<D, 2, true>(a, x, rope, map);
        case 6: return launch_rt<D, 3, false>(a, x, rope, map);
        case 7: return launch_rt<D, 3, true>(a, x, rope, map);
        case 8: return launch_rt<D, 4, false>(a, x, rope, map);
        case 9: return launch_rt<D, 4, true>(a, x, rope, map);
        default: return NQ_ERR_UNSUPPORTED;
    }
}

int launch_roundtrip_tensor(const LaunchArgs& a, int head_dim, int bits, bool strict, const void* x,
                            const float* rope, void* x_out) {
    if (a.slices == 0 || a.tokens == 0) return NQ_OK;
    CUtensorMap map;
    if (!make_row_tile_map(&map, x_out, head_dim, a.tokens, a.slices, kPairRows)) return NQ_ERR_CUDA;
    const __half* xh = static_cast<const __half*>(x);
    const float4* r = reinterpret_cast<const float4*>(rope);
    switch (head_dim) {
        case 64: return dispatch_bits<64>(a, bits, strict, xh, r, map);
        case 96: return dispatch_bits<96>(a, bits, strict, xh, r, map);
        case 128: return dispatch_bits<128>(a, bits, strict, xh, r, map);
        default: return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq
