// nq_decompress.cu -- fused decompression kernels: idx / coset / scale
// sections -> undo temporal delta -> unpack -> unscale -> inverse Hadamard ->
// RoPE re-apply (keys) -> fp16 rows.
//
// head_dim 96 / 128: a warp per 32-token tile of a slice, lane r owns row r
// (one thread per row; for the decode this beats two threads per row).  A
// tile's records (idx rows, coset words, scales) are contiguous and 16-byte
// aligned thanks to the per-slice padding of the record rows, so they stream
// through a 3-stage shared-memory ring by cp.async; keys run in blocks of
// warps that also stage the tile's RoPE table rows once for the block.
// Without a temporal delta every tile is a work item; with one, a run of up
// to 32 consecutive tiles of a chain is, walked in order.  The delta is undone
// in place on the record tile, column-wise (field-wise addition modulo 2^b),
// plus the running sum of the chain's earlier rows, carried in registers from
// tile to tile; a run that does not start its chain takes its starting sum
// from the workspace, where two light passes over the idx section leave it
// (nq_chain.cuh).  Coset words by an exclusive-or warp scan.  The reconstructed fp16 rows
// are written into a swizzled shared-memory tile and leave by one TMA tensor
// store per 64 columns, which clips the rows past the end of the slice and the
// columns past head_dim.  head_dim 64 uses two threads per row (16-row tiles).
#include "nq_chain.cuh"
#include "nq_decode.cuh"

namespace nq {

constexpr int kStages = 3;
constexpr int kRecIdx = 0;        // idx rows: 32 * RB <= 2048 bytes
constexpr int kRecCoset = 2048;   // 32 coset words: 64 bytes
constexpr int kRecScale = 2112;   // 32 * (Dp / group) fp16 <= 256 bytes
constexpr int kRecStage = 2560;   // stage pitch
constexpr int kOutBufs = 2;
// per-warp region, a multiple of 1024 bytes: the output tiles must sit on
// 1024-byte boundaries for the 128-byte swizzle pattern of the tensor store
constexpr int kWarpSmem = (kOutBufs * kTileBytes + kStages * kRecStage + 1023) / 1024 * 1024;
constexpr int kDecompressSmem = kWarpsPerBlock * kWarpSmem + 1024;  // + alignment slack

template <int RB>
__device__ __forceinline__ void load_records(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset,
                                             const __half* __restrict__ scales, int nsc, int64_t row0,
                                             uint32_t stage, int lane) {
    // idx: 32 * RB bytes = 2 * RB chunks
    const uint8_t* ib = idx + row0 * RB;
#pragma unroll
    for (int g = lane; g < 2 * RB; g += 32) cp_async16(stage + kRecIdx + 16 * g, ib + 16 * g, 16);
    if (lane < 4 && coset != nullptr) cp_async16(stage + kRecCoset + 16 * lane, coset + row0 + 8 * lane, 16);
    const int nsch = 4 * nsc;  // 32 * nsc * 2 / 16
    if (lane < nsch) cp_async16(stage + kRecScale + 16 * lane, scales + row0 * nsc + 8 * lane, 16);
}

// ------------------------------------------- temporal delta, tile-wise
//
// The delta is undone in place on the 32-row idx tile in shared memory, down
// its columns: lane l takes column unit l % NU (a 32-bit word of 16 two-bit or
// 8 four-bit fields, or a 3-word group holding four 24-bit block codes at 3
// bits) of the rows of segment l / NU; it forms the running field-wise sums
// (mod 2^b) down its segment, adds the exclusive sum of the segments above
// (a shuffle scan over the segments) and the carry of the chunk's earlier
// tiles, and writes the codes back.  Far fewer shuffles and additions than a
// 32-lane scan of every block of every row.
// rows: shared address of row 0 of the tile's ROWS idx rows (RB bytes each);
// carry: the lane's unit in the previous tile's last row (unused when first).
// With COSET, the lanes of unit 0 also undo the coset words' delta (exclusive
// or) down their segment's rows of the coset column at `cosets` (one 16-bit
// word per row), riding on the same segment scan; carry_c: the previous
// tile's last raw coset word (unused when first), updated to this tile's.
template <int BITS, int RB, int ROWS = 32, bool COSET = false>
__device__ __forceinline__ void undelta_tile(uint32_t rows, int lane, bool first,
                                             unsigned (&carry)[DeltaUnit<BITS>::NV], uint32_t cosets = 0,
                                             unsigned* carry_c = nullptr) {
    using DU = DeltaUnit<BITS>;
    constexpr int NV = DU::NV;
    constexpr int NU = RB / (4 * DU::U);  // units per row
    constexpr int SEGS = 32 / NU;
    constexpr int RPS = ROWS / SEGS;       // rows per segment
    static_assert(NU * SEGS == 32 && RPS * SEGS == ROWS, "tile split");
    const int u = lane % NU, sg = lane / NU;
    const uint32_t base = rows + uint32_t(sg * RPS * RB + 4 * DU::U * u);
    unsigned v[RPS][NV];
#pragma unroll
    for (int i = 0; i < RPS; ++i) DU::load(base + i * RB, v[i]);
    unsigned c[RPS], crun = 0u;
#pragma unroll
    for (int i = 0; i < RPS; ++i) c[i] = 0u;
    const uint32_t cbase = cosets + uint32_t(2 * sg * RPS);
    if constexpr (COSET) {
        if (u == 0) {
#pragma unroll
            for (int i = 0; i < RPS; ++i) c[i] = lds16(cbase + 2 * i);
#pragma unroll
            for (int i = 1; i < RPS; ++i) c[i] ^= c[i - 1];
            crun = c[RPS - 1];
        }
    }
#pragma unroll
    for (int i = 1; i < RPS; ++i)
#pragma unroll
        for (int n = 0; n < NV; ++n) v[i][n] = DU::add(v[i][n], v[i - 1][n]);
    unsigned run[NV], ex[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) run[n] = v[RPS - 1][n];
#pragma unroll
    for (int d = 1; d < SEGS; d *= 2) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const unsigned t = __shfl_up_sync(kFull, run[n], d * NU);
            if (sg >= d) run[n] = DU::add(run[n], t);
        }
        if constexpr (COSET) {
            const unsigned t = __shfl_up_sync(kFull, crun, d * NU);
            if (sg >= d) crun ^= t;
        }
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        ex[n] = __shfl_up_sync(kFull, run[n], NU);
        if (sg == 0) ex[n] = 0u;
        if (!first) ex[n] = DU::add(ex[n], carry[n]);
    }
#pragma unroll
    for (int i = 0; i < RPS; ++i) {
#pragma unroll
        for (int n = 0; n < NV; ++n) v[i][n] = DU::add(v[i][n], ex[n]);
        DU::store(base + i * RB, v[i]);
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) carry[n] = __shfl_sync(kFull, v[RPS - 1][n], u + (SEGS - 1) * NU);
    if constexpr (COSET) {
        unsigned exc = __shfl_up_sync(kFull, crun, NU);
        if (sg == 0) exc = 0u;
        if (!first) exc ^= *carry_c;
        if (u == 0) {
#pragma unroll
            for (int i = 0; i < RPS; ++i) {
                c[i] ^= exc;
                sts16(cbase + 2 * i, c[i]);
            }
        }
        *carry_c = __shfl_sync(kFull, c[RPS - 1], (SEGS - 1) * NU);
    }
}

// One record row (the lane's row of a 32-row record tile in `stage`) ->
// unscaled, inverse-transformed coordinates, before the RoPE re-apply.
template <int D, int BITS, bool JOINT>
__device__ __forceinline__ void decode_row(uint32_t stage, const uint8_t* stage_gen, int lane, int nsc, int gshift,
                                           bool delta, bool first,
                                           unsigned (&carry)[PaddedDim<D>::value / 8], unsigned& carry_c,
                                           float (&y)[PaddedDim<D>::value]) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    using C = Code<BITS>;
    using RP = RowPack<BITS, NB>;
    constexpr int RB = DP * BITS / 8;

    // ---- undo the temporal delta of the idx tile and its coset words in place
    //      (every lane takes part)
    if (delta) {
        constexpr int NV = DeltaUnit<BITS>::NV;
        unsigned cu[NV];
#pragma unroll
        for (int n = 0; n < NV; ++n) cu[n] = carry[n];
        undelta_tile<BITS, RB, 32, !JOINT>(stage + kRecIdx, lane, first, cu, stage + kRecCoset, &carry_c);
#pragma unroll
        for (int n = 0; n < NV; ++n) carry[n] = cu[n];
        __syncwarp();
    }

    // ---- the lane's record
    unsigned w[RP::WORDS];
    if constexpr (RB % 16 == 0) {
#pragma unroll
        for (int q = 0; q < RB / 16; ++q) {
            const uint4 v = lds128(stage + kRecIdx + lane * RB + 16 * q);
            w[4 * q] = v.x;
            w[4 * q + 1] = v.y;
            w[4 * q + 2] = v.z;
            w[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < RB / 8; ++q) {
            const uint2 v = lds64(stage + kRecIdx + lane * RB + 8 * q);
            w[2 * q] = v.x;
            w[2 * q + 1] = v.y;
        }
    }
    const uint16_t* stage_h = reinterpret_cast<const uint16_t*>(stage_gen);
    unsigned cw = JOINT ? 0u : unsigned(stage_h[kRecCoset / 2 + lane]);
    float scf[DP / 32];
#pragma unroll
    for (int s = 0; s < DP / 32; ++s)
        scf[s] = __half2float(__ushort_as_half(stage_h[kRecScale / 2 + lane * nsc + ((32 * s) >> gshift)]));
    __syncwarp();  // the stage may be refilled
    unsigned blk[NB];
    RP::unpack(w, blk);

    // (the coset words' delta was undone with the idx tile, in shared memory)

    if constexpr (JOINT) {  // strict joint format: the coset bits come out of the block codes
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            unsigned c;
            blk[k] = joint_split<BITS>(blk[k], c);
            cw |= c << k;
        }
    }
    row_decode_codes<D, BITS>(blk, cw, scf, y);
}

template <int D, int BITS, bool JOINT>
__global__ void __launch_bounds__(kThreads, 1)
    decompress_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset,
                      const __half* __restrict__ scales, const float4* __restrict__ rope,
                      const __grid_constant__ CUtensorMap out_map, int64_t slices, int tokens, int tpad,
                      int group, const ChainState cs) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    constexpr int RB = DP * BITS / 8;
    constexpr int NU = RB / (4 * DeltaUnit<BITS>::U);  // column units of the tile scan

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const uint32_t wbase = ((smem_u32(smem) + 1023u) & ~1023u) + (threadIdx.x >> 5) * kWarpSmem;
    const uint32_t outbuf = wbase;                           // kOutBufs x 8 KB, 1024-aligned
    const uint32_t ring = wbase + kOutBufs * kTileBytes;     // kStages x kRecStage
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int gshift = group == 32 ? 5 : (group == 64 ? 6 : 7);
    const int nsc = DP >> gshift;

    unsigned carry[NB];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NB; ++k) carry[k] = 0;

    // single tiles without a delta, groups of a chain's tiles with one
    auto run = [&](auto cur) {
        auto pre = cur;
#pragma unroll
        for (int s = 0; s < kStages - 1; ++s) {
            if (pre.valid()) {
                load_records<RB>(idx, coset, scales, nsc, pre.slice * tpad + pre.t0, ring + s * kRecStage, lane);
                pre.next();
            }
            cp_async_commit();
        }
        for (int i = 0; cur.valid(); ++i) {
            if (pre.valid()) {
                load_records<RB>(idx, coset, scales, nsc, pre.slice * tpad + pre.t0,
                                 ring + ((i + kStages - 1) % kStages) * kRecStage, lane);
                pre.next();
            }
            cp_async_commit();
            cp_async_wait<kStages - 1>();
            __syncwarp();
            const uint32_t stage = ring + (i % kStages) * kRecStage;
            const int t = cur.t0 + lane;
            bool first = false;  // row 0 starts its chain: no carry
            if constexpr (decltype(cur)::kGroups) {
                if (cur.group_start()) {
                    if (cs.gexcl != nullptr)
                        load_group_carry<BITS, RB>(cs, cur.G, lane % NU, carry, carry_c, !JOINT);
                    else
                        first = true;
                }
            } else {
                first = cur.t0 == cur.t_begin();  // chains of one chunk: its first tile
            }
            const uint8_t* stage_gen = smem + (stage - smem_u32(smem));
            float y[DP];
            decode_row<D, BITS, JOINT>(stage, stage_gen, lane, nsc, gshift, cs.delta, first, carry, carry_c, y);
            // ---- RoPE re-apply on keys: rotate each (i, i + D/2) pair by +angle
            if (rope != nullptr) {
                const float4* tab = rope + (t < tokens ? t : cur.t0);  // [D/4][tokens]
#pragma unroll
                for (int q = 0; q < D / 4; ++q) rope_apply_pairs<D>(y, q, __ldg(tab + int64_t(q) * tokens));
            }
            store_rows<D, 1>(y, outbuf + (i & 1) * kTileBytes, lane, &out_map, cur.t0, int(cur.slice));
            cur.next();
        }
    };
    // plain tiles without a delta; whole chunks, tile after tile, when every
    // chain fits one run; runs of a chain's tiles (carry from the workspace)
    // else.  Three call sites: the first keeps its chunk a constant.
    if (!cs.delta)
        run(TileWalk(warp, nwarps, slices, tokens, kTileRows));
    else if (cs.gexcl == nullptr)
        run(TileWalk(warp, nwarps, slices, tokens, int(cs.geo.tpc) * kTileRows));
    else
        run(GroupWalk<kTileRows>(warp, nwarps, slices, cs.geo));
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------ keys with a shared table
//
// Keys of head_dim 96 / 128: the 4 warps of a block decode the same 32-token
// tile of 4 consecutive slices (slice = 4 * group + warp), so the tile's RoPE
// table rows are staged in shared memory once per block instead of being read
// from L2 by every warp.  Three stages (table tile + the warps' record
// tiles), one output tile per warp; one block barrier per tile.  Two blocks
// per SM: a barrier holds 4 warps, not all 8.
constexpr int kKeyWarps = 4;
constexpr int kKeyThreads = 32 * kKeyWarps;
constexpr int kKeyStages = 3;

template <int D>
struct KeyStage {
    static constexpr int TABLE = D * 4 * kTileRows;  // head_dim/4 planes x 32 tokens x 16 B
    static constexpr int BYTES = TABLE + kKeyWarps * kRecStage;
    static constexpr int OUT = kKeyWarps * kTileBytes;
    static constexpr int SMEM = OUT + kKeyStages * BYTES + 1024;
};

template <int D, int BITS, bool JOINT>
__global__ void __launch_bounds__(kKeyThreads, 1)
    decompress_key_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset,
                          const __half* __restrict__ scales, const float4* __restrict__ rope,
                          const __grid_constant__ CUtensorMap out_map, int64_t slices, int tokens, int tpad,
                          int group, const ChainState cs) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    constexpr int RB = DP * BITS / 8;
    constexpr int NU = RB / (4 * DeltaUnit<BITS>::U);
    using KS = KeyStage<D>;

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;
    const uint8_t* gbase = smem + (base - smem_u32(smem));
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t outbuf = base + wib * kTileBytes;  // 1024-aligned
    const uint32_t stages = base + KS::OUT;
    const int gshift = group == 32 ? 5 : (group == 64 ? 6 : 7);
    const int nsc = DP >> gshift;
    const int64_t ngroups = (slices + kKeyWarps - 1) / kKeyWarps;

    // stage the table rows of tokens t0.. and the warp's record tile of slice group grp
    auto load_stage = [&](int64_t grp, int t0, uint32_t stage) {
        // the table tile: thread t copies token row t % 32 of planes t / 32 + 4 j
        constexpr int QS = kKeyThreads / kTileRows;  // plane step
        static_assert((D / 4) % QS == 0, "table copies per thread");
        const int tok = t0 + lane;
        const bool ok = tok < tokens;
        const float4* src = rope + int64_t(wib) * tokens + (ok ? tok : 0);
#pragma unroll
        for (int j = 0; j < (D / 4) / QS; ++j)
            cp_async16(stage + 16 * (threadIdx.x + kKeyThreads * j), src + int64_t(QS * j) * tokens, ok ? 16 : 0);
        const int64_t sl = grp * kKeyWarps + wib;
        if (sl < slices) load_records<RB>(idx, coset, scales, nsc, sl * tpad + t0, stage + KS::TABLE + wib * kRecStage, lane);
    };

    unsigned carry[NB];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NB; ++k) carry[k] = 0;

    // single tiles without a delta, groups of a chain's tiles with one (items over slice groups)
    auto run = [&](auto cur) {
        auto pre = cur;
#pragma unroll
        for (int st = 0; st < kKeyStages - 1; ++st) {
            if (pre.valid()) {
                load_stage(pre.slice, pre.t0, stages + st * KS::BYTES);
                pre.next();
            }
            cp_async_commit();
        }
        for (int i = 0; cur.valid(); ++i) {
            cp_async_wait<kKeyStages - 2>();  // this thread's copies of tile i are done
            __syncthreads();                  // everyone's are; everyone is done with tile i - 1
            if (pre.valid()) {
                load_stage(pre.slice, pre.t0, stages + ((i + kKeyStages - 1) % kKeyStages) * KS::BYTES);
                pre.next();
            }
            cp_async_commit();
            const uint32_t stage = stages + (i % kKeyStages) * KS::BYTES;
            const int64_t slice = cur.slice * kKeyWarps + wib;
            if (slice < slices) {  // warp-uniform
                bool first = false;
                if constexpr (decltype(cur)::kGroups) {
                    if (cur.group_start()) {
                        if (cs.gexcl != nullptr)
                            load_group_carry<BITS, RB>(cs, cur.slice_group(uint64_t(slice)), lane % NU, carry, carry_c,
                                                       !JOINT);
                        else
                            first = true;
                    }
                } else {
                    first = cur.t0 == cur.t_begin();
                }
                const uint32_t rec = stage + KS::TABLE + wib * kRecStage;
                float y[DP];
                decode_row<D, BITS, JOINT>(rec, gbase + (rec - base), lane, nsc, gshift, cs.delta, first, carry,
                                           carry_c, y);
#pragma unroll
                for (int q = 0; q < D / 4; ++q) {
                    const uint4 raw = lds128(stage + 16 * (q * kTileRows + lane));
                    rope_apply_pairs<D>(y, q, make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y),
                                                          __uint_as_float(raw.z), __uint_as_float(raw.w)));
                }
                store_rows<D, 0>(y, outbuf, lane, &out_map, cur.t0, int(slice));
            }
            cur.next();
        }
    };
    if (!cs.delta)
        run(TileWalk(blockIdx.x, gridDim.x, ngroups, tokens, kTileRows));
    else if (cs.gexcl == nullptr)
        run(TileWalk(blockIdx.x, gridDim.x, ngroups, tokens, int(cs.geo.tpc) * kTileRows));
    else
        run(GroupWalk<kTileRows>(blockIdx.x, gridDim.x, ngroups, cs.geo));
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------- two threads per row
//
// head_dim 64 and 128: lanes 2r and 2r+1 share record row r of a 16-row tile.
// Thread hf unpacks scale-group half hf (blocks [hf*NBT, (hf+1)*NBT)); the
// inverse Hadamard transform (textbook order) runs its bits below DP/4
// in-thread, bit DP/4 in-thread with a sign that leaves the odd thread's slot
// halves exchanged, and bit DP/2 as one symmetric shuffle exchange, after which
// the slots hold the RoPE pairs (PairMap layout; the odd thread's upper slots
// negated, undone by a sign flip of sin in the rotation and of the fp16 bits).
constexpr int kPairRecIdx = 0;      // 16 * RB <= 1024 bytes
constexpr int kPairRecCoset = 1024; // 16 coset words
constexpr int kPairRecScale = 1056; // 16 * (Dp / group) fp16 <= 128 bytes
constexpr int kPairRecStage = 1280;
constexpr int kPairWarpSmem = (kOutBufs * kPairTileBytes + kStages * kPairRecStage + 1023) / 1024 * 1024;
constexpr int kPairDecompressSmem = kWarpsPerBlock * kPairWarpSmem + 1024;

template <int RB>
__device__ __forceinline__ void load_pair_records(const uint8_t* __restrict__ idx,
                                                  const uint16_t* __restrict__ coset,
                                                  const __half* __restrict__ scales, int nsc, int64_t row0,
                                                  uint32_t stage, int lane) {
    const uint8_t* ib = idx + row0 * RB;  // 16 * RB bytes = RB chunks
#pragma unroll
    for (int g = lane; g < RB; g += 32) cp_async16(stage + kPairRecIdx + 16 * g, ib + 16 * g, 16);
    if (lane < 2 && coset != nullptr) cp_async16(stage + kPairRecCoset + 16 * lane, coset + row0 + 8 * lane, 16);
    const int nsch = 2 * nsc;  // 16 * nsc * 2 / 16
    if (lane < nsch) cp_async16(stage + kPairRecScale + 16 * lane, scales + row0 * nsc + 8 * lane, 16);
}

template <int NBYTES>
__device__ __forceinline__ void lds_words(uint32_t a, unsigned* w) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int q = 0; q < NBYTES / 16; ++q) {
            const uint4 v = lds128(a + 16 * q);
            w[4 * q] = v.x;
            w[4 * q + 1] = v.y;
            w[4 * q + 2] = v.z;
            w[4 * q + 3] = v.w;
        }
    } else if constexpr (NBYTES % 8 == 0) {
#pragma unroll
        for (int q = 0; q < NBYTES / 8; ++q) {
            const uint2 v = lds64(a + 8 * q);
            w[2 * q] = v.x;
            w[2 * q + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int q = 0; q < NBYTES / 4; ++q) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[q]) : "r"(a + 4 * q));
    }
}

template <int D, int BITS, bool JOINT>
__global__ void __launch_bounds__(kThreads, 2)
    decompress_pair_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset,
                           const __half* __restrict__ scales, const float4* __restrict__ rope,
                           const __grid_constant__ CUtensorMap out_map, int64_t slices, int tokens, int tpad,
                           int group, const ChainState cs) {
    constexpr int DP = D;
    using PM = PairMap<DP>;
    constexpr int HALF = PM::HALF;
    constexpr int Q = PM::Q;
    constexpr int NBT = PM::NBT;
    constexpr int NSUB = HALF / 32;
    using RP = RowPack<BITS, NBT>;
    constexpr int RB = DP * BITS / 8;
    constexpr int RBT = RB / 2;
    constexpr int NV = DeltaUnit<BITS>::NV;
    constexpr int NU = RB / (4 * DeltaUnit<BITS>::U);

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int hf = lane & 1;
    const int r = lane >> 1;
    const float sgn = hf ? -1.0f : 1.0f;
    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;
    const uint8_t* gbase = smem + (base - smem_u32(smem));
    const uint32_t wbase = base + (threadIdx.x >> 5) * kPairWarpSmem;
    const uint32_t outbuf = wbase;
    const uint32_t ring = wbase + kOutBufs * kPairTileBytes;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int gsh = group == 32 ? 0 : (group == 64 ? 1 : 2);  // log2 of 32-subgroups per scale
    const int nsc = DP >> (5 + gsh);

    unsigned carry[NBT];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NBT; ++k) carry[k] = 0;

    // single tiles without a delta, groups of a chain's tiles with one
    auto run = [&](auto cur) {
        auto pre = cur;
#pragma unroll
        for (int s = 0; s < kStages - 1; ++s) {
            if (pre.valid()) {
                load_pair_records<RB>(idx, coset, scales, nsc, pre.slice * tpad + pre.t0, ring + s * kPairRecStage, lane);
                pre.next();
            }
            cp_async_commit();
        }
        for (int i = 0; cur.valid(); ++i) {
            if (pre.valid()) {
                load_pair_records<RB>(idx, coset, scales, nsc, pre.slice * tpad + pre.t0,
                                      ring + ((i + kStages - 1) % kStages) * kPairRecStage, lane);
                pre.next();
            }
            cp_async_commit();
            cp_async_wait<kStages - 1>();
            __syncwarp();
            const uint32_t stage = ring + (i % kStages) * kPairRecStage;
            const uint8_t* gstage = gbase + (stage - base);
            const int t = cur.t0 + r;

            // ---- undo the temporal delta of the idx tile in place (every lane takes part)
            bool first = false;  // row 0 starts its chain: no carry
            if constexpr (decltype(cur)::kGroups) {
                if (cur.group_start()) {
                    if (cs.gexcl != nullptr) {
                        load_group_carry<BITS, RB>(cs, cur.G, lane % NU, carry, carry_c, !JOINT);
                        carry_c = (carry_c >> (hf * NBT)) & ((1u << NBT) - 1u);  // the thread's half of the word
                    } else {
                        first = true;
                    }
                }
                unsigned cu[NV];
#pragma unroll
                for (int n = 0; n < NV; ++n) cu[n] = carry[n];
                undelta_tile<BITS, RB, kPairRows>(stage + kPairRecIdx, lane, first, cu);
#pragma unroll
                for (int n = 0; n < NV; ++n) carry[n] = cu[n];
                __syncwarp();
            }

            // ---- the thread's half of the record
            unsigned w[RP::WORDS];
            lds_words<RBT>(stage + kPairRecIdx + r * RB + hf * RBT, w);
            const unsigned cw_full = JOINT ? 0u : unsigned(reinterpret_cast<const uint16_t*>(gstage + kPairRecCoset)[r]);
            unsigned cw = (cw_full >> (hf * NBT)) & ((1u << NBT) - 1u);
            float scf[NSUB];
#pragma unroll
            for (int s = 0; s < NSUB; ++s)
                scf[s] = __half2float(reinterpret_cast<const __half*>(gstage + kPairRecScale)[r * nsc + ((hf * NSUB + s) >> gsh)]);
            __syncwarp();  // the stage may be refilled
            unsigned blk[NBT];
            RP::unpack(w, blk);

            // ---- the coset words' delta: an exclusive-or scan over the rows (lane stride 2) + carry
            if (decltype(cur)::kGroups && !JOINT) {
#pragma unroll
                for (int off = 2; off < 32; off *= 2) {
                    const unsigned vc = __shfl_up_sync(kFull, cw, off);
                    if (lane >= off) cw ^= vc;
                }
                if (!first) cw ^= carry_c;
                carry_c = __shfl_sync(kFull, cw, 30 + hf);
            }

            if constexpr (JOINT) {  // strict joint format: the coset bits come out of the block codes
#pragma unroll
                for (int k = 0; k < NBT; ++k) {
                    unsigned c;
                    blk[k] = joint_split<BITS>(blk[k], c);
                    cw |= c << k;
                }
            }

            float y[HALF];
            pair_decode_codes<D, BITS>(blk, cw, scf, sgn, y);

            // ---- RoPE re-apply on keys: pairs (i, i + D/2) are slots (l, l + Q)
            if (rope != nullptr) {
                const float4* tab = rope + (t < tokens ? t : cur.t0);
#pragma unroll
                for (int qq = 0; qq < Q / 2; ++qq)
                    pair_rope_apply<D>(y, qq, __ldg(tab + int64_t(hf * (Q / 2) + qq) * tokens), sgn);
            }

            pair_store_rows<D, 1>(y, outbuf + (i & 1) * kPairTileBytes, r, hf, lane, &out_map, cur.t0, int(cur.slice));
            cur.next();
        }
    };
    if (!cs.delta)
        run(TileWalkT<kPairRows>(warp, nwarps, slices, tokens, kPairRows));
    else
        run(GroupWalk<kPairRows>(warp, nwarps, slices, cs.geo));
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Work items: single tiles without a delta, groups of a chain's tiles with
// one (units: slices, or the key kernel's groups of slices).
static int64_t work_items(const LaunchArgs& a, int64_t units, int rows, const ChainState& cs) {
    if (!cs.delta) return units * ((a.tokens + rows - 1) / rows);
    return units * int64_t(cs.geo.cps) * cs.geo.gpc;
}

template <int D, int BITS, bool JOINT>
static int launch_pair(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                       const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    auto kern = decompress_pair_kernel<D, BITS, JOINT>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), kPairDecompressSmem)) return NQ_ERR_CUDA;
    const int64_t items = work_items(a, a.slices, kPairRows, cs);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern), kPairDecompressSmem);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, kPairDecompressSmem, a.stream>>>(idx, coset, scales, rope, map, a.slices, a.tokens,
                                                            a.tpad, a.group, cs);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D, int BITS, bool JOINT>
static int launch(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                  const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    auto kern = decompress_kernel<D, BITS, JOINT>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), kDecompressSmem)) return NQ_ERR_CUDA;
    const int64_t items = work_items(a, a.slices, kTileRows, cs);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern), kDecompressSmem);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, kDecompressSmem, a.stream>>>(idx, coset, scales, rope, map, a.slices, a.tokens,
                                                        a.tpad, a.group, cs);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D, int BITS, bool JOINT>
static int launch_keys(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                       const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    auto kern = decompress_key_kernel<D, BITS, JOINT>;
    constexpr int smem = KeyStage<D>::SMEM;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem)) return NQ_ERR_CUDA;
    const int64_t ngroups = (a.slices + kKeyWarps - 1) / kKeyWarps;
    const int64_t items = work_items(a, ngroups, kTileRows, cs);
    if (items == 0) return NQ_OK;
    const int cap = grid_capacity_threads(reinterpret_cast<const void*>(kern), smem, kKeyThreads);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(items, cap));
    kern<<<grid, kKeyThreads, smem, a.stream>>>(idx, coset, scales, rope, map, a.slices, a.tokens, a.tpad,
                                                a.group, cs);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

// The starting sums of the groups of a delta-coded tensor whose chains are
// longer than one group: group totals, then the chain scan.
template <int BITS, int RB, int R>
static int launch_chain_sums(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const ChainState& cs) {
    const uint64_t groups = uint64_t(a.slices) * cs.geo.cps * cs.geo.gpc;
    if (groups == 0) return NQ_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NQ_ERR_CUDA;
    const int cap = 8 * sms;  // blocks of 8 warps, 8 resident per SM (the kernels hold few registers)
    int grid = int(std::min<uint64_t>(groups, uint64_t(cap)));  // a block per group
    if (a.stages & kStageRunTotals) {
        delta_group_kernel<BITS, RB, R><<<grid, kGroupWarps * 32, 0, a.stream>>>(idx, coset, a.slices, a.tpad,
                                                                                 cs.geo, cs.gsum, cs.slot_words);
        if (cudaGetLastError() != cudaSuccess) return NQ_ERR_CUDA;
    }
    if (!(a.stages & kStageChainScan)) return NQ_OK;
    const uint64_t chains = uint64_t(a.slices) * cs.geo.cps;
    grid = int(std::min<uint64_t>((chains + 7) / 8, uint64_t(cap)));
    delta_chain_kernel<BITS, RB><<<grid, 256, 0, a.stream>>>(a.slices, cs.geo, cs.gsum, cs.gexcl, cs.slot_words,
                                                             coset != nullptr);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D, int BITS, bool JOINT>
static int launch_any(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                      const float4* rope, const CUtensorMap& map, int max_bits) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int RB = DP * BITS / 8;
    constexpr int R = D == 64 ? kPairRows : kTileRows;
    ChainState cs;
    if (a.delta_chunk > 0) {
        const ChainPlan cp = chain_plan(a.slices, a.tokens, D, max_bits, a.delta_chunk);
        cs.delta = true;
        cs.geo = cp.geo;
        cs.slot_words = cp.slot_words;
        if (cp.total > 0) {  // chains longer than a group: starting sums from the workspace
            if (a.workspace == nullptr) return NQ_ERR_ARG;
            cs.gsum = reinterpret_cast<uint32_t*>(a.workspace + cp.gsum);
            cs.gexcl = reinterpret_cast<uint32_t*>(a.workspace + cp.gexcl);
            if (a.stages & (kStageRunTotals | kStageChainScan)) {
                const int st = launch_chain_sums<BITS, RB, R>(a, idx, coset, cs);
                if (st != NQ_OK) return st;
            }
        }
    }
    if (!(a.stages & kStageDecode)) return NQ_OK;
    if constexpr (D != 64) {
        if (rope != nullptr) return launch_keys<D, BITS, JOINT>(a, idx, coset, scales, rope, map, cs);
        return launch<D, BITS, JOINT>(a, idx, coset, scales, rope, map, cs);
    } else {
        return launch_pair<D, BITS, JOINT>(a, idx, coset, scales, rope, map, cs);
    }
}

template <int D>
static int dispatch_bits(const LaunchArgs& a, int bits, int max_bits, const uint8_t* idx, const uint16_t* coset,
                         const __half* scales, const float4* rope, const CUtensorMap& map) {
    // no coset words: the strict joint format, whose block codes carry the coset bits
    const bool joint = coset == nullptr;
    switch (bits) {
        case 2:
            return joint ? launch_any<D, 2, true>(a, idx, coset, scales, rope, map, max_bits)
                         : launch_any<D, 2, false>(a, idx, coset, scales, rope, map, max_bits);
        case 3:
            return joint ? launch_any<D, 3, true>(a, idx, coset, scales, rope, map, max_bits)
                         : launch_any<D, 3, false>(a, idx, coset, scales, rope, map, max_bits);
        case 4:
            return joint ? launch_any<D, 4, true>(a, idx, coset, scales, rope, map, max_bits)
                         : launch_any<D, 4, false>(a, idx, coset, scales, rope, map, max_bits);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

int launch_decompress_tensor(const LaunchArgs& a, int head_dim, int bits, int max_bits, const uint8_t* idx,
                             const uint16_t* coset, const uint16_t* scales, const float* rope, void* x_out) {
    CUtensorMap map;
    const int box_rows = head_dim != 64 ? kTileRows : kPairRows;
    if (!make_row_tile_map(&map, x_out, head_dim, a.tokens, a.slices, box_rows)) return NQ_ERR_CUDA;
    const __half* sh = reinterpret_cast<const __half*>(scales);
    const float4* r = reinterpret_cast<const float4*>(rope);
    switch (head_dim) {
        case 64:
            return dispatch_bits<64>(a, bits, max_bits, idx, coset, sh, r, map);
        case 96:
            return dispatch_bits<96>(a, bits, max_bits, idx, coset, sh, r, map);
        case 128:
            return dispatch_bits<128>(a, bits, max_bits, idx, coset, sh, r, map);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq
