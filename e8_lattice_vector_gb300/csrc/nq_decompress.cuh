// nq_decompress.cuh -- fused decompression kernels: idx / coset / scale
// sections -> undo temporal delta -> unpack -> unscale -> inverse Hadamard ->
// RoPE re-apply (keys) -> fp16 rows.
//
// head_dim 96 / 128: a warp per 32-token tile of a slice, lane r owns row r
// (one thread per row; for the decode this beats two threads per row).  A
// tile's records (idx rows, coset words, scales) are contiguous and 16-byte
// aligned thanks to the per-slice padding of the record rows, so they stream
// through a 3-stage shared-memory ring by cp.async; keys run in blocks of
// warps that also stage the tile's RoPE table rows once for the block.
// Without a temporal delta every tile is a work item; with one, a chain of at
// most one chunk, or else a run of up to 32 consecutive tiles of a chain, is,
// walked in order (the kernels are instantiated with and without a delta).
// The delta is undone in place on the record tile, column-wise (field-wise
// addition modulo 2^b), plus the running sum of the chain's earlier rows,
// carried in registers from tile to tile; a run that does not start its chain
// takes its starting sum from the workspace, where two light passes over the
// idx section leave it (nq_chain.cuh).  Three-bit tiles come back unpacked, one
// word per block code.  Coset words ride on the column scan (an exclusive-or
// warp scan for three-bit tiles).  The reconstructed fp16 rows are written
// into a swizzled shared-memory tile and leave by one TMA tensor store per 64
// columns, which clips the rows past the end of the slice and the columns past
// head_dim.  (head_dim 64, two threads per row: nq_decompress.cu.)
#pragma once

#include <type_traits>

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

// Running sums of the N = 2^k values v[i][n] (i = 0..N-1) of a lane's column,
// offset by a value that depends on their total, in the Brent-Kung form: the
// up-sweep leaves the total in v[N-1] after k levels (a short dependency chain
// for the scan of the totals that follows); the offset then goes into the k + 1
// prefixes the up-sweep has completed (v[2^j - 1], and v[0]) and the
// down-sweep carries it into the rest.  As many additions as the serial
// running sum plus one offset per value.
template <typename DU, int N, int NV>
__device__ __forceinline__ void scan_up(unsigned (&v)[N][NV], int n) {
#pragma unroll
    for (int w = 1; w < N; w *= 2)
#pragma unroll
        for (int i = 2 * w - 1; i < N; i += 2 * w) v[i][n] = DU::add(v[i][n], v[i - w][n]);
}
template <typename DU, int N, int NV>
__device__ __forceinline__ void scan_down(unsigned (&v)[N][NV], int n, unsigned off) {
    v[0][n] = DU::add(v[0][n], off);
#pragma unroll
    for (int k = 1; k < N; k *= 2) v[2 * k - 1][n] = DU::add(v[2 * k - 1][n], off);
#pragma unroll
    for (int w = N / 4; w >= 1; w /= 2)
#pragma unroll
        for (int i = 3 * w - 1; i < N; i += 2 * w) v[i][n] = DU::add(v[i][n], v[i - w][n]);
}

// LOWLAT trades additions for a shorter chain: the total by a separate tree
// while the serial running sums proceed beside it, and the offset added to
// every value (N - 1 more additions than the Brent-Kung form; the chain from
// the loads to the offset log2 N levels long, the one after it a single
// addition).  For
// decoders whose warps wait for each other at a barrier every tile, where the
// chain is not hidden by other warps' work.
template <typename DU, bool LOWLAT, int N, int NV>
__device__ __forceinline__ unsigned scan_total(unsigned (&v)[N][NV], int n) {
    if constexpr (LOWLAT) {
        unsigned t[N];
#pragma unroll
        for (int i = 0; i < N; ++i) t[i] = v[i][n];
#pragma unroll
        for (int w = 1; w < N; w *= 2)
#pragma unroll
            for (int i = 0; i + w < N; i += 2 * w) t[i] = DU::add(t[i], t[i + w]);
#pragma unroll
        for (int i = 1; i < N; ++i) v[i][n] = DU::add(v[i][n], v[i - 1][n]);
        return t[0];
    } else {
        scan_up<DU>(v, n);
        return v[N - 1][n];
    }
}
template <typename DU, bool LOWLAT, int N, int NV>
__device__ __forceinline__ void scan_offset(unsigned (&v)[N][NV], int n, unsigned off) {
    if constexpr (LOWLAT) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i][n] = DU::add(v[i][n], off);
    } else {
        scan_down<DU>(v, n, off);
    }
}

// The delta is undone in place on the 32-row idx tile in shared memory, down
// its columns: lane l takes column unit l % NU (a 32-bit word of 16 two-bit or
// 8 four-bit fields, or a 3-word group holding four 24-bit block codes at 3
// bits: the 16-row tiles of head_dim 64; 32-row three-bit tiles go by
// undelta_tile24) of the rows of segment l / NU; it forms the running field-wise sums
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
template <int BITS, int RB, int ROWS = 32, bool COSET = false, bool LOWLAT = false>
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
    unsigned run[NV], ex[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) run[n] = scan_total<DU, LOWLAT>(v, n);
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
    for (int n = 0; n < NV; ++n) scan_offset<DU, LOWLAT>(v, n, ex[n]);
#pragma unroll
    for (int i = 0; i < RPS; ++i) DU::store(base + i * RB, v[i]);
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

// Three-bit codes, 32-row tiles: a row holds sixteen 24-bit block codes,
// block c at byte 3c (RB = 48).  Lane l takes block column c = l % 16 of the
// rows of half h = l / 16, so each lane reads one byte-aligned code per row
// (two words and a byte permutation) and no code is shared between lanes.
// The 16 running sums of a column half go by scan_up / scan_down, with one
// shuffle for the lower half's total.  The codes go back unpacked, one word
// per block code: row r at 64 r, its 16-byte chunks rotated by (r / 2) % 4 so
// that decode_row's quarter-warp reads of whole rows hit distinct banks; the
// region holds 32 * 64 = 2048 bytes, which the stage's idx area provides.
// Coset words: an exclusive-or scan over the warp, lane l holding row l.
// carry: the lane's column code in the previous tile's last row.
template <bool COSET>
__device__ __forceinline__ void undelta_tile24(uint32_t rows, int lane, bool first, unsigned& carry,
                                               uint32_t cosets, unsigned* carry_c) {
    using DU = DeltaUnit<3>;
    constexpr int RB = 48;
    const int c = lane & 15, h = lane >> 4;
    const uint32_t off = 3u * uint32_t(c);
    const uint32_t src = rows + uint32_t(h * 16 * RB) + (off & ~3u);
    const unsigned sel = 0x3210u + 0x1111u * (off & 3u);  // bytes off..off+3 of the two words
    unsigned v[16][1];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i][0] = __byte_perm(lds32(src + i * RB), lds32(src + i * RB + 4), sel);
    // (the byte above the code is the next code's: the field-wise sums carry
    // only upward, so it never reaches the code's 24 bits, and the decoder
    // masks every field)
    unsigned cw = 0u;
    if constexpr (COSET) cw = lds16(cosets + 2 * lane);
    scan_up<DU>(v, 0);
    const unsigned lower = __shfl_sync(kFull, v[15][0], c);  // the lower half's column total
    unsigned ex = h ? lower : 0u;
    if (!first) ex = DU::add(ex, carry);
    if constexpr (COSET) {
#pragma unroll
        for (int d = 1; d < 32; d *= 2) {
            const unsigned t = __shfl_up_sync(kFull, cw, d);
            if (lane >= d) cw ^= t;
        }
        if (!first) cw ^= *carry_c;
    }
    scan_down<DU>(v, 0, ex);
    carry = __shfl_sync(kFull, v[15][0], 16 + c);
    __syncwarp();  // every lane has read its codes
    const uint32_t dst = rows + uint32_t(h * 16 * 64) + 4u * uint32_t(c & 3);
    const uint32_t q = uint32_t(c >> 2);
#pragma unroll
    for (int i = 0; i < 16; ++i) sts32(dst + i * 64 + 16u * (q ^ uint32_t((i >> 1) & 3)), v[i][0]);
    if constexpr (COSET) {
        sts16(cosets + 2 * lane, cw);
        *carry_c = __shfl_sync(kFull, cw, 31);
    }
}

// One record row (the lane's row of a 32-row record tile in `stage`) ->
// unscaled, inverse-transformed coordinates, before the RoPE re-apply.
template <int D, int BITS, bool JOINT, bool LOWLAT>
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
        if constexpr (BITS == 3) {  // the tile comes back unpacked (undelta_tile24)
            undelta_tile24<!JOINT>(stage + kRecIdx, lane, first, carry[0], stage + kRecCoset, &carry_c);
        } else {
            constexpr int NV = DeltaUnit<BITS>::NV;
            unsigned cu[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n) cu[n] = carry[n];
            undelta_tile<BITS, RB, 32, !JOINT, LOWLAT>(stage + kRecIdx, lane, first, cu, stage + kRecCoset, &carry_c);
#pragma unroll
            for (int n = 0; n < NV; ++n) carry[n] = cu[n];
        }
        __syncwarp();
    }

    // ---- the lane's record
    unsigned w[RP::WORDS];
    unsigned blk[NB];
    const bool unpacked = BITS == 3 && delta;
    if (unpacked) {  // row `lane` at 64 * lane, chunks rotated by (lane / 2) % 4
        const uint32_t row = stage + kRecIdx + 64u * uint32_t(lane);
        const uint32_t g = uint32_t(lane >> 1) & 3u;
#pragma unroll
        for (int q = 0; q < NB / 4; ++q) {
            const uint4 v = lds128(row + 16u * (uint32_t(q) ^ g));
            blk[4 * q] = v.x;
            blk[4 * q + 1] = v.y;
            blk[4 * q + 2] = v.z;
            blk[4 * q + 3] = v.w;
        }
    } else if constexpr (RB % 16 == 0) {
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
    if (!unpacked) RP::unpack(w, blk);

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

template <int D, int BITS, bool JOINT, bool DELTA>
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
                    if (cs.gexcl == nullptr)
                        first = true;
                    else if constexpr (BITS == 3)
                        load_group_carry24(cs, cur.G, lane & 15, carry[0], carry_c, !JOINT);
                    else
                        load_group_carry<BITS, RB>(cs, cur.G, lane % NU, carry, carry_c, !JOINT);
                }
            } else {
                first = cur.t0 == cur.t_begin();  // chains of one chunk: its first tile
            }
            const uint8_t* stage_gen = smem + (stage - smem_u32(smem));
            float y[DP];
            decode_row<D, BITS, JOINT, false>(stage, stage_gen, lane, nsc, gshift, DELTA, first, carry, carry_c, y);
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
    if constexpr (!DELTA)
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

template <int D, int BITS, bool JOINT, bool DELTA>
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
    // With a delta, the two- and four-bit instantiations keep the plain tile
    // walk compiled in beside the chain walks, the choice made at run time:
    // so built, the two-bit one measured 11 % faster on the Qwen2.5-14B-shaped
    // cache (4.22 -> 3.77 ms; the compiler schedules the kernel differently,
    // nothing else changes), the three-bit one 3 % slower.
    const bool delta = DELTA && (BITS == 3 || cs.delta);

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
                        if (cs.gexcl == nullptr)
                            first = true;
                        else if constexpr (BITS == 3)
                            load_group_carry24(cs, cur.slice_group(uint64_t(slice)), lane & 15, carry[0], carry_c,
                                               !JOINT);
                        else
                            load_group_carry<BITS, RB>(cs, cur.slice_group(uint64_t(slice)), lane % NU, carry, carry_c,
                                                       !JOINT);
                    }
                } else {
                    first = cur.t0 == cur.t_begin();
                }
                const uint32_t rec = stage + KS::TABLE + wib * kRecStage;
                float y[DP];
                decode_row<D, BITS, JOINT, true>(rec, gbase + (rec - base), lane, nsc, gshift, delta, first, carry,
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
    if (!delta)
        run(TileWalk(blockIdx.x, gridDim.x, ngroups, tokens, kTileRows));
    else if (cs.gexcl == nullptr)
        run(TileWalk(blockIdx.x, gridDim.x, ngroups, tokens, int(cs.geo.tpc) * kTileRows));
    else
        run(GroupWalk<kTileRows>(blockIdx.x, gridDim.x, ngroups, cs.geo));
    cp_async_wait<0>();
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Work items: single tiles without a delta, groups of a chain's tiles with
// one (units: slices, or the key kernel's groups of slices).
static int64_t work_items(const LaunchArgs& a, int64_t units, int rows, const ChainState& cs) {
    if (!cs.delta) return units * ((a.tokens + rows - 1) / rows);
    return units * int64_t(cs.geo.cps) * cs.geo.gpc;
}

template <int D, int BITS, bool JOINT, bool DELTA>
static int launch(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                  const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    auto kern = decompress_kernel<D, BITS, JOINT, DELTA>;
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

template <int D, int BITS, bool JOINT, bool DELTA>
static int launch_keys(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, const __half* scales,
                       const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    auto kern = decompress_key_kernel<D, BITS, JOINT, DELTA>;
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

// The decoders of head_dim 96 / 128 for one DELTA (keys when rope is set);
// each translation unit instantiates one of the two.
template <bool DELTA>
static int launch_wide_as(const LaunchArgs& a, int d, int bits, bool joint, const uint8_t* idx,
                          const uint16_t* coset, const __half* scales, const float4* rope, const CUtensorMap& map,
                          const ChainState& cs) {
    auto go = [&](auto dd, auto bb, auto jj) {
        constexpr int D = decltype(dd)::value;
        constexpr int BITS = decltype(bb)::value;
        constexpr bool JOINT = decltype(jj)::value;
        if (rope != nullptr) return launch_keys<D, BITS, JOINT, DELTA>(a, idx, coset, scales, rope, map, cs);
        return launch<D, BITS, JOINT, DELTA>(a, idx, coset, scales, rope, map, cs);
    };
    auto by_bits = [&](auto dd) {
        using T = std::true_type;
        using F = std::false_type;
        switch (bits) {
            case 2: return joint ? go(dd, std::integral_constant<int, 2>(), T()) : go(dd, std::integral_constant<int, 2>(), F());
            case 3: return joint ? go(dd, std::integral_constant<int, 3>(), T()) : go(dd, std::integral_constant<int, 3>(), F());
            case 4: return joint ? go(dd, std::integral_constant<int, 4>(), T()) : go(dd, std::integral_constant<int, 4>(), F());
            default: return int(NQ_ERR_UNSUPPORTED);
        }
    };
    if (d == 96) return by_bits(std::integral_constant<int, 96>());
    if (d == 128) return by_bits(std::integral_constant<int, 128>());
    return int(NQ_ERR_UNSUPPORTED);
}
int launch_wide_plain(const LaunchArgs& a, int d, int bits, bool joint, const uint8_t* idx, const uint16_t* coset,
                      const __half* scales, const float4* rope, const CUtensorMap& map, const ChainState& cs);
int launch_wide_delta(const LaunchArgs& a, int d, int bits, bool joint, const uint8_t* idx, const uint16_t* coset,
                      const __half* scales, const float4* rope, const CUtensorMap& map, const ChainState& cs);

}  // namespace nq
