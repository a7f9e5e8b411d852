// nq_decompress.cu -- the head_dim-64 decoder (two threads per row), the
// starting sums of long delta chains, and the dispatch of a decompression
// launch; the head_dim 96 / 128 decoders without a temporal delta are
// instantiated here, those with one in nq_decompress_delta.cu.
#include "nq_decompress.cuh"

namespace nq {

int launch_wide_plain(const LaunchArgs& a, int d, int bits, bool joint, const uint8_t* idx, const uint16_t* coset,
                      const __half* scales, const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    return launch_wide_as<false>(a, d, bits, joint, idx, coset, scales, rope, map, cs);
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
        return cs.delta ? launch_wide_delta(a, D, BITS, JOINT, idx, coset, scales, rope, map, cs)
                        : launch_wide_plain(a, D, BITS, JOINT, idx, coset, scales, rope, map, cs);
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
