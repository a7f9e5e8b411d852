// nq_compress.cu -- fused compression kernel: fp16 row -> RoPE removal (keys)
// -> zero-padded Hadamard -> group scale -> E8 nearest point -> b-bit codes ->
// temporal delta -> idx / coset / scale sections.
//
// Layout of the work: a warp owns 32 consecutive tokens of one (layer, batch,
// head) slice (a tile) and lane r owns token row r, in registers, so the
// Hadamard transform, the group scale and the E8 search need no shuffles; the
// previous token's codes for the delta come from the neighbouring lane.  The
// tiles are streamed through a 3-stage shared-memory ring per warp, filled by
// coalesced 16-byte cp.async copies two tiles ahead of the one being computed.
// The grid is one resident block per SM; warps take work items
// (slice, chunk of delta_chunk tokens, or 32 tokens without delta)
// round-robin.
#include "nq_internal.h"

namespace nq {

constexpr int kStages = 3;
constexpr int kCompressSmem = kWarpsPerBlock * kStages * kTileBytes;

// Copy the fp16 rows of a tile into a stage; rows past the chunk are zeros.
template <int D>
__device__ __forceinline__ void load_tile(const __half* __restrict__ x, const TileWalk& w, uint32_t stage,
                                          int lane) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    const int nvalid = min(kTileRows, w.t_end - w.t0);
    const __half* base = x + (w.slice * w.tokens + w.t0) * int64_t(D);
#pragma unroll
    for (int i = 0; i < CPR; ++i) {
        const int g = lane + 32 * i;
        const int r = g / CPR;
        const int c = g - r * CPR;
        const bool ok = r < nvalid;
        cp_async16(stage + swz(r, c), ok ? base + 8 * g : base, ok ? 16 : 0);
    }
}

template <int D, int BITS, bool STRICT>
__global__ void __launch_bounds__(kThreads, 1)
    compress_kernel(const __half* __restrict__ x, const float4* __restrict__ rope, int64_t slices,
                    int tokens, int tpad, int group, int chunk, bool delta, uint8_t* __restrict__ idx,
                    uint16_t* __restrict__ coset, __half* __restrict__ scales) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    constexpr int NSUB = DP / 32;
    using C = Code<BITS>;
    using RP = RowPack<BITS, NB>;
    constexpr int RB = DP * BITS / 8;  // idx bytes per row
    constexpr float STEP = float(DP) * C::H;

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem) + (threadIdx.x >> 5) * (kStages * kTileBytes);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int nsc = DP / group;

    TileWalk cur(warp, nwarps, slices, tokens, chunk);
    TileWalk pre = cur;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (pre.valid()) {
            load_tile<D>(x, pre, ring + s * kTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
    }

    unsigned carry[NB];
    unsigned carry_c = 0;
#pragma unroll
    for (int k = 0; k < NB; ++k) carry[k] = 0;

    for (int i = 0; cur.valid(); ++i) {
        if (pre.valid()) {
            load_tile<D>(x, pre, ring + ((i + kStages - 1) % kStages) * kTileBytes, lane);
            pre.next();
        }
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint32_t stage = ring + (i % kStages) * kTileBytes;

        const int t = cur.t0 + lane;
        const bool active = t < cur.t_end;

        // ---- the lane's row from the stage (fp16 -> fp32), zero padding to DP
        float y[DP];
#pragma unroll
        for (int q = 0; q < D / 8; ++q) h8_to_f(lds128(stage + swz(lane, q)), &y[8 * q]);
#pragma unroll
        for (int j = D; j < DP; ++j) y[j] = 0.0f;
        __syncwarp();  // every lane has its row: the stage may be refilled

        // ---- RoPE removal on keys: rotate each (i, i + D/2) pair by -angle
        if (rope != nullptr) {
            // table layout [D/4][tokens] float4: lanes read consecutive tokens
            const float4* cs = rope + (active ? t : cur.t_begin);
#pragma unroll
            for (int q = 0; q < D / 4; ++q) {
                const float4 v = __ldg(cs + int64_t(q) * tokens);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int j = 2 * q + p;
                    const float c = p ? v.z : v.x, s = p ? v.w : v.y;
                    const float a = y[j], b = y[j + D / 2];
                    y[j] = __fmaf_rn(a, c, __fmul_rn(b, s));
                    y[j + D / 2] = __fmaf_rn(b, c, -__fmul_rn(a, s));
                }
            }
        }

        // ---- Hadamard rotation (compression stage order)
        fwht_forward<DP>(y);

        // ---- group absmax -> fp16 scale -> reciprocal (per 32-subgroup)
        float amax[NSUB];
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
            float m = 0.0f;
#pragma unroll
            for (int j = 32 * s; j < 32 * s + 32; j += 2) m = fmax3(m, fabsf(y[j]), fabsf(y[j + 1]));
            amax[s] = m;
        }
        if (group >= 64) {
#pragma unroll
            for (int s = 0; s < NSUB; s += 2) amax[s] = amax[s + 1] = fmaxf(amax[s], amax[s + 1]);
        }
        if (group >= 128 && NSUB == 4) {
            const float m = fmaxf(amax[0], amax[2]);
#pragma unroll
            for (int s = 0; s < NSUB; ++s) amax[s] = m;
        }
        unsigned short sc[NSUB];
        float inv[NSUB];
        bool fast = true;
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
            sc[s] = group_scale(amax[s], STEP);
            const float scf = __half2float(__ushort_as_half(sc[s]));
            inv[s] = sc[s] ? __frcp_rn(__fmul_rn(scf, float(DP))) : 0.0f;
            fast = fast && (__fmul_rn(amax[s], inv[s]) < C::H);
        }

        // ---- E8 nearest point per 8-block -> block codes
        unsigned blk[NB];
        unsigned cw = 0;
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            float u[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) u[j] = __fmul_rn(y[8 * k + j], inv[k / 4]);
            unsigned c;
            if (!(fast && e8_fast<BITS, STRICT>(u, blk[k], c))) {
                const uint2 res = e8_slow<BITS, STRICT>(make_float4(u[0], u[1], u[2], u[3]),
                                                        make_float4(u[4], u[5], u[6], u[7]));
                blk[k] = res.x;
                c = res.y;
            }
            cw |= c << k;
        }

        // ---- temporal delta against the previous token of the chunk
        if (delta) {
            const bool first = cur.t0 == cur.t_begin;
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                unsigned prev = __shfl_up_sync(kFull, blk[k], 1);
                const unsigned last = __shfl_sync(kFull, blk[k], 31);
                if (lane == 0) prev = first ? 0u : carry[k];
                if (t != cur.t_begin) blk[k] = swar_sub<BITS>(blk[k], prev);
                carry[k] = last;  // raw codes of the tile's last token
            }
            unsigned pc = __shfl_up_sync(kFull, cw, 1);
            const unsigned lastc = __shfl_sync(kFull, cw, 31);
            if (lane == 0) pc = first ? 0u : carry_c;
            if (t != cur.t_begin) cw ^= pc;
            carry_c = lastc;
        }

        // ---- store the row's record (padding rows past the slice get zeros)
        if (!active) {
#pragma unroll
            for (int k = 0; k < NB; ++k) blk[k] = 0;
            cw = 0;
#pragma unroll
            for (int s = 0; s < NSUB; ++s) sc[s] = 0;
        }
        const int64_t rrow = cur.slice * tpad + t;
        unsigned w[RP::WORDS];
        RP::pack(blk, w);
        uint8_t* dst = idx + rrow * RB;
        if constexpr (RB % 16 == 0) {
#pragma unroll
            for (int q = 0; q < RB / 16; ++q)
                st_stream(reinterpret_cast<uint4*>(dst) + q,
                          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
        } else {
#pragma unroll
            for (int q = 0; q < RB / 8; ++q) reinterpret_cast<uint2*>(dst)[q] = make_uint2(w[2 * q], w[2 * q + 1]);
        }
        coset[rrow] = uint16_t(cw);
        __half* sdst = scales + rrow * nsc;
        const int stride = group / 32;
        for (int s = 0, g = 0; s < NSUB; s += stride, ++g) sdst[g] = __ushort_as_half(sc[s]);

        cur.next();
    }
    cp_async_wait<0>();
}

template <int D, int BITS, bool STRICT>
static int launch(const LaunchArgs& a, const __half* x, const float4* rope, uint8_t* idx,
                  uint16_t* coset, __half* scales) {
    auto kern = compress_kernel<D, BITS, STRICT>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), kCompressSmem)) return NQ_ERR_CUDA;
    const int chunk = a.delta_chunk > 0 ? a.delta_chunk : kTileRows;
    const int64_t items = a.slices * ((a.tokens + chunk - 1) / chunk);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern), kCompressSmem);
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, kCompressSmem, a.stream>>>(x, rope, a.slices, a.tokens, a.tpad, a.group, chunk,
                                                      a.delta_chunk > 0, idx, coset, scales);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D>
static int dispatch_bits(const LaunchArgs& a, int bits, bool strict, const __half* x,
                         const float4* rope, uint8_t* idx, uint16_t* coset, __half* scales) {
#define NQ_CASE(B)                                                         \
    case B:                                                                \
        return strict ? launch<D, B, true>(a, x, rope, idx, coset, scales) \
                      : launch<D, B, false>(a, x, rope, idx, coset, scales);
    switch (bits) {
        NQ_CASE(2)
        NQ_CASE(3)
        NQ_CASE(4)
        default:
            return NQ_ERR_UNSUPPORTED;
    }
#undef NQ_CASE
}

int launch_compress_tensor(const LaunchArgs& a, int head_dim, int bits, bool strict,
                           const void* x, const float* rope, uint8_t* idx, uint16_t* coset,
                           uint16_t* scales) {
    const __half* xh = static_cast<const __half*>(x);
    const float4* r = reinterpret_cast<const float4*>(rope);
    __half* sh = reinterpret_cast<__half*>(scales);
    switch (head_dim) {
        case 64:
            return dispatch_bits<64>(a, bits, strict, xh, r, idx, coset, sh);
        case 96:
            return dispatch_bits<96>(a, bits, strict, xh, r, idx, coset, sh);
        case 128:
            return dispatch_bits<128>(a, bits, strict, xh, r, idx, coset, sh);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq
