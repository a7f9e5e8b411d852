// nq_compress.cu -- fused compression kernel: fp16 row -> RoPE removal (keys)
// -> zero-padded Hadamard -> group scale -> E8 nearest point -> b-bit codes ->
// temporal delta -> idx / coset / scale sections.
//
// One thread owns one row (one head_dim vector) in registers, so the whole
// transform needs no shuffles or shared memory; a warp owns 32 consecutive
// tokens of one (layer, batch, head) slice, so its loads and stores cover
// contiguous memory and the previous token's codes (for the delta) come from
// the neighbouring lane.  Work items are (slice, chunk of delta_chunk tokens,
// or 32 tokens without delta), taken round-robin by all warps of a grid sized
// to the resident capacity of the GPU.
#include "nq_internal.h"

namespace nq {

template <int D, int BITS, bool STRICT>
__global__ void __launch_bounds__(kThreads, 1)
    compress_kernel(const __half* __restrict__ x, const float4* __restrict__ rope, int64_t slices,
                    int tokens, int group, int chunk, bool delta, uint8_t* __restrict__ idx,
                    uint16_t* __restrict__ coset, __half* __restrict__ scales) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    constexpr int NSUB = DP / 32;
    using C = Code<BITS>;
    using RP = RowPack<BITS, NB>;
    constexpr int RB = DP * BITS / 8;  // idx bytes per row
    constexpr float STEP = float(DP) * C::H;

    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int nchunks = (tokens + chunk - 1) / chunk;
    const int64_t items = slices * nchunks;
    const int nsc = DP / group;

    for (int64_t item = warp; item < items; item += nwarps) {
        const int64_t slice = item / nchunks;
        const int t_begin = int(item - slice * nchunks) * chunk;
        const int t_end = min(t_begin + chunk, tokens);
        unsigned carry[NB];
        uint16_t carry_c = 0;
#pragma unroll
        for (int k = 0; k < NB; ++k) carry[k] = 0;

        for (int t0 = t_begin; t0 < t_end; t0 += 32) {
            const int t = t0 + lane;
            const bool active = t < t_end;
            const int64_t row = slice * tokens + (active ? t : t_begin);

            // ---- load the row (fp16 -> fp32), zero padding to DP
            float y[DP];
            const uint4* src = reinterpret_cast<const uint4*>(x + row * D);
#pragma unroll
            for (int q = 0; q < D / 8; ++q) {
                uint4 v = ld_stream(src + q);
                h8_to_f(v, &y[8 * q]);
            }
#pragma unroll
            for (int i = D; i < DP; ++i) y[i] = 0.0f;

            // ---- RoPE removal on keys: rotate each (i, i + D/2) pair by -angle
            if (rope != nullptr) {
                const float4* cs = rope + int64_t(active ? t : t_begin) * (D / 4);
#pragma unroll
                for (int q = 0; q < D / 4; ++q) {
                    float4 v = __ldg(cs + q);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int i = 2 * q + p;
                        const float c = p ? v.z : v.x, s = p ? v.w : v.y;
                        const float a = y[i], b = y[i + D / 2];
                        y[i] = __fmaf_rn(a, c, __fmul_rn(b, s));
                        y[i + D / 2] = __fmaf_rn(b, c, -__fmul_rn(a, s));
                    }
                }
            }

            // ---- Hadamard rotation
            fwht<DP>(y);

            // ---- group absmax -> fp16 scale -> reciprocal (per 32-subgroup)
            float amax[NSUB];
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
                float m = 0.0f;
#pragma unroll
                for (int i = 32 * s; i < 32 * s + 32; ++i) m = fmaxf(m, fabsf(y[i]));
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
                if (fast) {
                    blk[k] = e8_fast<BITS, STRICT>(u, c);
                } else {
                    float r[8];
                    c = (unsigned)e8_general(u, STRICT, C::HI0, C::H, r);
                    blk[k] = pack_point<BITS>(r, int(c));
                }
                cw |= c << k;
            }

            // ---- temporal delta against the previous token of the chunk
            if (delta) {
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    unsigned prev = __shfl_up_sync(kFull, blk[k], 1);
                    const unsigned last = __shfl_sync(kFull, blk[k], 31);
                    if (lane == 0) prev = carry[k];
                    const unsigned raw = blk[k];
                    if (t != t_begin) blk[k] = swar_sub<BITS>(raw, prev);
                    carry[k] = last;
                }
                unsigned pc = __shfl_up_sync(kFull, cw, 1);
                const unsigned lastc = __shfl_sync(kFull, cw, 31);
                if (lane == 0) pc = carry_c;
                if (t != t_begin) cw ^= pc;
                carry_c = uint16_t(lastc & 0xffffu);
                // NB: carry holds raw codes; the xor above used the raw pc.
            }

            // ---- store the row's record
            if (active) {
                unsigned w[RP::WORDS];
                RP::pack(blk, w);
                uint8_t* dst = idx + row * RB;
                if constexpr (RB % 16 == 0) {
#pragma unroll
                    for (int q = 0; q < RB / 16; ++q)
                        st_stream(reinterpret_cast<uint4*>(dst) + q,
                                  make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
                } else {
#pragma unroll
                    for (int q = 0; q < RB / 8; ++q)
                        reinterpret_cast<uint2*>(dst)[q] = make_uint2(w[2 * q], w[2 * q + 1]);
                }
                coset[row] = uint16_t(cw);
                __half* sdst = scales + row * nsc;
                const int stride = group / 32;
                for (int s = 0, g = 0; s < NSUB; s += stride, ++g) sdst[g] = __ushort_as_half(sc[s]);
            }
        }
    }
}

template <int D, int BITS, bool STRICT>
static int launch(const LaunchArgs& a, const __half* x, const float4* rope, uint8_t* idx,
                  uint16_t* coset, __half* scales) {
    auto kern = compress_kernel<D, BITS, STRICT>;
    const int chunk = a.delta_chunk > 0 ? a.delta_chunk : 32;
    const int64_t items = a.slices * ((a.tokens + chunk - 1) / chunk);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern));
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, 0, a.stream>>>(x, rope, a.slices, a.tokens, a.group, chunk,
                                          a.delta_chunk > 0, idx, coset, scales);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D>
static int dispatch_bits(const LaunchArgs& a, int bits, bool strict, const __half* x,
                         const float4* rope, uint8_t* idx, uint16_t* coset, __half* scales) {
#define NQ_CASE(B)                                                                     \
    case B:                                                                            \
        return strict ? launch<D, B, true>(a, x, rope, idx, coset, scales)             \
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
