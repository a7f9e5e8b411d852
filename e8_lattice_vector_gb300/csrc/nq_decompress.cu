// nq_decompress.cu -- fused decompression kernel: idx / coset / scale sections
// -> undo temporal delta -> unpack -> unscale -> inverse Hadamard -> RoPE
// re-apply (keys) -> fp16 rows.
//
// Same work layout as compression: one thread per row, a warp per 32
// consecutive tokens of a slice, a chunk of delta_chunk tokens per work item.
// The delta is undone by an inclusive warp scan (field-wise addition modulo
// 2^b, exclusive-or for the coset word) plus the running total of the chunk's
// earlier tiles.
#include "nq_internal.h"

namespace nq {

template <int D, int BITS>
__global__ void __launch_bounds__(kThreads, 1)
    decompress_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset,
                      const __half* __restrict__ scales, const float4* __restrict__ rope,
                      int64_t slices, int tokens, int group, int chunk, bool delta,
                      __half* __restrict__ x) {
    constexpr int DP = PaddedDim<D>::value;
    constexpr int NB = DP / 8;
    using C = Code<BITS>;
    using RP = RowPack<BITS, NB>;
    constexpr int RB = DP * BITS / 8;

    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int nchunks = (tokens + chunk - 1) / chunk;
    const int64_t items = slices * nchunks;
    const int nsc = DP / group;
    const int gshift = group == 32 ? 5 : (group == 64 ? 6 : 7);

    for (int64_t item = warp; item < items; item += nwarps) {
        const int64_t slice = item / nchunks;
        const int t_begin = int(item - slice * nchunks) * chunk;
        const int t_end = min(t_begin + chunk, tokens);
        unsigned carry[NB];
        unsigned carry_c = 0;
#pragma unroll
        for (int k = 0; k < NB; ++k) carry[k] = 0;

        for (int t0 = t_begin; t0 < t_end; t0 += 32) {
            const int t = t0 + lane;
            const bool active = t < t_end;
            const int64_t row = slice * tokens + (active ? t : t_begin);

            // ---- load the record
            unsigned w[RP::WORDS];
            const uint8_t* src = idx + row * RB;
            if constexpr (RB % 16 == 0) {
#pragma unroll
                for (int q = 0; q < RB / 16; ++q) {
                    uint4 v = ld_stream(reinterpret_cast<const uint4*>(src) + q);
                    w[4 * q] = v.x;
                    w[4 * q + 1] = v.y;
                    w[4 * q + 2] = v.z;
                    w[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < RB / 8; ++q) {
                    uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + q);
                    w[2 * q] = v.x;
                    w[2 * q + 1] = v.y;
                }
            }
            unsigned blk[NB];
            RP::unpack(w, blk);
            unsigned cw = __ldg(coset + row);

            // ---- undo the temporal delta: inclusive scan over the tile + carry
            if (delta) {
#pragma unroll
                for (int off = 1; off < 32; off *= 2) {
#pragma unroll
                    for (int k = 0; k < NB; ++k) {
                        const unsigned v = __shfl_up_sync(kFull, blk[k], off);
                        if (lane >= off) blk[k] = swar_add<BITS>(blk[k], v);
                    }
                    const unsigned vc = __shfl_up_sync(kFull, cw, off);
                    if (lane >= off) cw ^= vc;
                }
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    blk[k] = swar_add<BITS>(blk[k], carry[k]);
                    carry[k] = __shfl_sync(kFull, blk[k], 31);
                }
                cw ^= carry_c;
                carry_c = __shfl_sync(kFull, cw, 31);
            }

            // ---- unpack, unscale: y = (code - offset) * scale  (exact)
            float scf[DP / 32];
#pragma unroll
            for (int s = 0; s < DP / 32; ++s)
                scf[s] = __half2float(__ldg(scales + row * nsc + ((32 * s) >> gshift)));
            float y[DP];
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const float off = ((cw >> k) & 1u) ? C::H : C::HI0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const unsigned m = (blk[k] >> (j * BITS)) & C::MASK;
                    const float mf = __fsub_rn(__uint_as_float(0x4B000000u | m), 8388608.0f);
                    y[8 * k + j] = __fmul_rn(__fsub_rn(mf, off), scf[k / 4]);
                }
            }

            // ---- inverse Hadamard: x = H (r * sc)
            fwht<DP>(y);

            // ---- RoPE re-apply on keys: rotate each (i, i + D/2) pair by +angle
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
                        y[i] = __fmaf_rn(a, c, -__fmul_rn(b, s));
                        y[i + D / 2] = __fmaf_rn(b, c, __fmul_rn(a, s));
                    }
                }
            }

            // ---- fp16 store
            if (active) {
                uint4* dst = reinterpret_cast<uint4*>(x + row * D);
#pragma unroll
                for (int q = 0; q < D / 8; ++q) st_stream(dst + q, f_to_h8(&y[8 * q]));
            }
        }
    }
}

template <int D, int BITS>
static int launch(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset,
                  const __half* scales, const float4* rope, __half* x) {
    auto kern = decompress_kernel<D, BITS>;
    const int chunk = a.delta_chunk > 0 ? a.delta_chunk : 32;
    const int64_t items = a.slices * ((a.tokens + chunk - 1) / chunk);
    const int64_t want = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (want == 0) return NQ_OK;
    const int cap = grid_capacity(reinterpret_cast<const void*>(kern));
    if (cap <= 0) return NQ_ERR_CUDA;
    const int grid = int(std::min<int64_t>(want, cap));
    kern<<<grid, kThreads, 0, a.stream>>>(idx, coset, scales, rope, a.slices, a.tokens, a.group,
                                          chunk, a.delta_chunk > 0, x);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

template <int D>
static int dispatch_bits(const LaunchArgs& a, int bits, const uint8_t* idx, const uint16_t* coset,
                         const __half* scales, const float4* rope, __half* x) {
    switch (bits) {
        case 2:
            return launch<D, 2>(a, idx, coset, scales, rope, x);
        case 3:
            return launch<D, 3>(a, idx, coset, scales, rope, x);
        case 4:
            return launch<D, 4>(a, idx, coset, scales, rope, x);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

int launch_decompress_tensor(const LaunchArgs& a, int head_dim, int bits, const uint8_t* idx,
                             const uint16_t* coset, const uint16_t* scales, const float* rope,
                             void* x_out) {
    const __half* sh = reinterpret_cast<const __half*>(scales);
    const float4* r = reinterpret_cast<const float4*>(rope);
    __half* xh = static_cast<__half*>(x_out);
    switch (head_dim) {
        case 64:
            return dispatch_bits<64>(a, bits, idx, coset, sh, r, xh);
        case 96:
            return dispatch_bits<96>(a, bits, idx, coset, sh, r, xh);
        case 128:
            return dispatch_bits<128>(a, bits, idx, coset, sh, r, xh);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq
