// nq_stats.cu -- symbol statistics of a compressed buffer, for the entropy
// report: per tensor, how often each b-bit field value occurs in the idx
// section (these are the temporal-delta symbols when the delta is on), how
// often each byte value occurs there (the order-0 statistics a byte-level
// entropy coder would see), and how many blocks sit in each coset (in the
// strict joint format, where the coset bit is the top bit of the block code,
// that top bit as stored).  Only the record rows of real tokens are counted,
// not the padding rows.
//
// A thread takes whole record rows.  Field values are counted in registers by
// SWAR equality tests on the 8-field block codes (one popcount per symbol and
// block); bytes go to a shared-memory histogram; each block adds its totals to
// the caller's 64-bit counters once at the end.
#include "nq_internal.h"

namespace nq {

constexpr int kHistThreads = 256;

// Number of the 8 b-bit fields of `code` equal to s.
template <int BITS>
__device__ __forceinline__ unsigned count_symbol(unsigned code, unsigned s) {
    constexpr unsigned LOW = Code<BITS>::FIELD_HI >> (BITS - 1);  // bit j*b of every field
    const unsigned m = ~(code ^ (s * LOW));                        // 1 where the bits agree
    unsigned e = m;
#pragma unroll
    for (int i = 1; i < BITS; ++i) e &= m >> i;
    return __popc(e & LOW);
}

template <int BITS, int NB>
__global__ void __launch_bounds__(kHistThreads)
    code_hist_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ coset, int64_t slices,
                     int tokens, int tpad, unsigned long long* __restrict__ counts) {
    constexpr int L = 1 << BITS;
    constexpr int RB = NB * BITS;  // idx bytes per row
    constexpr int WORDS = RB / 4;
    __shared__ unsigned sh[NQ_HIST_BINS];
    for (int i = threadIdx.x; i < NQ_HIST_BINS; i += kHistThreads) sh[i] = 0;
    __syncthreads();

    unsigned fc[L];
#pragma unroll
    for (int s = 0; s < L; ++s) fc[s] = 0;
    unsigned ones = 0, blocks = 0;
    const int64_t rows = slices * tokens;
    for (int64_t row = int64_t(blockIdx.x) * kHistThreads + threadIdx.x; row < rows;
         row += int64_t(gridDim.x) * kHistThreads) {
        const int64_t sl = row / tokens;
        const int64_t rec = sl * tpad + (row - sl * tokens);
        const unsigned* src = reinterpret_cast<const unsigned*>(idx + rec * RB);
        unsigned w[WORDS];
#pragma unroll
        for (int q = 0; q < WORDS; ++q) w[q] = __ldg(src + q);
#pragma unroll
        for (int q = 0; q < WORDS; ++q) {
#pragma unroll
            for (int b = 0; b < 4; ++b) atomicAdd(&sh[16 + ((w[q] >> (8 * b)) & 255u)], 1u);
        }
        unsigned blk[NB];
        RowPack<BITS, NB>::unpack(w, blk);
#pragma unroll
        for (int k = 0; k < NB; ++k) {
#pragma unroll
            for (int s = 0; s < L - 1; ++s) fc[s] += count_symbol<BITS>(blk[k], unsigned(s));
        }
        if (coset != nullptr) {
            ones += __popc(unsigned(__ldg(coset + rec)) & ((1u << NB) - 1u));
        } else {  // joint format: the top bit of each block code
#pragma unroll
            for (int k = 0; k < NB; ++k) ones += (blk[k] >> (8 * BITS - 1)) & 1u;
        }
        blocks += NB;
    }
    unsigned rest = 8 * blocks;  // fields of the last symbol: all the others
#pragma unroll
    for (int s = 0; s < L - 1; ++s) rest -= fc[s];
    fc[L - 1] = rest;
#pragma unroll
    for (int s = 0; s < L; ++s)
        if (fc[s]) atomicAdd(&sh[s], fc[s]);
    if (blocks) {
        atomicAdd(&sh[NQ_HIST_BINS - 2], blocks - ones);
        atomicAdd(&sh[NQ_HIST_BINS - 1], ones);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NQ_HIST_BINS; i += kHistThreads)
        if (sh[i]) atomicAdd(&counts[i], static_cast<unsigned long long>(sh[i]));
}

template <int BITS, int NB>
static int launch_hist(const LaunchArgs& a, const uint8_t* idx, const uint16_t* coset, uint64_t* counts) {
    const int64_t rows = a.slices * a.tokens;
    // enough blocks that no block's shared 32-bit byte counters can overflow
    const int64_t want = (rows + kHistThreads - 1) / kHistThreads;
    const int64_t floor_blocks = std::max<int64_t>(2432, rows >> 24);
    const int grid = int(std::min<int64_t>(want, std::min<int64_t>(floor_blocks, int64_t(1) << 30)));
    code_hist_kernel<BITS, NB><<<grid, kHistThreads, 0, a.stream>>>(
        idx, coset, a.slices, a.tokens, a.tpad, reinterpret_cast<unsigned long long*>(counts));
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

int launch_code_histogram(const LaunchArgs& a, int padded_dim, int bits, const uint8_t* idx,
                          const uint16_t* coset, uint64_t* counts) {
    if (a.slices == 0 || a.tokens == 0) return NQ_OK;
    const bool p128 = padded_dim == 128;
    switch (bits) {
        case 2: return p128 ? launch_hist<2, 16>(a, idx, coset, counts) : launch_hist<2, 8>(a, idx, coset, counts);
        case 3: return p128 ? launch_hist<3, 16>(a, idx, coset, counts) : launch_hist<3, 8>(a, idx, coset, counts);
        case 4: return p128 ? launch_hist<4, 16>(a, idx, coset, counts) : launch_hist<4, 8>(a, idx, coset, counts);
        default: return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq
