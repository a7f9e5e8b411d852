// nq_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/nq.h"
#include "nq_device.cuh"

namespace nq {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

template <int D>
struct PaddedDim {
    static constexpr int value = D <= 64 ? 64 : 128;
};

struct LaunchArgs {
    int64_t slices;  // layers * batch * kv_heads
    int tokens;
    int tpad;        // record rows per slice: tokens rounded up to a multiple of 32
    int group;
    int delta_chunk;
    cudaStream_t stream;
};

// Blocks of kThreads that fit on the current device at once for `kernel` with
// `smem` bytes of dynamic shared memory; -1 when it cannot be queried.
int grid_capacity(const void* kernel, int smem);
int grid_capacity_threads(const void* kernel, int smem, int threads);

// Allow `kernel` `smem` bytes of dynamic shared memory on the current device
// (once per device); false on a CUDA error.
bool ensure_smem(const void* kernel, int smem);

// TMA map of an fp16 [slices][tokens][head_dim] tensor as 3-D tiles of
// 64 columns x box_rows tokens x 1 slice, 128-byte swizzle.  false on failure.
bool make_row_tile_map(CUtensorMap* map, void* base, int head_dim, int tokens, int64_t slices, int box_rows);

// One tensor (K or V) of a call.  mode: 0 relaxed, 1 strict, 2 strict joint
// format (coset == nullptr: no coset words).  rope: device table or nullptr.
int launch_compress_tensor(const LaunchArgs& a, int head_dim, int bits, int mode, const void* x,
                           const float* rope, uint8_t* idx, uint16_t* coset, uint16_t* scales);
// coset == nullptr: the joint format.
int launch_decompress_tensor(const LaunchArgs& a, int head_dim, int bits, const uint8_t* idx,
                             const uint16_t* coset, const uint16_t* scales, const float* rope,
                             void* x_out);
int launch_roundtrip_tensor(const LaunchArgs& a, int head_dim, int bits, bool strict, const void* x,
                            const float* rope, void* x_out);
// Adds one tensor's symbol counts to counts[0, NQ_HIST_BINS) (zeroed by the caller).
int launch_code_histogram(const LaunchArgs& a, int padded_dim, int bits, const uint8_t* idx,
                          const uint16_t* coset, uint64_t* counts);

int launch_e8_nearest(const float* u, float* out, int64_t n_blocks, bool strict, int bits,
                      cudaStream_t stream);

}  // namespace nq
