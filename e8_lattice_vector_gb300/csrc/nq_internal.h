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

// Decompression with a temporal delta: the chained tiles of one tensor
// (tiles of R rows, tpc tiles per chain -- delta_chunk / R, a slice's last
// chain may be shorter) are decoded in runs of up to 32 consecutive tiles
// ("groups") that never cross a chain; a warp walks a group's tiles in order
// with the delta's running sum in registers.  A group that does not start its
// chain takes its starting sum from the workspace (nq_chain.cuh).
struct ChainGeom {
    uint32_t tiles;  // tiles per slice
    uint32_t tpc;    // tiles per chain
    uint32_t cps;    // chains per slice
    uint32_t gpc;    // groups per chain
};

// The decompression workspace: needed only when a chain is longer than one
// group (0 bytes otherwise); per group one slot of slot_words words (the idx
// row words, packed as in a record row, and a coset word, padded to 16 bytes
// and sized for the wider of the two bit widths) for the group's total and one
// for the sum of its chain's earlier groups, 256-byte aligned.
struct ChainPlan {
    ChainGeom geo{};
    int slot_words = 0;
    uint64_t groups = 0, gsum = 0, gexcl = 0, total = 0;
};

inline ChainPlan chain_plan(int64_t slices, int tokens, int head_dim, int max_bits, int delta_chunk) {
    ChainPlan c;
    if (delta_chunk <= 0 || slices <= 0 || tokens <= 0) return c;
    const int rows = head_dim == 64 ? 16 : 32;  // the decompressors' tile
    const int dp = head_dim <= 64 ? 64 : 128;
    c.geo.tiles = uint32_t((tokens + rows - 1) / rows);
    c.geo.tpc = uint32_t(delta_chunk / rows);
    c.geo.cps = (c.geo.tiles + c.geo.tpc - 1) / c.geo.tpc;
    c.geo.gpc = (std::min(c.geo.tpc, c.geo.tiles) + 31u) / 32u;
    c.slot_words = (dp * max_bits / 32 + 1 + 3) / 4 * 4;
    c.groups = uint64_t(slices) * c.geo.cps * c.geo.gpc;
    if (c.geo.gpc <= 1) return c;  // every group starts its chain: no workspace
    auto a256 = [](uint64_t v) { return (v + 255u) & ~uint64_t(255u); };
    c.gsum = 0;
    c.gexcl = a256(c.groups * c.slot_words * 4);
    c.total = c.gexcl + a256(c.groups * c.slot_words * 4);
    return c;
}

struct ChainState {
    bool delta = false;          // a temporal delta: walk groups of tiles
    uint32_t* gsum = nullptr;    // per group: its total (workspace)
    uint32_t* gexcl = nullptr;   // per group: the sum of its chain's earlier groups (nullptr: one group per chain)
    int slot_words = 0;
    ChainGeom geo{};
};

struct LaunchArgs {
    int64_t slices;  // layers * batch * kv_heads
    int tokens;
    int tpad;        // record rows per slice: tokens rounded up to a multiple of 32
    int group;
    int delta_chunk;
    cudaStream_t stream;
    uint8_t* workspace = nullptr;  // decompression with a delta: the running sums' scratch
    unsigned stages = 7u;          // decompression: which of kStageRunTotals | kStageChainScan | kStageDecode to launch
};

// The launches of one tensor's decompression, in stream order: the run totals
// and the chain scan (only for delta chains longer than a run of tiles), then
// the decoder.  A call can split them so that the value tensor's run totals
// overlap the key tensor's decoder.
constexpr unsigned kStageRunTotals = 1u, kStageChainScan = 2u, kStageDecode = 4u;

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
// max_bits: the wider of the call's two bit widths (it sizes the workspace slots).
int launch_decompress_tensor(const LaunchArgs& a, int head_dim, int bits, int max_bits, const uint8_t* idx,
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
