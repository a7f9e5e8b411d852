// nq_decompress_kv_static: decompression whose delta scratch is a static
// device array owned by the library, so the call needs no workspace and
// allocates nothing.
//
// Who needs it: callers that cannot allocate device memory at the point of
// the call and cannot hand over a workspace -- a plug-in that receives only
// the cache and record pointers from an engine owning all device memory in a
// pool fixed at start-up, or a C host program without a device allocator of
// its own.  nq_decompress_kv needs a workspace only for a temporal delta
// whose chains are longer than 32 record tiles; this entry point serves that
// case from the static array below, up to NQ_STATIC_WORKSPACE_BYTES.
//
// The scratch is written and read by the same call (per run of tiles: its
// total, then the running sum of the runs before it in its chain); nothing in
// it has to start at zero, and nothing is left in it that a later call reads.
// There is one array per device, so calls that overlap in time on one device
// (two host threads, or work enqueued on two streams) race on it; calls must
// be ordered on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nq.h"

static __device__ __align__(256) unsigned char g_nq_static_scratch[NQ_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The scratch's device address on the current device, looked up once per
// device (with that device current) and remembered.
int static_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_nq_static_scratch) != cudaSuccess || p == nullptr) return NQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return NQ_OK;
}

}  // namespace

extern "C" int nq_decompress_kv_static(const void* in, size_t in_bytes, const float* rope_table,
                                       const nq_shape* shape, const nq_params* params, void* k_f16_out,
                                       void* v_f16_out, void* stream) {
    nq_layout L;
    const int st = nq_plan(shape, params, &L);
    if (st != NQ_OK) return st;
    if (L.workspace_bytes > NQ_STATIC_WORKSPACE_BYTES) return NQ_ERR_SIZE;
    void* ws = nullptr;
    if (L.workspace_bytes > 0) {
        const int s = static_scratch(&ws);
        if (s != NQ_OK) return s;
    }
    return nq_decompress_kv(in, in_bytes, rope_table, shape, params, k_f16_out, v_f16_out, ws, L.workspace_bytes,
                            stream);
}
