// nq_api.cu -- the C ABI of libnq: argument validation, the compressed-buffer
// layout, the RoPE table, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "nq_internal.h"

namespace nq {

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t align256(uint64_t v) { return (v + 255u) & ~uint64_t(255u); }

int padded_dim(int head_dim) { return head_dim <= 64 ? 64 : 128; }

int check(const nq_shape* s, const nq_params* p) {
    if (!s || !p) return NQ_ERR_ARG;
    if (s->layers < 0 || s->batch < 0 || s->kv_heads < 0 || s->tokens < 0) return NQ_ERR_ARG;
    if (s->head_dim != 64 && s->head_dim != 96 && s->head_dim != 128) return NQ_ERR_UNSUPPORTED;
    if (p->key_bits < 2 || p->key_bits > 4 || p->value_bits < 2 || p->value_bits > 4)
        return NQ_ERR_UNSUPPORTED;
    const int dp = padded_dim(s->head_dim);
    if (p->group_size != 32 && p->group_size != 64 && p->group_size != 128) return NQ_ERR_UNSUPPORTED;
    if (p->group_size > dp) return NQ_ERR_UNSUPPORTED;
    if (p->strict < 0 || p->strict > 2) return NQ_ERR_ARG;
    if (p->delta_chunk < 0 || (p->delta_chunk % 32) != 0) return NQ_ERR_ARG;
    if (!std::isfinite(p->rope_theta)) return NQ_ERR_ARG;
    return NQ_OK;
}

int pad_tokens(int tokens) { return (tokens + 31) / 32 * 32; }

// A stream of the library's own per device, with a fork and a join event:
// the value tensor's delta run totals (a pure read of its idx section) run on
// it while the key tensor's decoder runs on the caller's stream, so the
// re-read overlaps the decoder instead of following it.  Created on first
// use with the device current; the mutex also keeps one call's fork/join
// pair from interleaving with another thread's.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
std::mutex g_side_mu;
SideStream g_side[kMaxSideDevices];

SideStream* side_stream_locked() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
    SideStream& ss = g_side[dev];
    if (ss.stream == nullptr) {
        cudaStream_t st = nullptr;
        cudaEvent_t f = nullptr, j = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
            if (f) cudaEventDestroy(f);
            cudaStreamDestroy(st);
            return nullptr;
        }
        ss.stream = st;
        ss.fork = f;
        ss.join = j;
    }
    return &ss;
}

// The coset words of a tensor, or null in the strict joint format (strict = 2),
// whose block codes carry the coset bit themselves.
uint16_t* coset_section(uint8_t* base, uint64_t off, const nq_params* p) {
    return p->strict == 2 ? nullptr : reinterpret_cast<uint16_t*>(base + off);
}
const uint16_t* coset_section(const uint8_t* base, uint64_t off, const nq_params* p) {
    return p->strict == 2 ? nullptr : reinterpret_cast<const uint16_t*>(base + off);
}

void make_layout(const nq_shape* s, const nq_params* p, nq_layout* L) {
    const int dp = padded_dim(s->head_dim);
    const uint64_t slices = uint64_t(s->layers) * s->batch * s->kv_heads;
    const uint64_t rows = slices * uint64_t(pad_tokens(s->tokens));
    std::memset(L, 0, sizeof(*L));
    L->version = NQ_FORMAT_VERSION;
    L->padded_dim = uint32_t(dp);
    L->tokens_padded = uint32_t(pad_tokens(s->tokens));
    L->rows = rows;
    L->k_idx_row_bytes = uint64_t(dp) * p->key_bits / 8;
    L->v_idx_row_bytes = uint64_t(dp) * p->value_bits / 8;
    L->scales_per_row = uint64_t(dp / p->group_size);
    uint64_t off = 0;
    L->k_idx = off;
    off = align256(off + rows * L->k_idx_row_bytes);
    const uint64_t coset_bytes = p->strict == 2 ? 0 : 2;  // the joint format has no coset words
    L->k_coset = off;
    off = align256(off + rows * coset_bytes);
    L->k_scale = off;
    off = align256(off + rows * L->scales_per_row * 2);
    L->v_idx = off;
    off = align256(off + rows * L->v_idx_row_bytes);
    L->v_coset = off;
    off = align256(off + rows * coset_bytes);
    L->v_scale = off;
    off = align256(off + rows * L->scales_per_row * 2);
    L->total_bytes = off;
    L->workspace_bytes = chain_plan(int64_t(slices), s->tokens, s->head_dim, std::max(p->key_bits, p->value_bits),
                                    p->delta_chunk).total;
}

}  // namespace

int grid_capacity_threads(const void* kernel, int smem, int threads) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, size_t(smem)) != cudaSuccess)
        return -1;
    if (per_sm <= 0) return -1;  // the kernel cannot be resident at all
    return sms * per_sm;
}

int grid_capacity(const void* kernel, int smem) { return grid_capacity_threads(kernel, smem, kThreads); }

bool ensure_smem(const void* kernel, int smem) {
    // (kernel, device) pairs already configured; the attribute is per device
    static std::mutex mu;
    static const void* done_kernel[256];
    static int done_dev[256];
    static int n_done = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_kernel[i] == kernel && done_dev[i] == dev) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return false;
    if (n_done < 256) {
        done_kernel[n_done] = kernel;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return true;
}

bool make_row_tile_map(CUtensorMap* map, void* base, int head_dim, int tokens, int64_t slices, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) return false;
    const cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(tokens), cuuint64_t(slices)};
    const cuuint64_t strides[2] = {cuuint64_t(head_dim) * 2, cuuint64_t(head_dim) * 2 * cuuint64_t(tokens)};
    const cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ e8 test entry

template <int BITS, bool STRICT>
__global__ void e8_nearest_kernel(const float* __restrict__ u, float* __restrict__ out, int64_t n) {
    for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < n;
         b += int64_t(gridDim.x) * blockDim.x) {
        float v[8], r[8];
        float umax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = u[8 * b + j];
            umax = fmaxf(umax, fabsf(v[j]));
        }
        if constexpr (BITS > 0) {
            using C = Code<BITS>;
            unsigned c, code;
            if (umax < C::H && e8_fast<BITS, STRICT>(v, code, c)) {
                // the path compression takes for in-box blocks
                const float off = c ? C::H : C::HI0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    r[j] = __fsub_rn(float((code >> (j * BITS)) & C::MASK), off);
            } else {
                e8_general(v, STRICT, C::HI0, C::H, r);
            }
        } else {
            e8_general(v, STRICT, INFINITY, INFINITY, r);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) out[8 * b + j] = r[j];
    }
}

template <int BITS>
static int launch_e8(const float* u, float* out, int64_t n, bool strict, cudaStream_t st) {
    const int64_t want = (n + 255) / 256;
    const int grid = int(std::min<int64_t>(want, 4096));
    if (strict)
        e8_nearest_kernel<BITS, true><<<grid, 256, 0, st>>>(u, out, n);
    else
        e8_nearest_kernel<BITS, false><<<grid, 256, 0, st>>>(u, out, n);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

int launch_e8_nearest(const float* u, float* out, int64_t n, bool strict, int bits, cudaStream_t st) {
    switch (bits) {
        case 0:
            return launch_e8<0>(u, out, n, strict, st);
        case 2:
            return launch_e8<2>(u, out, n, strict, st);
        case 3:
            return launch_e8<3>(u, out, n, strict, st);
        case 4:
            return launch_e8<4>(u, out, n, strict, st);
        default:
            return NQ_ERR_UNSUPPORTED;
    }
}

}  // namespace nq

// =================================================================== C ABI

extern "C" {

int nq_plan(const nq_shape* shape, const nq_params* params, nq_layout* out) {
    const int st = nq::check(shape, params);
    if (st != NQ_OK) return st;
    if (!out) return NQ_ERR_ARG;
    nq::make_layout(shape, params, out);
    return NQ_OK;
}

int nq_rope_table(const int32_t* positions, int32_t tokens, int32_t head_dim, float rope_theta,
                  float* table) {
    if (tokens < 0 || head_dim <= 0 || (head_dim & 1) || !(rope_theta > 0.0f) ||
        !std::isfinite(rope_theta))
        return NQ_ERR_ARG;
    if (tokens > 0 && !table) return NQ_ERR_ARG;
    if (head_dim % 4) return NQ_ERR_ARG;
    const int half = head_dim / 2;
    for (int32_t t = 0; t < tokens; ++t) {
        const double p = positions ? double(positions[t]) : double(t);
        for (int i = 0; i < half; ++i) {
            const double angle = p * std::pow(double(rope_theta), -2.0 * double(i) / double(head_dim));
            // quad q = i / 2 holds the pairs 2q and 2q + 1 of token t
            float* quad = table + (size_t(i / 2) * size_t(tokens) + size_t(t)) * 4;
            quad[2 * (i & 1)] = float(std::cos(angle));
            quad[2 * (i & 1) + 1] = float(std::sin(angle));
        }
    }
    return NQ_OK;
}

int nq_compress_kv(const void* k_f16, const void* v_f16, const float* rope_table,
                   const nq_shape* shape, const nq_params* params, void* out, size_t out_bytes,
                   void* stream) {
    int st = nq::check(shape, params);
    if (st != NQ_OK) return st;
    nq_layout L;
    nq::make_layout(shape, params, &L);
    if (L.rows == 0) return NQ_OK;
    const bool rope = params->rope_theta > 0.0f;
    if (!k_f16 || !v_f16 || !out || (rope && !rope_table)) return NQ_ERR_ARG;
    if (!nq::aligned16(k_f16) || !nq::aligned16(v_f16) || !nq::aligned16(out) ||
        (rope && !nq::aligned16(rope_table)))
        return NQ_ERR_ARG;
    if (out_bytes < L.total_bytes) return NQ_ERR_SIZE;
    nq::LaunchArgs a;
    a.slices = int64_t(shape->layers) * shape->batch * shape->kv_heads;
    a.tokens = shape->tokens;
    a.tpad = int(L.tokens_padded);
    a.group = params->group_size;
    a.delta_chunk = params->delta_chunk;
    a.stream = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(out);
    st = nq::launch_compress_tensor(a, shape->head_dim, params->key_bits, params->strict, k_f16,
                                    rope ? rope_table : nullptr, base + L.k_idx,
                                    nq::coset_section(base, L.k_coset, params),
                                    reinterpret_cast<uint16_t*>(base + L.k_scale));
    if (st != NQ_OK) return st;
    return nq::launch_compress_tensor(a, shape->head_dim, params->value_bits, params->strict,
                                      v_f16, nullptr, base + L.v_idx,
                                      nq::coset_section(base, L.v_coset, params),
                                      reinterpret_cast<uint16_t*>(base + L.v_scale));
}

int nq_roundtrip_kv(const void* k_f16, const void* v_f16, const float* rope_table,
                    const nq_shape* shape, const nq_params* params, void* k_f16_out, void* v_f16_out,
                    void* stream) {
    int st = nq::check(shape, params);
    if (st != NQ_OK) return st;
    nq_layout L;
    nq::make_layout(shape, params, &L);
    if (L.rows == 0) return NQ_OK;
    const bool rope = params->rope_theta > 0.0f;
    if (!k_f16 || !v_f16 || !k_f16_out || !v_f16_out || (rope && !rope_table)) return NQ_ERR_ARG;
    if (!nq::aligned16(k_f16) || !nq::aligned16(v_f16) || !nq::aligned16(k_f16_out) ||
        !nq::aligned16(v_f16_out) || (rope && !nq::aligned16(rope_table)))
        return NQ_ERR_ARG;
    nq::LaunchArgs a;
    a.slices = int64_t(shape->layers) * shape->batch * shape->kv_heads;
    a.tokens = shape->tokens;
    a.tpad = int(L.tokens_padded);
    a.group = params->group_size;
    a.delta_chunk = 0;
    a.stream = static_cast<cudaStream_t>(stream);
    st = nq::launch_roundtrip_tensor(a, shape->head_dim, params->key_bits, params->strict != 0, k_f16,
                                     rope ? rope_table : nullptr, k_f16_out);
    if (st != NQ_OK) return st;
    return nq::launch_roundtrip_tensor(a, shape->head_dim, params->value_bits, params->strict != 0, v_f16,
                                       nullptr, v_f16_out);
}

int nq_code_histogram(const void* in, size_t in_bytes, const nq_shape* shape, const nq_params* params,
                      uint64_t* counts, void* stream) {
    int st = nq::check(shape, params);
    if (st != NQ_OK) return st;
    nq_layout L;
    nq::make_layout(shape, params, &L);
    if (!counts || (reinterpret_cast<uintptr_t>(counts) & 7u) != 0) return NQ_ERR_ARG;
    if (L.rows > 0 && (!in || !nq::aligned16(in))) return NQ_ERR_ARG;
    if (in_bytes < L.total_bytes) return NQ_ERR_SIZE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counts, 0, 2 * NQ_HIST_BINS * sizeof(uint64_t), s) != cudaSuccess) return NQ_ERR_CUDA;
    if (L.rows == 0) return NQ_OK;
    nq::LaunchArgs a;
    a.slices = int64_t(shape->layers) * shape->batch * shape->kv_heads;
    a.tokens = shape->tokens;
    a.tpad = int(L.tokens_padded);
    a.group = params->group_size;
    a.delta_chunk = params->delta_chunk;
    a.stream = s;
    const uint8_t* base = static_cast<const uint8_t*>(in);
    st = nq::launch_code_histogram(a, int(L.padded_dim), params->key_bits, base + L.k_idx,
                                   nq::coset_section(base, L.k_coset, params), counts);
    if (st != NQ_OK) return st;
    return nq::launch_code_histogram(a, int(L.padded_dim), params->value_bits, base + L.v_idx,
                                     nq::coset_section(base, L.v_coset, params), counts + NQ_HIST_BINS);
}

int nq_decompress_kv(const void* in, size_t in_bytes, const float* rope_table,
                     const nq_shape* shape, const nq_params* params, void* k_f16_out,
                     void* v_f16_out, void* workspace, size_t workspace_bytes, void* stream) {
    int st = nq::check(shape, params);
    if (st != NQ_OK) return st;
    nq_layout L;
    nq::make_layout(shape, params, &L);
    if (L.rows == 0) return NQ_OK;
    const bool rope = params->rope_theta > 0.0f;
    if (!in || !k_f16_out || !v_f16_out || (rope && !rope_table)) return NQ_ERR_ARG;
    if (!nq::aligned16(in) || !nq::aligned16(k_f16_out) || !nq::aligned16(v_f16_out) ||
        (rope && !nq::aligned16(rope_table)))
        return NQ_ERR_ARG;
    if (L.workspace_bytes > 0 && (!workspace || !nq::aligned16(workspace))) return NQ_ERR_ARG;
    if (in_bytes < L.total_bytes || workspace_bytes < L.workspace_bytes) return NQ_ERR_SIZE;
    nq::LaunchArgs a;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.slices = int64_t(shape->layers) * shape->batch * shape->kv_heads;
    a.tokens = shape->tokens;
    a.tpad = int(L.tokens_padded);
    a.group = params->group_size;
    a.delta_chunk = params->delta_chunk;
    a.stream = static_cast<cudaStream_t>(stream);
    const uint8_t* base = static_cast<const uint8_t*>(in);
    const int max_bits = std::max(params->key_bits, params->value_bits);
    auto keys = [&](const nq::LaunchArgs& la) {
        return nq::launch_decompress_tensor(la, shape->head_dim, params->key_bits, max_bits, base + L.k_idx,
                                            nq::coset_section(base, L.k_coset, params),
                                            reinterpret_cast<const uint16_t*>(base + L.k_scale),
                                            rope ? rope_table : nullptr, k_f16_out);
    };
    auto values = [&](const nq::LaunchArgs& la) {
        return nq::launch_decompress_tensor(la, shape->head_dim, params->value_bits, max_bits, base + L.v_idx,
                                            nq::coset_section(base, L.v_coset, params),
                                            reinterpret_cast<const uint16_t*>(base + L.v_scale), nullptr,
                                            v_f16_out);
    };
    if (L.workspace_bytes > 0) {
        // Long delta chains: key run totals and scan; then the value run totals
        // on the side stream (they overwrite only the totals, which the key
        // scan has consumed) while the keys decode (they read only the scan's
        // results); then, joined, the value scan and decoder.
        std::lock_guard<std::mutex> lock(nq::g_side_mu);
        nq::SideStream* ss = nq::side_stream_locked();
        if (ss != nullptr) {
            nq::LaunchArgs ka = a, va = a;
            ka.stages = nq::kStageRunTotals | nq::kStageChainScan;
            st = keys(ka);
            if (st != NQ_OK) return st;
            if (cudaEventRecord(ss->fork, a.stream) != cudaSuccess ||
                cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
                return NQ_ERR_CUDA;
            va.stream = ss->stream;
            va.stages = nq::kStageRunTotals;
            const int sv = values(va);
            ka.stages = nq::kStageDecode;
            const int sk = keys(ka);
            // join even after a failed launch, so the caller's stream never runs ahead of the side stream
            if (cudaEventRecord(ss->join, ss->stream) != cudaSuccess ||
                cudaStreamWaitEvent(a.stream, ss->join, 0) != cudaSuccess)
                return NQ_ERR_CUDA;
            if (sv != NQ_OK) return sv;
            if (sk != NQ_OK) return sk;
            va.stream = a.stream;
            va.stages = nq::kStageChainScan | nq::kStageDecode;
            return values(va);
        }
    }
    st = keys(a);
    if (st != NQ_OK) return st;
    return values(a);
}

int nq_get_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NQ_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

int nq_e8_nearest(const float* u, float* out, int64_t n_blocks, int strict, int bits, void* stream) {
    if (n_blocks < 0 || (strict != 0 && strict != 1)) return NQ_ERR_ARG;
    if (bits != 0 && (bits < 2 || bits > 4)) return NQ_ERR_UNSUPPORTED;
    if (n_blocks == 0) return NQ_OK;
    if (!u || !out) return NQ_ERR_ARG;
    return nq::launch_e8_nearest(u, out, n_blocks, strict != 0, bits,
                                 static_cast<cudaStream_t>(stream));
}

const char* nq_strerror(int status) {
    switch (status) {
        case NQ_OK:
            return "ok";
        case NQ_ERR_ARG:
            return "invalid argument (null, misaligned or out-of-range value)";
        case NQ_ERR_UNSUPPORTED:
            return "unsupported head_dim, bit width or group size";
        case NQ_ERR_SIZE:
            return "caller buffer smaller than the planned size";
        case NQ_ERR_CUDA:
            return "CUDA launch or runtime error";
        default:
            return "unknown status";
    }
}

}  // extern "C"
