// nq_layers.cu -- per-layer bit widths and layers kept in fp16 (the method's
// graduated bit profiles and boundary-layer protection): a host loop over the
// layers on top of the single-layer entry points.  The buffer is one part per
// layer, 256-byte aligned: the single-layer compressed buffer of that layer's
// bit widths, or the layer's K then V copied as they are.
#include <vector>

#include "nq_internal.h"

namespace {

uint64_t align256(uint64_t v) { return (v + 255u) & ~uint64_t(255u); }

bool kept(const nq_layer_bits& b) { return b.key_bits == 0 && b.value_bits == 0; }

nq_params layer_params(const nq_params* p, const nq_layer_bits& b) {
    nq_params o = *p;
    if (!kept(b)) {
        o.key_bits = b.key_bits;
        o.value_bits = b.value_bits;
    }
    return o;
}

nq_shape one_layer(const nq_shape* s) {
    nq_shape o = *s;
    o.layers = 1;
    return o;
}

uint64_t layer_bytes(const nq_shape* s) {  // fp16 bytes of one tensor's layer
    return uint64_t(s->batch) * s->kv_heads * s->tokens * s->head_dim * 2;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Keys carry RoPE: the table every compressed layer will need, checked before
// the first layer is enqueued (a kept layer's copies would otherwise be in
// flight when a later layer rejects the table).
bool rope_ok(const nq_params* p, const float* rope_table) {
    return !(p->rope_theta > 0.0f) || (rope_table && aligned16(rope_table));
}

// Plan, then check the pointers the loop will use.
int prepare(const nq_shape* shape, const nq_params* params, const nq_layer_bits* per_layer,
            std::vector<uint64_t>& offs, uint64_t* total, uint64_t* ws = nullptr) {
    if (!shape) return NQ_ERR_ARG;
    offs.assign(size_t(shape->layers > 0 ? shape->layers : 0), 0);
    return nq_plan_layers(shape, params, per_layer, offs.data(), total, ws);
}

int copy(void* dst, const void* src, uint64_t bytes, cudaStream_t s) {
    if (dst == src || bytes == 0) return NQ_OK;
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

}  // namespace

extern "C" {

int nq_plan_layers(const nq_shape* shape, const nq_params* params, const nq_layer_bits* per_layer,
                   uint64_t* offsets, uint64_t* total_bytes, uint64_t* workspace_bytes) {
    if (!shape || !params || !total_bytes) return NQ_ERR_ARG;
    nq_layout whole;
    int st = nq_plan(shape, params, &whole);  // validates the shape and the shared parameters
    if (st != NQ_OK) return st;
    if (shape->layers > 0 && (!per_layer || !offsets)) return NQ_ERR_ARG;
    const nq_shape s1 = one_layer(shape);
    uint64_t off = 0, ws = 0;
    for (int l = 0; l < shape->layers; ++l) {
        uint64_t bytes = 2 * layer_bytes(shape);
        if (!kept(per_layer[l])) {
            const nq_params p = layer_params(params, per_layer[l]);
            nq_layout L;
            st = nq_plan(&s1, &p, &L);
            if (st != NQ_OK) return st;
            bytes = L.total_bytes;
            ws = std::max<uint64_t>(ws, L.workspace_bytes);
        }
        offsets[l] = off;
        off = align256(off + bytes);
    }
    *total_bytes = off;
    if (workspace_bytes) *workspace_bytes = ws;
    return NQ_OK;
}

int nq_compress_kv_layers(const void* k_f16, const void* v_f16, const float* rope_table, const nq_shape* shape,
                          const nq_params* params, const nq_layer_bits* per_layer, void* out, size_t out_bytes,
                          void* stream) {
    std::vector<uint64_t> offs;
    uint64_t total = 0;
    int st = prepare(shape, params, per_layer, offs, &total);
    if (st != NQ_OK) return st;
    const uint64_t lb = layer_bytes(shape);
    if (offs.empty() || lb == 0) return NQ_OK;
    if (!k_f16 || !v_f16 || !out || !aligned16(k_f16) || !aligned16(v_f16) || !aligned16(out)) return NQ_ERR_ARG;
    if (!rope_ok(params, rope_table)) return NQ_ERR_ARG;
    if (out_bytes < total) return NQ_ERR_SIZE;
    const nq_shape s1 = one_layer(shape);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t l = 0; l < offs.size() && st == NQ_OK; ++l) {
        const char* k = static_cast<const char*>(k_f16) + l * lb;
        const char* v = static_cast<const char*>(v_f16) + l * lb;
        char* part = static_cast<char*>(out) + offs[l];
        const uint64_t room = (l + 1 < offs.size() ? offs[l + 1] : total) - offs[l];
        if (kept(per_layer[l])) {
            st = copy(part, k, lb, s);
            if (st == NQ_OK) st = copy(part + lb, v, lb, s);
        } else {
            const nq_params p = layer_params(params, per_layer[l]);
            st = nq_compress_kv(k, v, rope_table, &s1, &p, part, room, stream);
        }
    }
    return st;
}

int nq_decompress_kv_layers(const void* in, size_t in_bytes, const float* rope_table, const nq_shape* shape,
                            const nq_params* params, const nq_layer_bits* per_layer, void* k_f16_out,
                            void* v_f16_out, void* workspace, size_t workspace_bytes, void* stream) {
    std::vector<uint64_t> offs;
    uint64_t total = 0, ws = 0;
    int st = prepare(shape, params, per_layer, offs, &total, &ws);
    if (st != NQ_OK) return st;
    const uint64_t lb = layer_bytes(shape);
    if (offs.empty() || lb == 0) return NQ_OK;
    if (!in || !k_f16_out || !v_f16_out || !aligned16(in) || !aligned16(k_f16_out) || !aligned16(v_f16_out))
        return NQ_ERR_ARG;
    if (!rope_ok(params, rope_table)) return NQ_ERR_ARG;
    if (ws > 0 && (!workspace || !aligned16(workspace))) return NQ_ERR_ARG;
    if (in_bytes < total || workspace_bytes < ws) return NQ_ERR_SIZE;
    const nq_shape s1 = one_layer(shape);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t l = 0; l < offs.size() && st == NQ_OK; ++l) {
        char* k = static_cast<char*>(k_f16_out) + l * lb;
        char* v = static_cast<char*>(v_f16_out) + l * lb;
        const char* part = static_cast<const char*>(in) + offs[l];
        const uint64_t room = (l + 1 < offs.size() ? offs[l + 1] : total) - offs[l];
        if (kept(per_layer[l])) {
            st = copy(k, part, lb, s);
            if (st == NQ_OK) st = copy(v, part + lb, lb, s);
        } else {
            const nq_params p = layer_params(params, per_layer[l]);
            st = nq_decompress_kv(part, room, rope_table, &s1, &p, k, v, workspace, workspace_bytes, stream);
        }
    }
    return st;
}

int nq_roundtrip_kv_layers(const void* k_f16, const void* v_f16, const float* rope_table, const nq_shape* shape,
                           const nq_params* params, const nq_layer_bits* per_layer, void* k_f16_out,
                           void* v_f16_out, void* stream) {
    std::vector<uint64_t> offs;
    uint64_t total = 0;
    int st = prepare(shape, params, per_layer, offs, &total);
    if (st != NQ_OK) return st;
    const uint64_t lb = layer_bytes(shape);
    if (offs.empty() || lb == 0) return NQ_OK;
    if (!k_f16 || !v_f16 || !k_f16_out || !v_f16_out || !aligned16(k_f16) || !aligned16(v_f16) ||
        !aligned16(k_f16_out) || !aligned16(v_f16_out))
        return NQ_ERR_ARG;
    if (!rope_ok(params, rope_table)) return NQ_ERR_ARG;
    const nq_shape s1 = one_layer(shape);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t l = 0; l < offs.size() && st == NQ_OK; ++l) {
        const char* k = static_cast<const char*>(k_f16) + l * lb;
        const char* v = static_cast<const char*>(v_f16) + l * lb;
        char* ko = static_cast<char*>(k_f16_out) + l * lb;
        char* vo = static_cast<char*>(v_f16_out) + l * lb;
        if (kept(per_layer[l])) {
            st = copy(ko, k, lb, s);
            if (st == NQ_OK) st = copy(vo, v, lb, s);
        } else {
            const nq_params p = layer_params(params, per_layer[l]);
            st = nq_roundtrip_kv(k, v, rope_table, &s1, &p, ko, vo, stream);
        }
    }
    return st;
}

}  // extern "C"
