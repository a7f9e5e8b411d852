/*
 * nq.h -- C ABI of libnq: E8 lattice KV-cache compression on GB300 (sm_103a).
 *
 * The method (NexusQuant write-ups, "E8 walkthrough" post and the paper "E8
 * Lattice Key Quantization for Low-Bit KV-Cache Compression"): after prefill,
 * keys have their rotary embedding removed; keys and values get a
 * Walsh-Hadamard rotation over head_dim (zero-padded to a power of two), a
 * per-group absmax scale, and a nearest-point search in the E8 lattice per
 * 8-float block (Conway-Sloane two-coset decoder, strict or relaxed parity);
 * the lattice codes are packed into b-bit indices, optionally delta-coded
 * across tokens.  Decompression inverts every step.
 *
 * Conventions for every entry point:
 *  - Plain C types; no allocation and no freeing inside the library; the
 *    caller owns every buffer.  Device pointers must be 16-byte aligned.
 *  - Work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = the
 *    legacy default stream) and is asynchronous: a return of NQ_OK means the
 *    launch was accepted.  Launch failures return NQ_ERR_CUDA; the CUDA error
 *    state is left for the caller to inspect.
 *  - Arguments are validated before anything is enqueued; on any error
 *    nothing has been written.
 *  - Inputs must be finite; NaN or infinite inputs give unspecified codes.
 *
 * Tensor layout: K and V are contiguous fp16 [layers, batch, kv_heads,
 * tokens, head_dim] (for batch 1 this is [layers, kv_heads, tokens,
 * head_dim]).  A "row" is one head_dim vector.  A slice is one (layer,
 * batch, head); slice s = (l * batch + b) * kv_heads + h.  In the compressed
 * buffer every slice holds tokens_padded = 32 * ceil(tokens / 32) record
 * rows: record row s * tokens_padded + t describes token t, and the rows for
 * t >= tokens are zero.
 *
 * Compressed buffer (format version NQ_FORMAT_VERSION), sections in the
 * order below, each starting at a 256-byte aligned offset given by nq_plan:
 *   K idx   [rows][Dp * key_bits / 8]   bytes   (rows = slices * tokens_padded)
 *   K coset [rows]                       uint16, bit k = coset of block k
 *                                         (empty when strict = 2, the joint format)
 *   K scale [rows][Dp / group_size]      fp16
 *   V idx / V coset / V scale            the same with value_bits.
 * Dp = padded head_dim (64 for head_dim 64, 128 for 96 and 128).  Within an
 * idx row, coordinate i's code sits at bit i*b, least significant bit first,
 * little-endian bytes; code = lattice coordinate + offset, offset = 2^(b-1)-1
 * for the integer coset and (2^b - 1)/2 for the half-integer coset.  With
 * delta coding on, every row whose token index is not a multiple of
 * delta_chunk holds its codes minus the previous token's codes (per field,
 * modulo 2^b) and its coset word XOR the previous one; scales are never
 * delta-coded.  In the joint format the delta applies to the stored fields
 * (the coset bit included) the same way.
 */
#ifndef NQ_H
#define NQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NQ_FORMAT_VERSION 1u

enum {
    NQ_OK = 0,
    NQ_ERR_ARG = 1,         /* null pointer, bad shape, misaligned pointer  */
    NQ_ERR_UNSUPPORTED = 2, /* head_dim, bit width or group size not served */
    NQ_ERR_SIZE = 3,        /* a caller buffer is smaller than required     */
    NQ_ERR_CUDA = 4         /* a CUDA call or kernel launch failed          */
};

/* Cache shape.  head_dim in {64, 96, 128}; tokens >= 0; zero-sized tensors
 * are accepted and do nothing. */
typedef struct {
    int32_t layers, batch, kv_heads, tokens, head_dim;
} nq_shape;

/* Codec parameters.
 *  key_bits, value_bits: 2, 3 or 4 bits per coordinate ("K3V2", "K2V2").
 *  group_size: 32, 64 or 128 coordinates per fp16 scale; must divide Dp.
 *  strict: 1 = strict E8 (both cosets even-sum), 0 = relaxed parity (the
 *          half-integer coset drops its even-sum rule), 2 = strict E8 in the
 *          joint format: every block is exactly 8b bits and there are no
 *          coset words (the field sum of a strict point is even, so the low
 *          bit of the last field is implied and its place holds the coset
 *          bit: fields 0..6, then m_7 >> 1 in b - 1 bits, then the coset bit).
 *          Relaxed codes need the extra bit per block that the coset words
 *          carry ("What Makes E8 Special", "The Relaxed Parity Discovery").
 *  delta_chunk: 0 = no temporal delta; otherwise a positive multiple of 32:
 *          codes are delta-coded along tokens and the chain restarts at every
 *          token index that is a multiple of delta_chunk (one chain per
 *          (layer, batch, head) slice when delta_chunk >= tokens).
 *  rope_theta: > 0 keys carry split-half RoPE with this base and a table from
 *          nq_rope_table is required; <= 0 keys are treated like values. */
typedef struct {
    int32_t key_bits, value_bits;
    int32_t group_size;
    int32_t strict;
    int32_t delta_chunk;
    float rope_theta;
} nq_params;

/* Byte offsets and sizes of the compressed buffer's sections, and the size
 * of the workspace that decompression with a temporal delta needs. */
typedef struct {
    uint32_t version;
    uint32_t padded_dim;
    uint32_t tokens_padded; /* record rows per slice: tokens rounded up to 32 */
    uint32_t reserved;
    uint64_t rows;          /* record rows per tensor: slices * tokens_padded */
    uint64_t k_idx_row_bytes, v_idx_row_bytes, scales_per_row;
    uint64_t k_idx, k_coset, k_scale, v_idx, v_coset, v_scale;
    uint64_t total_bytes;
    uint64_t workspace_bytes; /* nq_decompress_kv's workspace: 0 without a delta */
} nq_layout;

/* Validate shape and params and describe the compressed buffer.  Host only.
 * Format: the section table above.  The method stores the lattice indices
 * packed into bytes ("E8 walkthrough", section "Bit Rate Accounting") and
 * gives every group of coordinates an fp16 scale; that section and "Why
 * Per-Group Scaling?" scale every 8 values (and the per-head variant every
 * 128), while this format keeps one fp16 scale per group_size coordinates
 * (64 in the target workloads). */
int nq_plan(const nq_shape* shape, const nq_params* params, nq_layout* out);

/* RoPE (cos, sin) table for split-half rotary embedding ("E8 walkthrough",
 * "What Makes This Hard in Practice", item 2; README "Supported models").
 * Host only, double precision rounded once to fp32.  With angle(t, i) =
 * p_t * theta^(-2i/head_dim), i < head_dim/2, p_t = positions[t] (host int32)
 * or t when positions is NULL, the table is head_dim/4 planes of `tokens`
 * float4, plane q holding for every token (cos, sin) of pair 2q then of pair
 * 2q + 1:  table[(q * tokens + t) * 4 + 2m + {0: cos, 1: sin}] for pair 2q + m.
 * (Token-minor planes let the kernels read it with coalesced 16-byte loads.)
 * table: caller-owned host buffer of tokens * head_dim floats.  Build it once
 * per (positions, theta, head_dim), copy it to the device and pass it to
 * nq_compress_kv / nq_decompress_kv. */
int nq_rope_table(const int32_t* positions, int32_t tokens, int32_t head_dim, float rope_theta,
                  float* table);

/* Compress K and V (device fp16, layout above) into `out` (device,
 * out_bytes >= nq_plan().total_bytes).  rope_table: device copy of the
 * nq_rope_table() table for these tokens, required when rope_theta > 0,
 * ignored otherwise.  Steps: RoPE removal on keys, zero-padded Hadamard
 * rotation ("E8 quantizes 8 numbers at once", "Handling outliers"), group
 * absmax scale, two-coset E8 nearest point ("E8 walkthrough", "The
 * Conway-Sloane Nearest-Point Algorithm"; relaxed parity per "What Makes E8
 * Special", "The Relaxed Parity Discovery"), b-bit packing, temporal delta
 * ("Negative results", delta coding entry). */
int nq_compress_kv(const void* k_f16, const void* v_f16, const float* rope_table,
                   const nq_shape* shape, const nq_params* params, void* out, size_t out_bytes,
                   void* stream);

/* Decompress `in` (device, produced by nq_compress_kv with the same shape and
 * params) into K and V (device fp16, layout above): undo the delta, unpack,
 * unscale, inverse Hadamard, re-apply RoPE to keys, round to fp16 ("E8
 * walkthrough", quantize() dequantizes the lattice point; "What Makes This
 * Hard in Practice": RoPE removed before quantization and reapplied after).
 *
 * workspace: caller-owned device scratch of workspace_bytes >=
 * nq_plan().workspace_bytes (16-byte aligned).  It is needed only when a
 * delta chain is longer than 32 record tiles (1024 tokens; 512 at head_dim
 * 64), up to the method's single chain per slice; otherwise the size is 0 and
 * it may be NULL.  The decoder walks each chain in runs of up to 32 tiles,
 * carrying the delta's running sum in registers; two light passes over the
 * idx section first leave in the workspace, per run, the running sum of its
 * chain's earlier rows (field-wise modulo 2^b, coset words by exclusive or).
 * Its contents are overwritten by every call; calls that share a workspace
 * must be ordered on one stream.  No kernel waits for another. */
int nq_decompress_kv(const void* in, size_t in_bytes, const float* rope_table,
                     const nq_shape* shape, const nq_params* params, void* k_f16_out,
                     void* v_f16_out, void* workspace, size_t workspace_bytes, void* stream);

/* nq_decompress_kv without a workspace argument: the delta scratch is a
 * static device array of NQ_STATIC_WORKSPACE_BYTES owned by the library (one
 * per device), and the call allocates nothing.  The pages have no counterpart
 * of this call: it serves callers that cannot allocate device memory or hand
 * over a workspace (a plug-in given only the cache and record pointers by an
 * engine that owns all device memory in a pool fixed at start-up, a C host
 * program without a device allocator).  Arguments, layout, ownership and
 * results as nq_decompress_kv, bit for bit.
 *
 * Limit: NQ_ERR_SIZE when nq_plan().workspace_bytes exceeds
 * NQ_STATIC_WORKSPACE_BYTES (enough for one delta chain per slice on 384
 * slices of 131072 tokens at up to 4 bits; shorter chains or no delta need
 * none).  The first call on a device that needs the scratch looks up its
 * address (cudaGetSymbolAddress, with that device current) and keeps it for
 * later calls; that first call should come before any stream capture.
 * Nothing in the scratch has to start at zero: each call writes every word it
 * reads.  Calls that overlap in time on one device race on the scratch (two
 * host threads, or work on two streams): order them on one stream. */
#define NQ_STATIC_WORKSPACE_BYTES (8u << 20)
int nq_decompress_kv_static(const void* in, size_t in_bytes, const float* rope_table,
                            const nq_shape* shape, const nq_params* params, void* k_f16_out,
                            void* v_f16_out, void* stream);

/* The deferred status of the work enqueued on `stream`: waits for the stream
 * to finish, then returns NQ_ERR_CUDA if the stream or an earlier launch
 * failed (the CUDA error is left for the caller to inspect), else NQ_OK.  The
 * other entry points return as soon as their work is enqueued, so a fault in
 * a kernel surfaces here (or at the caller's next synchronisation). */
int nq_get_status(void* stream);

/* The round trip in one pass: K and V (device fp16) -> the reconstruction
 * decompress(compress(.)) written to k_f16_out / v_f16_out (device fp16, same
 * layout), with no compressed buffer in memory.  This is the method's own use
 * of the codec: compress_kv_cache(mode="quant_only") quantizes the cache and
 * hands back the dequantized tensors in place ("E8 walkthrough", quantize()
 * returns the dequantized point; nexusquant README, usage).  The result equals
 * nq_decompress_kv(nq_compress_kv(.)) bit for bit (delta_chunk has no effect:
 * the delta is lossless).  The outputs may alias the inputs (in-place); any
 * other overlap is an error of the caller.  rope_table as for nq_compress_kv.
 * Errors: as nq_compress_kv (NQ_ERR_ARG for null or misaligned pointers). */
int nq_roundtrip_kv(const void* k_f16, const void* v_f16, const float* rope_table,
                    const nq_shape* shape, const nq_params* params, void* k_f16_out, void* v_f16_out,
                    void* stream);

/* Per-layer bit widths ("graduated" profiles that spend more bits on some
 * layers) and layers kept in fp16 (boundary-layer protection): nexusquant
 * README, configuration table, per-layer settings.  One entry per layer:
 * key_bits, value_bits in 2..4, or both 0 to keep that layer's K and V as
 * they are.  The shared nq_params supply group_size, strict, delta_chunk and
 * rope_theta (its key_bits / value_bits must be valid and are otherwise
 * unused).  The buffer holds one part per layer at offsets[l] (256-byte
 * aligned): the nq_compress_kv buffer of that layer alone (shape with
 * layers = 1 and the layer's bit widths), or the layer's fp16 K followed by its
 * fp16 V.  Host-side loops over the single-layer entry points, asynchronous on
 * the stream; errors as those (a layer with one of its bit widths 0 is
 * NQ_ERR_UNSUPPORTED). */
typedef struct {
    int32_t key_bits, value_bits;
} nq_layer_bits;

/* offsets: caller-owned host array of shape->layers entries; *total_bytes:
 * the buffer size; *workspace_bytes (may be NULL): the workspace that
 * nq_decompress_kv_layers needs (the largest single layer's).  Host only. */
int nq_plan_layers(const nq_shape* shape, const nq_params* params, const nq_layer_bits* per_layer,
                   uint64_t* offsets, uint64_t* total_bytes, uint64_t* workspace_bytes);
/* K, V (device fp16, layout above) -> `out` (device, out_bytes >= total).
 * per_layer: host array of shape->layers entries. */
int nq_compress_kv_layers(const void* k_f16, const void* v_f16, const float* rope_table,
                          const nq_shape* shape, const nq_params* params, const nq_layer_bits* per_layer,
                          void* out, size_t out_bytes, void* stream);
/* The inverse of nq_compress_kv_layers (same shape, params and table);
 * workspace as for nq_decompress_kv, sized by nq_plan_layers. */
int nq_decompress_kv_layers(const void* in, size_t in_bytes, const float* rope_table,
                            const nq_shape* shape, const nq_params* params,
                            const nq_layer_bits* per_layer, void* k_f16_out, void* v_f16_out,
                            void* workspace, size_t workspace_bytes, void* stream);
/* nq_roundtrip_kv per layer; kept layers are copied (nothing to do in place). */
int nq_roundtrip_kv_layers(const void* k_f16, const void* v_f16, const float* rope_table,
                           const nq_shape* shape, const nq_params* params,
                           const nq_layer_bits* per_layer, void* k_f16_out, void* v_f16_out,
                           void* stream);

/* Symbol statistics of a compressed buffer, for judging how much an entropy
 * coder could still take off (the pages pack the indices, delta-code them
 * along tokens and hand them to zstd: "E8 walkthrough", "Bit Rate
 * Accounting"; "Negative results", delta coding entry).  Per tensor
 * (K first, then V) NQ_HIST_BINS 64-bit counters:
 *   [0, 16)    occurrences of each b-bit field value in the idx section (the
 *              temporal-delta symbols when delta_chunk > 0; values >= 2^b
 *              stay zero)
 *   [16, 272)  occurrences of each byte value in the idx section
 *   [272]      blocks in the integer coset (coset bit 0), [273] in the
 *              half-integer coset (coset bit 1)
 * Only the record rows of real tokens count, not the padding rows.
 * in: device buffer from nq_compress_kv with this shape and params (in_bytes
 * >= nq_plan().total_bytes).  counts: device uint64[2 * NQ_HIST_BINS],
 * overwritten (zeroed on the stream, then accumulated); 8-byte aligned. */
#define NQ_HIST_BINS 274
int nq_code_histogram(const void* in, size_t in_bytes, const nq_shape* shape, const nq_params* params,
                      uint64_t* counts, void* stream);

/* Nearest point of the E8 codebook for n_blocks 8-float blocks ("E8
 * walkthrough", nearest_point()).  u, out: device float [n_blocks][8].
 * bits = 0: the unbounded lattice (|u| < 2^22 required); bits in 2..4: the
 * box-constrained codebook of a b-bit code.  Test and inspection entry. */
int nq_e8_nearest(const float* u, float* out, int64_t n_blocks, int strict, int bits, void* stream);

/* Static description of a status code. */
const char* nq_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif
