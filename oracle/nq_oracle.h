/*
 * nq_oracle.h -- plain, slow, single-threaded CPU oracle for E8 lattice
 * KV-cache compression.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * Sources (page titles of the method's write-ups):
 *   [WALK]  "E8 walkthrough" post -- sections "The E8 Lattice, Briefly",
 *           "The Conway-Sloane Nearest-Point Algorithm", "Python
 *           Implementation" (nearest_point, quantize), "Why Per-Group
 *           Scaling?", "Bit Rate Accounting", "What Makes This Hard in
 *           Practice".
 *   [RELAX] "What Makes E8 Special" post -- section "The Relaxed Parity
 *           Discovery".
 *   [QUANT] "E8 quantizes 8 numbers at once" post -- sections "E8: quantize 8
 *           at a time", "Handling outliers" (Hadamard rotation).
 *   [NEG]   "Negative results" post -- temporal delta coding entry.
 *   [README] nexusquant README -- "Supported models" (split-half RoPE).
 *
 * Floating point: everything that decides an integer (a lattice code, a coset
 * bit, a parity fix-up coordinate) is evaluated in IEEE binary32 with the op
 * order written out below; the library compiles with -ffp-contract=off so no
 * multiply-add is fused except where fmaf() is written.  Readings of the pages
 * that the code depends on are marked "Reading:".
 */
#ifndef NQ_ORACLE_H
#define NQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Padded transform length: the next power of two >= head_dim (at least 8). */
int orc_padded_dim(int head_dim);

/* IEEE binary16 <-> binary32.  h2f is exact; f2h rounds to nearest even,
 * overflowing to +-inf like an IEEE conversion. */
float orc_h2f(uint16_t h);
uint16_t orc_f2h_rn(float f);

/* RoPE angle table: cs[t][i][0] = (float)cos(pos_t * theta^(-2i/D)),
 * cs[t][i][1] = (float)sin(...), i < D/2, evaluated in double and rounded once.
 * pos may be NULL (positions 0..T-1). */
void orc_rope_table(const int32_t* pos, int tokens, int head_dim, float theta, float* cs);

/* Undo (remove) / re-apply split-half rotary embedding on one row of D floats
 * with the D/2 (cos, sin) pairs of its position. */
void orc_rope_remove(float* x, int head_dim, const float* cs_row);
void orc_rope_apply(float* x, int head_dim, const float* cs_row);

/* Unnormalised Sylvester Walsh-Hadamard transform in place, n a power of two:
 * orc_fwht in the textbook butterfly order h = 1, 2, 4, ..., n/2 (inverse
 * direction); orc_fwht_forward with the last two stages exchanged (h = 1, ...,
 * n/8, n/2, n/4; compression direction). */
void orc_fwht(float* x, int n);
void orc_fwht_forward(float* x, int n);

/* Group scale: the smallest non-negative binary16 value v (returned as bits)
 * such that v * (dp * (2^bits - 1) / 2) >= amax. */
uint16_t orc_group_scale(float amax, int bits, int dp);

/* Nearest point of the (strict or relaxed) E8 codebook to one 8-block u.
 * bits = 0: unbounded lattice; bits in 2..4: the box-constrained codebook of
 * the b-bit code.  Writes the point to r, returns the coset (0 integer, 1
 * half-integer). */
int orc_e8_block(const float* u, int strict, int bits, float* r);
void orc_e8_nearest(const float* u, float* r, int64_t n_blocks, int strict, int bits);

/* One row: raw codes (no delta).  x: D fp16 values; cs_row NULL for values or
 * when RoPE is off.  idx: dp*bits/8 bytes; scales: dp/group fp16.  Decoding
 * saturates at +-65504 (a finite cache never reconstructs to infinity). */
void orc_encode_row(const uint16_t* x, const float* cs_row, int head_dim, int bits, int group,
                    int strict, uint8_t* idx, uint16_t* coset, uint16_t* scales);
void orc_decode_row(const uint8_t* idx, uint16_t coset, const uint16_t* scales,
                    const float* cs_row, int head_dim, int bits, int group, uint16_t* x_out);

/* Temporal delta of one row against the previous token's raw codes (in place)
 * and its inverse (in place, given the previous token's restored codes). */
void orc_delta_row(uint8_t* idx, uint16_t* coset, const uint8_t* prev_idx, uint16_t prev_coset,
                   int dp, int bits);
void orc_undelta_row(uint8_t* idx, uint16_t* coset, const uint8_t* prev_idx, uint16_t prev_coset,
                     int dp, int bits);

/* Whole tensor [slices][tokens][head_dim] fp16 -> sections idx / coset /
 * scales (rows in the same order).  cs: RoPE table or NULL.  delta_chunk: 0
 * off, else the delta restarts at every multiple of delta_chunk tokens.
 * strict: 0 relaxed, 1 strict, 2 strict in the joint format (coset words 0). */
void orc_compress_tensor(const uint16_t* x, int64_t slices, int tokens, int head_dim,
                         const float* cs, int bits, int group, int strict, int delta_chunk,
                         uint8_t* idx, uint16_t* coset, uint16_t* scales);
void orc_decompress_tensor(const uint8_t* idx, const uint16_t* coset, const uint16_t* scales,
                           int64_t slices, int tokens, int head_dim, const float* cs, int bits,
                           int group, int delta_chunk, int joint, uint16_t* x_out);

/* Strict joint format (strict = 2 in orc_compress_tensor, joint = 1 in
 * orc_decompress_tensor): per block, field 7 holds (m_7 >> 1) and the coset
 * bit above it; the low bit of m_7 is the parity of m_0 + ... + m_6.  Pack
 * writes the coset bits of `coset` into the row; split restores m_7 in place
 * and returns the coset word. */
void orc_joint_pack_row(uint8_t* idx, uint16_t coset, int dp, int bits);
uint16_t orc_joint_split_row(uint8_t* idx, int dp, int bits);

/* Counts of field values [0, 16), idx bytes [16, 272) and coset bits
 * [272], [273] over `rows` record rows; counts: 274 entries, overwritten. */
void orc_code_histogram(const uint8_t* idx, const uint16_t* coset, int64_t rows, int dp, int bits,
                        uint64_t* counts);

#ifdef __cplusplus
}
#endif
#endif
