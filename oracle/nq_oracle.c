/*
 * nq_oracle.c -- plain CPU oracle for E8 lattice KV-cache compression.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  Written from the
 * method's description; shares no code with the CUDA library.
 *
 * Build: cc -std=c11 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -lm
 * (oracle/build.py).  Every function follows the steps of the method in the
 * order the pages give them; readings of the pages are marked "Reading:".
 */
#include "nq_oracle.h"

#include <math.h>
#include <string.h>

int orc_padded_dim(int head_dim) {
    int p = 8;
    while (p < head_dim) p *= 2;
    return p;
}

/* ---------------------------------------------------------------- binary16 */

float orc_h2f(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    float v;
    if (expo == 0) {
        v = ldexpf((float)mant, -24); /* zero / subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(mant | 0x400), expo - 25); /* (1.mant) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

uint16_t orc_f2h_rn(float f) {
    /* Round the binary32 value to the nearest binary16 value, ties to even. */
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    float a = fabsf(f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00u); /* rounds past 65504 */
    if (a < ldexpf(1.0f, -14)) {
        /* subnormal range: multiples of 2^-24; a * 2^24 is exact in binary32 */
        float q = rintf(ldexpf(a, 24));
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 is the smallest normal */
    }
    int e;
    (void)frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    int expo = e - 1;     /* a in [2^expo, 2^(expo+1)) */
    float q = rintf(ldexpf(a, 10 - expo)); /* significand scaled to [1024, 2048] */
    if (q >= 2048.0f) {
        q = 1024.0f;
        expo += 1;
    }
    return (uint16_t)(sign | (uint16_t)((expo + 15) << 10) | ((uint16_t)q & 0x3ffu));
}

/* -------------------------------------------------------------------- RoPE */

/* Reading: the pages name split-half ("rotate_half", Llama/Mistral) rotary
 * embedding [README "Supported models"; WALK "What Makes This Hard in
 * Practice" item 2] but print no formula; the standard one is used: pair
 * (i, i + D/2), frequency theta^(-2i/D), angle pos * frequency. */
void orc_rope_table(const int32_t* pos, int tokens, int head_dim, float theta, float* cs) {
    int half = head_dim / 2;
    for (int t = 0; t < tokens; ++t) {
        double p = pos ? (double)pos[t] : (double)t;
        for (int i = 0; i < half; ++i) {
            double freq = pow((double)theta, -2.0 * (double)i / (double)head_dim);
            double ang = p * freq;
            cs[((size_t)t * half + i) * 2 + 0] = (float)cos(ang);
            cs[((size_t)t * half + i) * 2 + 1] = (float)sin(ang);
        }
    }
}

/* Remove: rotate each pair by -angle.  fp32 order: one product, one fmaf. */
void orc_rope_remove(float* x, int head_dim, const float* cs_row) {
    int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        float c = cs_row[2 * i], s = cs_row[2 * i + 1];
        float a = x[i], b = x[i + half];
        x[i] = fmaf(a, c, b * s);
        x[i + half] = fmaf(b, c, -(a * s));
    }
}

/* Apply: rotate each pair by +angle (the inverse of orc_rope_remove). */
void orc_rope_apply(float* x, int head_dim, const float* cs_row) {
    int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        float c = cs_row[2 * i], s = cs_row[2 * i + 1];
        float a = x[i], b = x[i + half];
        x[i] = fmaf(a, c, -(b * s));
        x[i + half] = fmaf(b, c, a * s);
    }
}

/* ---------------------------------------------------------------- Hadamard */

/* [QUANT "Handling outliers"]: each vector is multiplied by the transpose of
 * the Sylvester Hadamard matrix H, which is symmetric.  Reading: the unnormalised transform is
 * used; its factor sqrt(n) is absorbed by the group scale (compression) and
 * divided out exactly as a power of two (decompression). */
static void butterfly_stage(float* x, int n, int h) {
    for (int i = 0; i < n; i += 2 * h) {
        for (int j = i; j < i + h; ++j) {
            float a = x[j], b = x[j + h];
            x[j] = a + b;
            x[j + h] = a - b;
        }
    }
}

/* Textbook order h = 1, 2, 4, ..., n/2 (used by decompression). */
void orc_fwht(float* x, int n) {
    for (int h = 1; h < n; h *= 2) butterfly_stage(x, n, h);
}

/* Reading: every butterfly order computes H x; in fp32 the order fixes the
 * rounding, so compression fixes one: the textbook order with its last two
 * stages exchanged (h = 1, ..., n/8, then n/2, then n/4). */
void orc_fwht_forward(float* x, int n) {
    for (int h = 1; h < n / 4; h *= 2) butterfly_stage(x, n, h);
    if (n >= 4) butterfly_stage(x, n, n / 2);
    if (n >= 4) butterfly_stage(x, n, n / 4);
    if (n == 2) butterfly_stage(x, n, 1);
}

/* ------------------------------------------------------------- group scale */

static uint16_t half_next_up(uint16_t v) { return (uint16_t)(v + 1); }   /* v >= 0 finite */
static uint16_t half_next_down(uint16_t v) { return (uint16_t)(v - 1); } /* v > 0 */

/* [WALK "Python Implementation" quantize(): the scale is the absolute maximum
 * over half the number of levels].
 * Reading: the divisor is (levels - 1)/2 so that the half-integer grid of the
 * box holds exactly 2^bits levels (the pages' levels/2 box holds more lattice
 * points than b bits can index).  The scale is stored as binary16, one per
 * group [WALK "Why Per-Group Scaling?" uses groups of 8 values and the
 * per-head variant groups of 128; this format takes the group size as a
 * parameter, 64 in the target workloads]; the smallest binary16 value
 * that does not clip is taken, so no scaled coordinate leaves the box.  The
 * Hadamard gain dp is folded in so the stored scale never overflows binary16. */
uint16_t orc_group_scale(float amax, int bits, int dp) {
    if (!(amax > 0.0f)) return 0;
    float step = (float)dp * (float)((1 << bits) - 1) * 0.5f; /* exact small integer */
    float q = amax / step;
    uint16_t v = orc_f2h_rn(q);
    while (orc_h2f(v) * step < amax) v = half_next_up(v); /* products are exact */
    while (v > 0 && orc_h2f(half_next_down(v)) * step >= amax) v = half_next_down(v);
    return v;
}

/* ---------------------------------------------------------- E8 nearest point */

/* One coset's candidate [WALK "The Conway-Sloane Nearest-Point Algorithm"]:
 * round every coordinate to the coset, then, if the even-sum rule applies and
 * the sum is odd, move the coordinate that was farthest from its rounded value
 * one step toward the input (the prose's rule; the printed code's argmin is not
 * the nearest point).  Returns the squared distance.
 *
 * Readings:
 *  - box: with a b-bit code each coordinate stays in [-hi, hi], hi = 2^(b-1)-1
 *    for integers and (2^b-1)/2 for half-integers; rounding clamps into the box
 *    and a fix-up step that would leave it goes the other way.  This makes the
 *    result the exact nearest point of codebook-and-box.
 *  - ties: integers round half to even (torch.round); the half-integer point of
 *    u is ceil(u) - 1/2, so an integer u goes down.
 *  - the fix-up coordinate is the first index of the largest score, the score
 *    being |e| for a step toward u and -|e| for a step away from it.
 *  - distance: sum of e_j^2 in j order by fmaf, plus the fix-up's cost
 *    1 - 2*score (the added cost of the flip the prose describes), evaluated as
 *    d + fmaf(-2, score, 1). */
static float coset_candidate(const float* u, int half, int enforce_parity, int bits, float* r) {
    float hi;
    if (bits == 0) hi = INFINITY;
    else if (half) hi = (float)((1 << bits) - 1) * 0.5f;
    else hi = (float)((1 << (bits - 1)) - 1);

    float e[8];
    long sum = 0;
    for (int j = 0; j < 8; ++j) {
        float v = half ? ceilf(u[j]) - 0.5f : rintf(u[j]);
        if (v > hi) v = hi;
        if (v < -hi) v = -hi;
        r[j] = v;
        e[j] = u[j] - v;
        sum += (long)(half ? v - 0.5f : v); /* integer part; half adds 8 * 1/2 = 4 */
    }
    float d = 0.0f;
    for (int j = 0; j < 8; ++j) d = fmaf(e[j], e[j], d);

    if (enforce_parity && (sum % 2) != 0) {
        int k = -1;
        float best = 0.0f, best_dir = 0.0f;
        for (int j = 0; j < 8; ++j) {
            float dir = (e[j] >= 0.0f) ? 1.0f : -1.0f;
            float score = fabsf(e[j]);
            if (r[j] + dir > hi || r[j] + dir < -hi) {
                dir = -dir;
                score = -score;
            }
            if (k < 0 || score > best) {
                k = j;
                best = score;
                best_dir = dir;
            }
        }
        r[k] += best_dir;
        d = d + fmaf(-2.0f, best, 1.0f);
    }
    return d;
}

/* E8 = D8 u (D8 + 1/2) [WALK "The E8 Lattice, Briefly"]: nearest point of each
 * coset, then the closer one; a tie goes to the integer coset (the printed
 * code replaces the integer point only where d_half < d_int).  strict = 0 is
 * the relaxed variant [RELAX]: the half-integer coset drops its even-sum rule,
 * the integer coset keeps it. */
int orc_e8_block(const float* u, int strict, int bits, float* r) {
    float r0[8], r1[8];
    float d0 = coset_candidate(u, 0, 1, bits, r0);
    float d1 = coset_candidate(u, 1, strict, bits, r1);
    int c = (d1 < d0) ? 1 : 0;
    memcpy(r, c ? r1 : r0, sizeof(r0));
    return c;
}

void orc_e8_nearest(const float* u, float* r, int64_t n_blocks, int strict, int bits) {
    for (int64_t b = 0; b < n_blocks; ++b) (void)orc_e8_block(u + 8 * b, strict, bits, r + 8 * b);
}

/* ------------------------------------------------------------------ fields */

/* Reading: coordinate i's b-bit code sits at bit i*b of the row's bit string,
 * least significant bit first, bytes little-endian [WALK "Bit Rate
 * Accounting": b bits for each of a block's 8 coordinates, the indices packed
 * into bytes]. */
static unsigned get_field(const uint8_t* idx, int i, int bits) {
    unsigned v = 0;
    for (int q = 0; q < bits; ++q) {
        int bit = i * bits + q;
        v |= (unsigned)((idx[bit >> 3] >> (bit & 7)) & 1u) << q;
    }
    return v;
}

static void put_field(uint8_t* idx, int i, int bits, unsigned v) {
    for (int q = 0; q < bits; ++q) {
        int bit = i * bits + q;
        idx[bit >> 3] = (uint8_t)((idx[bit >> 3] & ~(1u << (bit & 7))) | (((v >> q) & 1u) << (bit & 7)));
    }
}

/* ------------------------------------------------------------------- rows */

void orc_encode_row(const uint16_t* x, const float* cs_row, int head_dim, int bits, int group,
                    int strict, uint8_t* idx, uint16_t* coset, uint16_t* scales) {
    int dp = orc_padded_dim(head_dim);
    float y[128];
    for (int i = 0; i < dp; ++i) y[i] = (i < head_dim) ? orc_h2f(x[i]) : 0.0f;
    if (cs_row) orc_rope_remove(y, head_dim, cs_row);
    orc_fwht_forward(y, dp); /* zero padding to dp happened above */

    memset(idx, 0, (size_t)dp * bits / 8);
    uint16_t cw = 0;
    int levels = 1 << bits;
    for (int g = 0; g < dp / group; ++g) {
        float amax = 0.0f;
        for (int i = g * group; i < (g + 1) * group; ++i) amax = fmaxf(amax, fabsf(y[i]));
        uint16_t sc = orc_group_scale(amax, bits, dp);
        scales[g] = sc;
        float inv = (sc == 0) ? 0.0f : 1.0f / (orc_h2f(sc) * (float)dp);
        for (int blk = g * group / 8; blk < (g + 1) * group / 8; ++blk) {
            float u[8], r[8];
            for (int j = 0; j < 8; ++j) u[j] = y[8 * blk + j] * inv;
            int c = orc_e8_block(u, strict, bits, r);
            cw |= (uint16_t)(c << blk);
            /* index = point + offset: integers [0, L-2], half-integers [0, L-1] */
            float off = c ? (float)(levels - 1) * 0.5f : (float)(levels / 2 - 1);
            for (int j = 0; j < 8; ++j) put_field(idx, 8 * blk + j, bits, (unsigned)(r[j] + off));
        }
    }
    *coset = cw;
}

void orc_decode_row(const uint8_t* idx, uint16_t coset, const uint16_t* scales,
                    const float* cs_row, int head_dim, int bits, int group, uint16_t* x_out) {
    int dp = orc_padded_dim(head_dim);
    int levels = 1 << bits;
    float y[128];
    for (int i = 0; i < dp; ++i) {
        int c = (coset >> (i / 8)) & 1;
        float off = c ? (float)(levels - 1) * 0.5f : (float)(levels / 2 - 1);
        float r = (float)get_field(idx, i, bits) - off;
        y[i] = r * orc_h2f(scales[i / group]); /* exact: few significant bits */
    }
    /* x = H (r * sc): H H = dp I and u = y / (sc * dp) */
    orc_fwht(y, dp);
    if (cs_row) orc_rope_apply(y, head_dim, cs_row);
    /* Reading: the cache was finite, so the reconstruction saturates at the
     * largest finite fp16 value instead of overflowing to infinity. */
    for (int i = 0; i < head_dim; ++i) x_out[i] = orc_f2h_rn(fmaxf(fminf(y[i], 65504.0f), -65504.0f));
}

/* [NEG, temporal delta entry]: subtract the previous token's index.  Reading:
 * the forward difference (this token's code minus the previous token's) per
 * field modulo 2^b, the coset bits by exclusive or; scales are stored as they
 * are.  (The entry's wording, read literally, subtracts in the other order;
 * both orders are lossless and give the same symbol entropy.) */
void orc_delta_row(uint8_t* idx, uint16_t* coset, const uint8_t* prev_idx, uint16_t prev_coset,
                   int dp, int bits) {
    unsigned mask = (1u << bits) - 1u;
    for (int i = 0; i < dp; ++i)
        put_field(idx, i, bits, (get_field(idx, i, bits) - get_field(prev_idx, i, bits)) & mask);
    *coset = (uint16_t)(*coset ^ prev_coset);
}

void orc_undelta_row(uint8_t* idx, uint16_t* coset, const uint8_t* prev_idx, uint16_t prev_coset,
                     int dp, int bits) {
    unsigned mask = (1u << bits) - 1u;
    for (int i = 0; i < dp; ++i)
        put_field(idx, i, bits, (get_field(idx, i, bits) + get_field(prev_idx, i, bits)) & mask);
    *coset = (uint16_t)(*coset ^ prev_coset);
}

/* ----------------------------------------------------------------- tensors */

/* The strict joint format (strict = 2).  Reading: the pages print no format
 * for it; in strict E8 the field sum of a block is even in both cosets (the
 * coordinate sum is even and the offsets add 8 times (2^b - 2)/2 or 8 times
 * (2^b - 1)/2, both even), so the low bit of m_7 follows from m_0..m_6 and its
 * place holds the block's coset bit: field 7 stores (m_7 >> 1) with the coset
 * bit above it, and a block is exactly 8b bits. */
void orc_joint_pack_row(uint8_t* idx, uint16_t coset, int dp, int bits) {
    for (int k = 0; k < dp / 8; ++k) {
        unsigned m7 = get_field(idx, 8 * k + 7, bits);
        unsigned c = (coset >> k) & 1u;
        put_field(idx, 8 * k + 7, bits, (m7 >> 1) | (c << (bits - 1)));
    }
}

uint16_t orc_joint_split_row(uint8_t* idx, int dp, int bits) {
    unsigned coset = 0;
    for (int k = 0; k < dp / 8; ++k) {
        unsigned f = get_field(idx, 8 * k + 7, bits);
        unsigned c = f >> (bits - 1);
        unsigned half7 = f & ((1u << (bits - 1)) - 1u);
        unsigned sum = 0;
        for (int j = 0; j < 7; ++j) sum += get_field(idx, 8 * k + j, bits);
        put_field(idx, 8 * k + 7, bits, (half7 << 1) | (sum & 1u));
        coset |= c << k;
    }
    return (uint16_t)coset;
}

void orc_compress_tensor(const uint16_t* x, int64_t slices, int tokens, int head_dim,
                         const float* cs, int bits, int group, int strict, int delta_chunk,
                         uint8_t* idx, uint16_t* coset, uint16_t* scales) {
    int dp = orc_padded_dim(head_dim);
    size_t rb = (size_t)dp * bits / 8;
    int ng = dp / group;
    uint8_t prev_idx[64];
    uint16_t prev_coset = 0;
    for (int64_t s = 0; s < slices; ++s) {
        for (int t = 0; t < tokens; ++t) {
            int64_t row = s * tokens + t;
            const float* cs_row = cs ? cs + (size_t)t * head_dim : 0; /* D/2 pairs of 2 */
            orc_encode_row(x + row * head_dim, cs_row, head_dim, bits, group, strict ? 1 : 0,
                           idx + row * rb, coset + row, scales + row * ng);
            if (strict == 2) { /* joint format: the coset bits move into the codes */
                orc_joint_pack_row(idx + row * rb, coset[row], dp, bits);
                coset[row] = 0;
            }
            if (delta_chunk > 0) {
                uint8_t raw_idx[64];
                uint16_t raw_coset = coset[row];
                memcpy(raw_idx, idx + row * rb, rb);
                if (t % delta_chunk != 0)
                    orc_delta_row(idx + row * rb, coset + row, prev_idx, prev_coset, dp, bits);
                memcpy(prev_idx, raw_idx, rb);
                prev_coset = raw_coset;
            }
        }
    }
}

void orc_decompress_tensor(const uint8_t* idx, const uint16_t* coset, const uint16_t* scales,
                           int64_t slices, int tokens, int head_dim, const float* cs, int bits,
                           int group, int delta_chunk, int joint, uint16_t* x_out) {
    int dp = orc_padded_dim(head_dim);
    size_t rb = (size_t)dp * bits / 8;
    int ng = dp / group;
    uint8_t cur_idx[64];
    uint16_t cur_coset = 0;
    for (int64_t s = 0; s < slices; ++s) {
        for (int t = 0; t < tokens; ++t) {
            int64_t row = s * tokens + t;
            const float* cs_row = cs ? cs + (size_t)t * head_dim : 0;
            if (delta_chunk > 0 && t % delta_chunk != 0) {
                uint8_t prev[64];
                uint16_t prev_coset = cur_coset;
                memcpy(prev, cur_idx, rb);
                memcpy(cur_idx, idx + row * rb, rb);
                cur_coset = coset[row];
                orc_undelta_row(cur_idx, &cur_coset, prev, prev_coset, dp, bits);
            } else {
                memcpy(cur_idx, idx + row * rb, rb);
                cur_coset = coset[row];
            }
            if (joint) {
                uint8_t split[64];
                memcpy(split, cur_idx, rb);
                uint16_t c = orc_joint_split_row(split, dp, bits);
                orc_decode_row(split, c, scales + row * ng, cs_row, head_dim, bits, group, x_out + row * head_dim);
            } else {
                orc_decode_row(cur_idx, cur_coset, scales + row * ng, cs_row, head_dim, bits, group,
                               x_out + row * head_dim);
            }
        }
    }
}

/* Symbol statistics of compressed rows, for the entropy report (the pages
 * delta-code the packed indices and hand them to an entropy coder: "E8
 * walkthrough", "Bit Rate Accounting").  counts[274]: [0, 16) field values,
 * [16, 272) idx bytes, [272] integer-coset blocks, [273] half-coset blocks.
 * Plain counting over every field, byte and block of `rows` record rows;
 * coset NULL (the joint format) takes each block's top stored bit. */
void orc_code_histogram(const uint8_t* idx, const uint16_t* coset, int64_t rows, int dp, int bits,
                        uint64_t* counts) {
    size_t rb = (size_t)dp * bits / 8;
    int nb = dp / 8;
    for (int i = 0; i < 274; ++i) counts[i] = 0;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* row = idx + (size_t)r * rb;
        for (int i = 0; i < dp; ++i) counts[get_field(row, i, bits)] += 1;
        for (size_t b = 0; b < rb; ++b) counts[16 + row[b]] += 1;
        for (int k = 0; k < nb; ++k) {
            /* joint format (no coset words): the top bit of field 7 */
            unsigned c = coset ? ((coset[r] >> k) & 1u) : (get_field(row, 8 * k + 7, bits) >> (bits - 1));
            counts[272 + c] += 1;
        }
    }
}
