/*
 * kv_append_oracle.c -- plain CPU definition of the KV append that precedes a
 * verify call: the W_r new key and value rows of every request's window are
 * written into their paged-cache slots, as bf16 or quantised to NVFP4.
 *
 * TEST INFRASTRUCTURE ONLY, under the same rules as spec_attn_oracle.c: only
 * the test suite, the smoke check and the bench's CPU-baseline leg may load
 * it; it shares no code, header, table or constant with the CUDA library.
 *
 * Placement (page "perf(dflash): widen the verify window past the compact
 * graph's four-row limit", section "What changed": the window writes its rows
 * into the cache, later steps overwrite the rows a rejection leaves stale,
 * and attention reads only seq_len entries).  seq_len_r already counts the
 * window, so window row i of request r is key ctx_r + i = seq_len_r - W_r + i
 * and lands in page block_table[r][pos / page_size], slot pos % page_size,
 * for K and V alike and for every KV head.
 *
 * NVFP4 quantisation.  The pages name "nvfp4" only (page "ChunkedSmallT
 * re-streams full KV per query chunk", section "Measurement"); the reading
 * here is the layout the attention oracle decodes -- one e2m1 code per
 * element, one e4m3 scale per 16 contiguous head_dim elements, one fp32
 * decode scale g per tensor, value = e2m1 * e4m3 * g -- with each block
 * quantised against the caller's g:
 *     amax = max |x_e| over the block's 16 elements
 *     s    = e4m3_rne_sat(amax / (6 * g))                (6: largest e2m1)
 *     den  = decoded(s) * g
 *     code = den == 0 ? +0 : e2m1_rne_sat(x_e / den)
 * Quotients and products are taken in binary32 (the pages fix no precision
 * for the quantiser; this is the kernel's, so both sides decide every code
 * on the same float), each operation rounded once to nearest even, in the
 * order written.  Rounding to e4m3 / e2m1 goes to the nearest representable
 * magnitude, ties to the even code, and saturates at the largest finite one
 * (448 / 6); the sign of x is kept, so a negative value that rounds to zero
 * gives the negative-zero code.  Inputs holding NaN or infinities are
 * outside the contract.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

double oracle_e2m1(unsigned code);   /* spec_attn_oracle.c */
double oracle_e4m3(unsigned byte);   /* spec_attn_oracle.c */

static float bf16_to_float(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round |x| to the nearest of the ordered magnitudes value(0) < value(1) <
 * ... < value(n-1) (ties to the even index, saturating at n-1).  Neighbouring
 * magnitudes and their midpoints are exact in double, so every comparison is
 * exact. */
static unsigned nearest_even(double a, double (*value)(unsigned), unsigned n) {
    unsigned b = 0;
    while (b + 1 < n && value(b + 1) <= a) ++b;
    if (b + 1 == n) return b;
    const double mid = 0.5 * (value(b) + value(b + 1));
    if (a > mid) return b + 1;
    if (a < mid) return b;
    return (b % 2 == 0) ? b : b + 1;
}

/* e4m3 magnitudes in code order: bytes 0x00..0x7E (0x7F is NaN). */
static double e4m3_mag(unsigned b) { return oracle_e4m3(b); }
/* e2m1 magnitudes in code order: codes 0..7. */
static double e2m1_mag(unsigned c) { return oracle_e2m1(c); }

/* binary32 -> OCP E4M3 byte, nearest-even, saturating at 448. */
unsigned oracle_e4m3_encode(float x) {
    const unsigned sign = signbit(x) ? 0x80u : 0u;
    return sign | nearest_even(fabs((double)x), e4m3_mag, 127u);
}

/* binary32 -> OCP E2M1 code (4 bits), nearest-even, saturating at 6. */
unsigned oracle_e2m1_encode(float x) {
    const unsigned sign = signbit(x) ? 0x8u : 0u;
    return sign | nearest_even(fabs((double)x), e2m1_mag, 8u);
}

/* One 16-element block: codes[8] (low nibble = even element), *scale. */
void oracle_nvfp4_quantise_block(const uint16_t x_bf16[16], float g, uint8_t codes[8],
                                 uint8_t* scale) {
    float x[16];
    float amax = 0.0f;
    for (int e = 0; e < 16; ++e) {
        x[e] = bf16_to_float(x_bf16[e]);
        const float a = fabsf(x[e]);
        if (a > amax) amax = a;
    }
    const float six_g = 6.0f * g;
    const float s = amax / six_g;
    const unsigned sb = oracle_e4m3_encode(s);
    const float den = (float)oracle_e4m3(sb) * g;
    unsigned c[16];
    for (int e = 0; e < 16; ++e) {
        if (den == 0.0f) {
            c[e] = 0u;
        } else {
            const float t = x[e] / den;
            c[e] = oracle_e2m1_encode(t);
        }
    }
    for (int k = 0; k < 8; ++k) codes[k] = (uint8_t)(c[2 * k] | (c[2 * k + 1] << 4));
    *scale = (uint8_t)sb;
}

/* Return codes (as spec_attn_oracle.c). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)

/*
 * Write every request's window rows into the pools, in place.
 *   k_new, v_new  [total_rows, Hkv, d] bf16 bit patterns, rows in q_indptr order
 *   kv_dtype 0: k_pool/v_pool bf16 [num_pages, Hkv, ps, d]
 *   kv_dtype 1: k_pool/v_pool codes [num_pages, Hkv, ps, d/2] bytes,
 *               k_scales/v_scales e4m3 [num_pages, Hkv, ps, d/16] bytes,
 *               k_gscale/v_gscale the tensors' decode scales (> 0)
 * A request whose window or seq_len is inconsistent, or whose block table
 * names a page outside [0, num_pages), makes the call return ORACLE_BAD_ARG
 * before anything is written.
 */
int spec_attn_oracle_append_kv(int num_reqs, int total_rows, int num_kv_heads, int head_dim,
                               int page_size, int num_pages, int kv_dtype, const uint16_t* k_new,
                               const uint16_t* v_new, void* k_pool, void* v_pool,
                               uint8_t* k_scales, uint8_t* v_scales, float k_gscale,
                               float v_gscale, const int32_t* block_table, int bt_stride,
                               const int32_t* seq_lens, const int32_t* q_indptr) {
    if (num_reqs < 0 || head_dim % 16 != 0 || page_size <= 0 || num_kv_heads <= 0) return ORACLE_BAD_ARG;
    if (kv_dtype == 1 && !(k_gscale > 0.0f && v_gscale > 0.0f)) return ORACLE_BAD_ARG;
    for (int r = 0; r < num_reqs; ++r) {
        const int row0 = q_indptr[r], w = q_indptr[r + 1] - row0, len = seq_lens[r];
        if (w < 0 || row0 < 0 || row0 + w > total_rows || len < w) return ORACLE_BAD_ARG;
        if (w > 0 && (len - 1) / page_size >= bt_stride) return ORACLE_BAD_ARG;
        for (int i = 0; i < w; ++i) {
            const int page = block_table[(int64_t)r * bt_stride + (len - w + i) / page_size];
            if (page < 0 || page >= num_pages) return ORACLE_BAD_ARG;
        }
    }
    const int d = head_dim;
    for (int r = 0; r < num_reqs; ++r) {
        const int row0 = q_indptr[r], w = q_indptr[r + 1] - row0, len = seq_lens[r];
        for (int i = 0; i < w; ++i) {
            const int pos = len - w + i;
            const int64_t page = block_table[(int64_t)r * bt_stride + pos / page_size];
            const int slot = pos % page_size;
            for (int h = 0; h < num_kv_heads; ++h) {
                const int64_t src = ((int64_t)(row0 + i) * num_kv_heads + h) * d;
                const int64_t dst = (page * num_kv_heads + h) * page_size + slot;   /* token-head index */
                if (kv_dtype == 0) {
                    memcpy((uint16_t*)k_pool + dst * d, k_new + src, (size_t)d * 2);
                    memcpy((uint16_t*)v_pool + dst * d, v_new + src, (size_t)d * 2);
                } else {
                    for (int b = 0; b < d / 16; ++b) {
                        oracle_nvfp4_quantise_block(k_new + src + 16 * b, k_gscale,
                                                    (uint8_t*)k_pool + dst * (d / 2) + 8 * b,
                                                    k_scales + dst * (d / 16) + b);
                        oracle_nvfp4_quantise_block(v_new + src + 16 * b, v_gscale,
                                                    (uint8_t*)v_pool + dst * (d / 2) + 8 * b,
                                                    v_scales + dst * (d / 16) + b);
                    }
                }
            }
        }
    }
    return ORACLE_OK;
}
