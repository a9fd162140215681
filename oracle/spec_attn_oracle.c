/*
 * spec_attn_oracle.c -- plain CPU fp64 oracle for speculative-decoding block
 * attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the bench's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA path, and the CUDA path never
 * calls it.
 *
 * What it computes (one call = one layer's attention for a batch of windows):
 *
 *   P requests.  Request r owns W_r = q_indptr[r+1] - q_indptr[r] query rows
 *   (its speculative window: the seed token plus k drafted tokens) and a
 *   paged K/V cache holding seq_len[r] keys.  The window's own W_r keys are
 *   the last W_r of those, so the context length is ctx_r = seq_len[r] - W_r.
 *   Key j of request r lives in page block_table[r][j / page_size] at slot
 *   j % page_size.  Only window rows get an output; context rows never do
 *   (page "DFlash2 leaves the paged graph fast path at every c>1 ...",
 *   sections "The cost" and "Scope").
 *
 *   Masks:
 *     causal-in-block: window row i sees keys 0 .. ctx_r + i (inclusive);
 *     non-causal:      every window row sees all seq_len[r] keys
 *                      (same page, section "The cost": the draft layers are
 *                      not causal, each row attends over its request's whole
 *                      span).
 *   Dense block operand (block_k / block_v non-NULL; bf16 caches): the
 *   window's own W_r keys are not in the cache but in dense [total_rows, Hkv,
 *   d] tensors, row by row in q_indptr order (page "DFlash2 leaves the paged
 *   graph fast path ...", section "Scope": the "Narrow" shape keeps the
 *   window's K/V apart from the paged context).  Key ctx_r + i is then row
 *   q_indptr[r] + i of the block tensors; keys below ctx_r come from the
 *   cache as before, and the block table need only cover them.  In the trace
 *   a block key counts like any other and adds -(1 + its row) to the slot sum.
 *   Sliding window (window_left > 0; causal only): the same page, same
 *   section, notes that the non-causal draft layers leave an attention window
 *   unapplied, without defining it.  The plainest reading, used here: row i
 *   sees only the window_left most recent keys up to its own,
 *   max(0, ctx_r + i - window_left + 1) .. ctx_r + i.  Non-causal calls take
 *   no window.
 *   Only keys below seq_len[r] are ever read (page "perf(dflash): widen the
 *   verify window past the compact graph's four-row limit", section "What
 *   changed": attention reads only seqlen entries).
 *
 *   GQA: query head h reads KV head h / G with G = Hq / Hkv.
 *
 *   For every selected (row, head):
 *     s_j = sm_scale * sum_e q[row,h,e] * K[j,kvh,e]       (j visible)
 *     m   = max_j s_j,  l = sum_j exp(s_j - m)
 *     O   = sum_j exp(s_j - m) * V[j,kvh,:] / l
 *     LSE = m + ln(l)                                     (natural log)
 *   all in fp64 from the exact input values (bf16, or NVFP4 decoded).
 *
 * Steps follow the materialised shape the pages describe for their fallback
 * path (page "DFlash2 leaves ...", section "The route change": gather every
 * context row out of the paged store, then attend): each request's K/V is
 * first gathered into a dense fp64 array through the block table, then a
 * dense softmax is taken per row.  No blocking, no online softmax, no split.
 *
 * NVFP4 KV (page "ChunkedSmallT re-streams full KV per query chunk",
 * section "Measurement", row "16K nvfp4"; the pages give no format, the
 * reading used here): each K/V element is an e2m1 code (two per byte, low
 * nibble = even element), each run of 16 contiguous head_dim elements has one
 * e4m3 scale byte, and each tensor has one fp32 global scale:
 *     value = e2m1(code) * e4m3(block scale) * global scale.
 *
 * Parallelism: OpenMP over independent output rows only; the arithmetic of
 * each output is the plain sequential definition above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- scalar decoders, written from the format definitions ---------------- */

/* bfloat16 is the upper half of an IEEE-754 binary32 bit pattern. */
static double oracle_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal (0 or 0.5).  No inf/NaN encodings. */
double oracle_e2m1(unsigned code) {
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * exponent 0 subnormal, S.1111.111 is NaN, no infinities. */
double oracle_e4m3(unsigned byte) {
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    double mag;
    if (e == 15u && m == 7u)
        mag = NAN;
    else if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

double oracle_bf16_value(unsigned bits) { return oracle_bf16((uint16_t)bits); }

/* Round an fp64 value to the nearest bfloat16 (ties to even), returning the
 * bf16 bit pattern.  Two steps: fp64 -> fp32 by the C cast (IEEE RNE), then
 * fp32 -> bf16 RNE.  The double rounding can differ from a direct fp64->bf16
 * RNE only when the fp32 result is exactly a bf16 midpoint, which callers of
 * the tolerance-based comparisons do not depend on. */
unsigned oracle_round_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN */
        return (unsigned)((u >> 16) | 0x40u) & 0xffffu;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (unsigned)(u >> 16) & 0xffffu;
}

/* ---- the oracle ---------------------------------------------------------- */

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEMORY (-2)

/*
 * kv_dtype 0: k_pool/v_pool are bf16 bit patterns [num_pages, Hkv, ps, d].
 * kv_dtype 1: k_pool/v_pool are NVFP4 codes [num_pages, Hkv, ps, d/2] bytes,
 *             k_scales/v_scales e4m3 bytes [num_pages, Hkv, ps, d/16].
 * mask_mode 0: causal-in-block, 1: non-causal.
 * window_left: 0 (none) or the sliding window of causal rows (keys).
 * block_k, block_v: NULL, or the dense block operand (bf16 bit patterns
 *        [total_rows, Hkv, d]; kv_dtype 0 only).
 * row_select: optional [total_rows * Hq] bytes; nonzero = compute that
 *             (row, head).  Unselected outputs are left untouched.
 * o:   [total_rows, Hq, d] fp64 (may be NULL when only the trace is wanted)
 * lse: [total_rows, Hq]    fp64 (may be NULL)
 * trace: optional [total_rows, Hq, 2] int64: number of visible keys and the
 *        sum of their physical slot ids (page * page_size + slot).
 */
int spec_attn_oracle_run(int num_reqs, int total_rows, int num_q_heads, int num_kv_heads,
                         int head_dim, int page_size, int num_pages, int mask_mode,
                         int window_left, int kv_dtype, double sm_scale, const uint16_t* q,
                         const void* k_pool, const void* v_pool, const uint8_t* k_scales,
                         const uint8_t* v_scales, double k_gscale, double v_gscale,
                         const uint16_t* block_k, const uint16_t* block_v,
                         const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                         const int32_t* q_indptr, const uint8_t* row_select, double* o,
                         double* lse, int64_t* trace) {
    if (num_reqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        page_size <= 0 || head_dim > 1024 || num_q_heads % num_kv_heads != 0)
        return ORACLE_BAD_ARG;
    if (kv_dtype == 1 && head_dim % 16 != 0) return ORACLE_BAD_ARG;
    if (window_left < 0 || (window_left > 0 && mask_mode != 0)) return ORACLE_BAD_ARG;
    if ((block_k == NULL) != (block_v == NULL) || (block_k && kv_dtype != 0)) return ORACLE_BAD_ARG;
    const int G = num_q_heads / num_kv_heads;
    const int d = head_dim;
    const int Hkv = num_kv_heads;

    for (int r = 0; r < num_reqs; ++r) {
        const int row0 = q_indptr[r];
        const int W = q_indptr[r + 1] - q_indptr[r];
        const int L = seq_lens[r];
        if (W < 0 || L < W || row0 < 0 || row0 + W > total_rows) return ORACLE_BAD_ARG;
        if (W == 0) continue;
        const int ctx = L - W;

        /* 1. Gather the request's keys and values into dense fp64 arrays
         *    Kd[j][kvh][e], Vd[j][kvh][e] through the block table. */
        size_t n = (size_t)L * (size_t)Hkv * (size_t)d;
        double* Kd = (double*)malloc(n * sizeof(double));
        double* Vd = (double*)malloc(n * sizeof(double));
        int64_t* slot_id = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
        if (!Kd || !Vd || !slot_id) {
            free(Kd);
            free(Vd);
            free(slot_id);
            return ORACLE_NO_MEMORY;
        }
        int bad_page = 0;
#pragma omp parallel for schedule(static) reduction(| : bad_page)
        for (int j = 0; j < L; ++j) {
            if (block_k && j >= ctx) {
                /* the window's own key: row row0 + (j - ctx) of the block operand */
                const size_t row = (size_t)row0 + (size_t)(j - ctx);
                slot_id[j] = -1 - (int64_t)row;
                for (int kvh = 0; kvh < Hkv; ++kvh) {
                    double* kd = Kd + ((size_t)j * Hkv + (size_t)kvh) * d;
                    double* vd = Vd + ((size_t)j * Hkv + (size_t)kvh) * d;
                    const uint16_t* kb = block_k + (row * Hkv + (size_t)kvh) * d;
                    const uint16_t* vb = block_v + (row * Hkv + (size_t)kvh) * d;
                    for (int e = 0; e < d; ++e) {
                        kd[e] = oracle_bf16(kb[e]);
                        vd[e] = oracle_bf16(vb[e]);
                    }
                }
                continue;
            }
            const int page = block_table[(size_t)r * (size_t)bt_stride + (size_t)(j / page_size)];
            const int slot = j % page_size;
            if (page < 0 || page >= num_pages) {
                bad_page = 1;
                continue;
            }
            slot_id[j] = (int64_t)page * page_size + slot;
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                const size_t tok = ((size_t)page * Hkv + (size_t)kvh) * (size_t)page_size + (size_t)slot;
                double* kd = Kd + ((size_t)j * Hkv + (size_t)kvh) * d;
                double* vd = Vd + ((size_t)j * Hkv + (size_t)kvh) * d;
                if (kv_dtype == 0) {
                    const uint16_t* kp = (const uint16_t*)k_pool + tok * (size_t)d;
                    const uint16_t* vp = (const uint16_t*)v_pool + tok * (size_t)d;
                    for (int e = 0; e < d; ++e) {
                        kd[e] = oracle_bf16(kp[e]);
                        vd[e] = oracle_bf16(vp[e]);
                    }
                } else {
                    const uint8_t* kc = (const uint8_t*)k_pool + tok * (size_t)(d / 2);
                    const uint8_t* vc = (const uint8_t*)v_pool + tok * (size_t)(d / 2);
                    const uint8_t* ks = k_scales + tok * (size_t)(d / 16);
                    const uint8_t* vs = v_scales + tok * (size_t)(d / 16);
                    for (int e = 0; e < d; ++e) {
                        unsigned kcode = (e % 2 == 0) ? (kc[e / 2] & 0xfu) : (kc[e / 2] >> 4);
                        unsigned vcode = (e % 2 == 0) ? (vc[e / 2] & 0xfu) : (vc[e / 2] >> 4);
                        kd[e] = oracle_e2m1(kcode) * oracle_e4m3(ks[e / 16]) * k_gscale;
                        vd[e] = oracle_e2m1(vcode) * oracle_e4m3(vs[e / 16]) * v_gscale;
                    }
                }
            }
        }
        if (bad_page) {
            free(Kd);
            free(Vd);
            free(slot_id);
            return ORACLE_BAD_ARG;
        }

        /* 2. Dense softmax attention for every selected (window row, head). */
        int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2) reduction(| : fail)
        for (int i = 0; i < W; ++i) {
            for (int h = 0; h < num_q_heads; ++h) {
                const int row = row0 + i;
                if (row_select && !row_select[(size_t)row * num_q_heads + h]) continue;
                const int kvh = h / G;
                const int hi = (mask_mode == 0) ? ctx + i : L - 1; /* inclusive */
                const int lo = (window_left > 0 && hi - window_left + 1 > 0) ? hi - window_left + 1 : 0;
                const int nvis = hi - lo + 1;
                double* s = (double*)malloc((size_t)nvis * sizeof(double));
                if (!s) {
                    fail = 1;
                    continue;
                }
                const uint16_t* qrow = q + ((size_t)row * num_q_heads + (size_t)h) * d;
                double qd[1024];
                for (int e = 0; e < d; ++e) qd[e] = oracle_bf16(qrow[e]);

                /* s[j] is the score of key lo + j */
                for (int j = 0; j < nvis; ++j) {
                    const double* kd = Kd + ((size_t)(lo + j) * Hkv + (size_t)kvh) * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += qd[e] * kd[e];
                    s[j] = sm_scale * acc;
                }
                double m = -INFINITY;
                for (int j = 0; j < nvis; ++j)
                    if (s[j] > m) m = s[j];
                double l = 0.0;
                for (int j = 0; j < nvis; ++j) {
                    s[j] = exp(s[j] - m); /* s now holds the unnormalised weights */
                    l += s[j];
                }
                if (o) {
                    double* orow = o + ((size_t)row * num_q_heads + (size_t)h) * d;
                    for (int e = 0; e < d; ++e) {
                        double acc = 0.0;
                        for (int j = 0; j < nvis; ++j)
                            acc += s[j] * Vd[((size_t)(lo + j) * Hkv + (size_t)kvh) * d + e];
                        orow[e] = acc / l;
                    }
                }
                if (lse) lse[(size_t)row * num_q_heads + h] = m + log(l);
                if (trace) {
                    int64_t sum = 0;
                    for (int j = 0; j < nvis; ++j) sum += slot_id[lo + j];
                    trace[((size_t)row * num_q_heads + h) * 2 + 0] = nvis;
                    trace[((size_t)row * num_q_heads + h) * 2 + 1] = sum;
                }
                free(s);
            }
        }
        free(Kd);
        free(Vd);
        free(slot_id);
        if (fail) return ORACLE_NO_MEMORY;
    }
    return ORACLE_OK;
}

/* Number of threads the oracle's parallel regions use. */
int spec_attn_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
