// Device helpers shared by the split-KV kernels and the LSE merge.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "spec_attn_internal.h"

namespace spec_attn {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Two floats as fp16 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_half2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// A bf16 pair as an fp16 pair (round to nearest even, saturating to +-65504).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));   // first operand -> upper half
    return d;
}

// Hardware base-2 exponential (MUFU.EX2), flush-to-zero; ex2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// OCP FP4 E2M1 code (low 4 bits) -> float.  Sign bit 3, exponent bits 2..1
// (bias 1), mantissa bit 0; exponent 0 encodes 0 and 0.5.  The magnitude's
// fp32 bit pattern is assembled directly: exponent field e-1+127, mantissa
// top bit m.
__device__ __forceinline__ float e2m1_to_float(uint32_t code) {
    const uint32_t e = (code >> 1) & 3u, m = code & 1u;
    uint32_t mag = (e != 0u) ? (((e + 126u) << 23) | (m << 22)) : (m ? 0x3f000000u : 0u);
    return __uint_as_float(mag | ((code & 8u) << 28));
}

// OCP FP8 E4M3 byte -> float.  Bias 7, exponent 0 subnormal (m * 2^-9),
// S.1111.111 is NaN, no infinities.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float mag;
    if (e == 15u && m == 7u)
        mag = __uint_as_float(0x7fc00000u);
    else if (e == 0u)
        mag = (float)m * 0.001953125f;  // 2^-9
    else
        mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80u) ? -mag : mag;
}

// A request's window and cache, validated against the plan.  Invalid
// requests set a status bit (when status != nullptr) and are skipped.
struct ReqInfo {
    int row0;       // first Q/O row
    int w;          // window rows
    int len;        // seq_len (keys incl. the window's)
    int ctx;        // len - w
    int cache_len;  // keys read from the cache: len, or ctx with the dense block operand
    int key_base;   // first key any row may see, rounded down to the split alignment
    int nsplits;    // splits of keys_per_split covering [key_base, cache_len) (at least one)
    int split0;     // key_base / keys_per_split (whole when the alignment is keys_per_split)
};

// window_left > 0: a causal sliding window; no row sees a key below
// ctx - window_left + 1 (row 0's bound), so the splits start at that key
// rounded down to split_align (64, the key tile; or keys_per_split where
// split boundaries must sit at fixed key positions).  dense_block: the
// window's own keys come from the dense block operand; the splits cover the
// cache keys [key_base, ctx) and the last one also takes the window's keys.
__device__ __forceinline__ bool load_request(const int32_t* seq_lens, const int32_t* q_indptr,
                                             int r, int max_w, int total_rows,
                                             long long max_seq_len, int cap_keys,
                                             int keys_per_split, unsigned int* status,
                                             ReqInfo& ri, int window_left = 0, int split_align = 64,
                                             int dense_block = 0) {
    // three independent loads: one memory round trip
    const int row0 = q_indptr[r];
    const int row1 = q_indptr[r + 1];
    const int len = seq_lens[r];
    const int w = row1 - row0;
    if (w < 0 || w > max_w || row0 < 0 || row1 > total_rows) {
        if (status) atomicOr(status, kDevBadWindow);
        return false;
    }
    if (w == 0) return false;
    const int cache_len = dense_block ? len - w : len;
    if (len < w || (long long)len > max_seq_len || cache_len > cap_keys) {
        if (status) atomicOr(status, kDevBadSeqLen);
        return false;
    }
    ri.row0 = row0;
    ri.w = w;
    ri.len = len;
    ri.ctx = len - w;
    ri.cache_len = cache_len;
    ri.key_base = 0;
    ri.split0 = 0;
    if (window_left > 0) {
        const int lo0 = max(0, ri.ctx - window_left + 1);
        ri.key_base = lo0 / split_align * split_align;
        ri.split0 = ri.key_base / keys_per_split;
    }
    ri.nsplits = max(1, (cache_len - ri.key_base + keys_per_split - 1) / keys_per_split);
    return true;
}

// Programmatic dependent launch controls (sm_90+).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace spec_attn
