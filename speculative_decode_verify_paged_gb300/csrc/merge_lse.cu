// LSE merge of split-KV partials (the "reduce kernel" that follows
// key-splitting on the page "ChunkedSmallT re-streams full KV per query chunk
// (DFlash K>=8 verify at long context)", section "Finding").
//
// Split s of a request leaves, per (row, head), the normalised partial
// O_s = (sum_j 2^(s_j - m_s) v_j) / l_s in fp32 and lse_s = m_s + log2 l_s
// (base 2, scores pre-scaled by log2 e; -inf when the split saw no key of
// that row).  The merge is
//   lse = log2 sum_s 2^(lse_s),  O = sum_s 2^(lse_s - lse) O_s,
// written as bf16 O (round to nearest even) and natural-log LSE (lse * ln 2).
//
// One CTA per (window row, query head).  Its 256 threads are split into
// split groups x head_dim vectors: thread (g, v) owns float4 v of the splits
// g, g + SG, g + 2 SG, ...  It issues the loads of up to kBatch of its splits
// (LSE and partial row) at once -- one memory round trip for the usual split
// counts -- and folds them with a running maximum (online LSE combination).
// The groups are then combined once through shared memory.  Requests with a
// single split were finished by the split kernel and are skipped here.  The
// kernel may be launched as a programmatic dependent of the split kernel: it
// waits on griddepcontrol before touching partials.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace spec_attn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kBatch = 8;

template <int D>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_lse_kernel(const MergeParams p) {
    constexpr int VEC = D / 4;                 // float4 vectors per row
    constexpr int SG = kMergeThreads / VEC;    // split groups
    __shared__ float4 part[SG][VEC];
    __shared__ float part_m[SG], part_l[SG];
    const int tid = threadIdx.x;
    const int v = tid % VEC, g = tid / VEC;
    const int pair = blockIdx.x;
    const int r = blockIdx.y;
    const int i = pair / p.num_q_heads;
    const int h = pair % p.num_q_heads;

    ReqInfo ri;
    const bool ok = load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                                 p.bt_capacity_keys, p.keys_per_split, nullptr, ri);
    if (!ok || i >= ri.w || ri.nsplits <= 1) {
        pdl_wait_primary();
        return;
    }
    const size_t oi = (size_t)(ri.row0 + i) * p.num_q_heads + h;
    const size_t split_stride = (size_t)p.total_rows * p.num_q_heads;
    const int n = ri.nsplits;
    // Wait for the split kernel's partials (no-op without a programmatic edge).
    pdl_wait_primary();

    float m_run = -INFINITY, l_run = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = g; s0 < n; s0 += SG * kBatch) {
        float ls[kBatch];
        float4 o[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int s = s0 + k * SG;
            if (s < n) {
                ls[k] = p.ws_lse[s * split_stride + oi];
                o[k] = *reinterpret_cast<const float4*>(p.ws_o + (s * split_stride + oi) * D + v * 4);
            } else {
                ls[k] = -INFINITY;
                o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            if (ls[k] == -INFINITY) continue;
            if (ls[k] > m_run) {
                const float a = fast_exp2(m_run - ls[k]);   // 0 when m_run is -inf
                acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
                l_run *= a;
                m_run = ls[k];
            }
            const float w = fast_exp2(ls[k] - m_run);
            acc.x = fmaf(w, o[k].x, acc.x);
            acc.y = fmaf(w, o[k].y, acc.y);
            acc.z = fmaf(w, o[k].z, acc.z);
            acc.w = fmaf(w, o[k].w, acc.w);
            l_run += w;
        }
    }
    part[g][v] = acc;
    if (v == 0) {
        part_m[g] = m_run;
        part_l[g] = l_run;
    }
    __syncthreads();
    if (g != 0) return;
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < SG; ++k) mx = fmaxf(mx, part_m[k]);
    float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
#pragma unroll
    for (int k = 0; k < SG; ++k) {
        if (part_m[k] == -INFINITY) continue;
        const float a = fast_exp2(part_m[k] - mx);
        tot.x = fmaf(a, part[k][v].x, tot.x);
        tot.y = fmaf(a, part[k][v].y, tot.y);
        tot.z = fmaf(a, part[k][v].z, tot.z);
        tot.w = fmaf(a, part[k][v].w, tot.w);
        wsum = fmaf(a, part_l[k], wsum);
    }
    const float inv = 1.f / wsum;
    const uint32_t lo = float_to_bf16_bits(tot.x * inv) | ((uint32_t)float_to_bf16_bits(tot.y * inv) << 16);
    const uint32_t hi = float_to_bf16_bits(tot.z * inv) | ((uint32_t)float_to_bf16_bits(tot.w * inv) << 16);
    *reinterpret_cast<uint2*>(p.o + oi * D + v * 4) = make_uint2(lo, hi);
    if (p.lse && v == 0) p.lse[oi] = (mx + log2f(wsum)) * kLn2;
}

}  // namespace

cudaError_t merge_launch(const MergeParams& p, cudaStream_t stream, bool programmatic) {
    dim3 grid(p.max_w * p.num_q_heads, p.num_reqs, 1);
    dim3 block(kMergeThreads, 1, 1);
    void (*k)(const MergeParams) = nullptr;
    switch (p.head_dim) {
        case 64: k = &merge_lse_kernel<64>; break;
        case 128: k = &merge_lse_kernel<128>; break;
        case 256: k = &merge_lse_kernel<256>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace spec_attn
