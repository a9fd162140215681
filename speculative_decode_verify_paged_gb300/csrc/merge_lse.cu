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
// One warp per (window row, query head); lane l owns head_dim elements
// [l*D/32, (l+1)*D/32), so every partial row is read with coalesced 16-byte
// loads.  Requests with a single split were finished by the split kernel and
// are skipped here.  The kernel may be launched as a programmatic dependent
// of the split kernel: it waits on griddepcontrol before touching partials.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace spec_attn {
namespace {

constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_lse_kernel(const MergeParams p) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int r = blockIdx.y;
    const int i = pair / p.num_q_heads;
    const int h = pair % p.num_q_heads;

    ReqInfo ri;
    const bool ok = load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                                 p.bt_capacity_keys, p.keys_per_split, nullptr, ri);
    // Wait for the split kernel's partials (no-op without a programmatic edge).
    pdl_wait_primary();
    if (!ok || i >= ri.w || ri.nsplits <= 1) return;

    const size_t oi = (size_t)(ri.row0 + i) * p.num_q_heads + h;
    const size_t split_stride = (size_t)p.total_rows * p.num_q_heads;
    const int n = ri.nsplits;

    float mx = -INFINITY;
    for (int s = lane; s < n; s += 32) mx = fmaxf(mx, p.ws_lse[s * split_stride + oi]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));

    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < n; ++s) {
        const float ls = p.ws_lse[s * split_stride + oi];
        const float w = (ls == -INFINITY) ? 0.f : fast_exp2(ls - mx);
        wsum += w;
        const float* src = p.ws_o + (s * split_stride + oi) * D + lane * DPL;
        if constexpr (DPL % 4 == 0) {
#pragma unroll
            for (int e = 0; e < DPL; e += 4) {
                const float4 v = *reinterpret_cast<const float4*>(src + e);
                acc[e] = fmaf(w, v.x, acc[e]);
                acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
                acc[e + 2] = fmaf(w, v.z, acc[e + 2]);
                acc[e + 3] = fmaf(w, v.w, acc[e + 3]);
            }
        } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            acc[0] = fmaf(w, v.x, acc[0]);
            acc[1] = fmaf(w, v.y, acc[1]);
        }
    }
    const float inv = 1.f / wsum;
    uint16_t* op = p.o + oi * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
        const uint32_t lo = float_to_bf16_bits(acc[e] * inv);
        const uint32_t hi = float_to_bf16_bits(acc[e + 1] * inv);
        *reinterpret_cast<uint32_t*>(op + e) = lo | (hi << 16);
    }
    if (p.lse && lane == 0) p.lse[oi] = (mx + log2f(wsum)) * kLn2;
}

}  // namespace

cudaError_t merge_launch(const MergeParams& p, cudaStream_t stream, bool programmatic) {
    const int pairs = p.max_w * p.num_q_heads;
    dim3 grid((pairs + kMergeWarps - 1) / kMergeWarps, p.num_reqs, 1);
    dim3 block(kMergeWarps * 32, 1, 1);
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
