// LSE merge of split-KV partials (the "reduce kernel" that follows
// key-splitting on the page "ChunkedSmallT re-streams full KV per query chunk
// (DFlash K>=8 verify at long context)", section "Finding").
//
// Split s of a request leaves, per (row, head), the normalised partial
// O_s = (sum_j 2^(s_j - m_s) v_j) / l_s, stored as fp16 of O_s / scale_s with
// scale_s = max |O_s|, and lse_s = m_s + log2 l_s (base 2, scores pre-scaled
// by log2 e; -inf when the split saw no key of that row).  The merge is
//   lse = log2 sum_s 2^(lse_s),  O = sum_s 2^(lse_s - lse) O_s,
// written as bf16 O (round to nearest even) and natural-log LSE (lse * ln 2).
//
// Work layout.  The unit of work is one 8-element chunk of one (window row,
// query head) pair: chunk u of a (KV head, request) block of partials, in the
// partials' own chunk-major order (partial_chunk), so consecutive units are
// consecutive 16-byte chunks.  A thread owns one unit and the splits g, g + SG,
// g + 2 SG, ... of it, where SG (split groups) is chosen at launch so that a
// thread has at most kBatch splits: all its loads (LSE and partial chunks) are
// issued at once, one memory round trip, and folded with a running maximum
// (online LSE combination).  A 256-thread CTA covers 256 / SG consecutive
// units of one block (consecutive threads, consecutive chunks: coalesced), and
// its SG groups are combined once through shared memory.  Requests with a
// single split were finished by the split kernel and are skipped, except in
// W-invariant mode, where every request is merged and SG is the largest the
// CTA allows for D, a constant.  Split s (counted from key 0, also when a
// sliding window lets the request's splits start later) then always lands in
// group s mod SG, each group folds its splits in ascending order and the
// groups are combined in group order, so the sum order of a (row, head) pair
// never depends on the split count: a row that sees fewer keys than its
// request's last row only has splits with lse = -inf, which every fold step
// skips.  The kernel may be launched as a programmatic dependent of the split
// kernel: it waits on griddepcontrol before touching partials, and it lets
// the next kernel in the stream launch early (that kernel waits for this
// grid's completion before reading its outputs).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace spec_attn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kBatch = 5;

template <int D>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_lse_kernel(const MergeParams p, const int sg) {
    constexpr int VEC = D / 8;                  // 8-element chunks per row
    __shared__ float4 part[kMergeThreads][2];
    __shared__ float part_m[kMergeThreads], part_l[kMergeThreads];
    const int tid = threadIdx.x;
    pdl_launch_dependents();
    const int upc = kMergeThreads / sg;         // units per CTA
    const int g = tid / upc, lu = tid % upc;
    const int kvh = blockIdx.y, r = blockIdx.z;
    const int G = p.group;

    ReqInfo ri;
    bool req_ok;
    int first = g;   // the first split of this thread's group
    if (p.window_left > 0 || p.w_invariant || p.dense_block) {
        req_ok = load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len, p.bt_capacity_keys,
                              p.keys_per_split, nullptr, ri, p.window_left, p.split_align, p.dense_block);
        // W-invariant mode: group g takes the splits whose index counted from
        // key 0 (split0 + s) is g mod SG, whatever the request's first split
        if (req_ok && p.w_invariant) first = ((g - ri.split0) % sg + sg) % sg;
    } else {
        req_ok = load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len, p.bt_capacity_keys,
                              p.keys_per_split, nullptr, ri);
    }
    // unit u of the request's (KV head) block: chunk c of row m (partial_chunk order)
    const int rows = req_ok ? ri.w * G : 0;
    const int u = blockIdx.x * upc + lu;
    const bool active = req_ok && u < rows * VEC && (ri.nsplits > 1 || p.w_invariant);
    const int c = active ? u / rows : 0, m = active ? u % rows : 0;
    // Wait for the split kernel's partials (no-op without a programmatic edge).
    pdl_wait_primary();

    float m_run = -INFINITY, l_run = 0.f;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    if (active) {
        const size_t split_stride = (size_t)p.total_rows * p.num_q_heads;
        const size_t blk0 = partial_pair(0, p.total_rows, p.num_q_heads, G, kvh, ri.row0, 0);
        const int n = ri.nsplits;
        for (int s0 = first; s0 < n; s0 += sg * kBatch) {
            float ls[kBatch], sc[kBatch];
            uint4 hv[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int s = s0 + k * sg;
                if (s < n) {
                    const float2 lsc = p.ws_ls[s * split_stride + blk0 + m];
                    ls[k] = lsc.x;
                    sc[k] = lsc.y;
                    hv[k] = *reinterpret_cast<const uint4*>(p.ws_o + (s * split_stride + blk0) * D + (size_t)u * 8);
                } else {
                    ls[k] = -INFINITY;
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (ls[k] == -INFINITY) continue;
                float4 o0, o1;
                {
                    const float2 a = unpack_half2(hv[k].x), b = unpack_half2(hv[k].y);
                    const float2 cc = unpack_half2(hv[k].z), d = unpack_half2(hv[k].w);
                    o0 = make_float4(a.x * sc[k], a.y * sc[k], b.x * sc[k], b.y * sc[k]);
                    o1 = make_float4(cc.x * sc[k], cc.y * sc[k], d.x * sc[k], d.y * sc[k]);
                }
                if (ls[k] > m_run) {
                    const float a = fast_exp2(m_run - ls[k]);   // 0 while m_run is -inf
                    a0.x *= a; a0.y *= a; a0.z *= a; a0.w *= a;
                    a1.x *= a; a1.y *= a; a1.z *= a; a1.w *= a;
                    l_run *= a;
                    m_run = ls[k];
                }
                const float w = fast_exp2(ls[k] - m_run);
                a0.x = fmaf(w, o0.x, a0.x); a0.y = fmaf(w, o0.y, a0.y);
                a0.z = fmaf(w, o0.z, a0.z); a0.w = fmaf(w, o0.w, a0.w);
                a1.x = fmaf(w, o1.x, a1.x); a1.y = fmaf(w, o1.y, a1.y);
                a1.z = fmaf(w, o1.z, a1.z); a1.w = fmaf(w, o1.w, a1.w);
                l_run += w;
            }
        }
    }
    part[tid][0] = a0;
    part[tid][1] = a1;
    part_m[tid] = m_run;
    part_l[tid] = l_run;
    __syncthreads();
    if (!active || g != 0) return;
    float mx = -INFINITY;
    for (int k = 0; k < sg; ++k) mx = fmaxf(mx, part_m[lu + k * upc]);
    float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0;
    float wsum = 0.f;
    for (int k = 0; k < sg; ++k) {
        const int j = lu + k * upc;
        if (part_m[j] == -INFINITY) continue;
        const float a = fast_exp2(part_m[j] - mx);
        const float4 q0 = part[j][0], q1 = part[j][1];
        t0.x = fmaf(a, q0.x, t0.x); t0.y = fmaf(a, q0.y, t0.y); t0.z = fmaf(a, q0.z, t0.z); t0.w = fmaf(a, q0.w, t0.w);
        t1.x = fmaf(a, q1.x, t1.x); t1.y = fmaf(a, q1.y, t1.y); t1.z = fmaf(a, q1.z, t1.z); t1.w = fmaf(a, q1.w, t1.w);
        wsum = fmaf(a, part_l[j], wsum);
    }
    const float inv = 1.f / wsum;
    uint4 out;
    out.x = float_to_bf16_bits(t0.x * inv) | ((uint32_t)float_to_bf16_bits(t0.y * inv) << 16);
    out.y = float_to_bf16_bits(t0.z * inv) | ((uint32_t)float_to_bf16_bits(t0.w * inv) << 16);
    out.z = float_to_bf16_bits(t1.x * inv) | ((uint32_t)float_to_bf16_bits(t1.y * inv) << 16);
    out.w = float_to_bf16_bits(t1.z * inv) | ((uint32_t)float_to_bf16_bits(t1.w * inv) << 16);
    const size_t oi = (size_t)(ri.row0 + m / G) * p.num_q_heads + kvh * G + m % G;
    *reinterpret_cast<uint4*>(p.o + oi * D + c * 8) = out;
    if (p.lse && c == 0) p.lse[oi] = (mx + log2f(wsum)) * kLn2;
}

}  // namespace

cudaError_t merge_launch(const MergeParams& p, cudaStream_t stream, bool programmatic) {
    const int vec = p.head_dim / 8;
    int sg = (p.max_splits + kBatch - 1) / kBatch;
    if (sg < 1) sg = 1;
    if (sg > kMergeThreads / vec) sg = kMergeThreads / vec;
    if (p.w_invariant) sg = kMergeThreads / vec;   // a constant of D: the fold order is fixed
    const int upc = kMergeThreads / sg;            // units per CTA
    const int chunks = p.max_w * p.group * vec;    // of the largest (KV head, request) block
    dim3 grid((chunks + upc - 1) / upc, p.num_kv_heads, p.num_reqs);
    dim3 block(kMergeThreads, 1, 1);
    void (*k)(const MergeParams, const int) = nullptr;
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
    return cudaLaunchKernelEx(&cfg, k, p, sg);
}

}  // namespace spec_attn
