// Internal interface between the host library (plan / run) and the kernels.
// Not installed; the public ABI is include/spec_attn.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct spec_attn_plan;   // the public ABI's opaque plan (spec_attn.cu)

namespace spec_attn {

// Everything the LSE merge of split partials needs (merge_lse.cu).
struct MergeParams {
    const int32_t* seq_lens;
    const int32_t* q_indptr;
    const uint16_t* ws_o;
    const float2* ws_ls;
    uint16_t* o;
    float* lse;
    int num_reqs;
    int total_rows;
    int max_w;
    int num_q_heads;
    int num_kv_heads;
    int group;                  // Hq / Hkv
    int head_dim;
    int keys_per_split;
    int max_splits;
    long long max_seq_len;
    int bt_capacity_keys;       // bt_stride * page_size
    int w_invariant;            // merge every request (one split too), splits folded in order
    int window_left;            // as SplitParams
    int split_align;
    int dense_block;
};

// Everything one split-KV launch needs.  Plain pointers and ints only.
struct SplitParams {
    const uint16_t* q;          // [total_rows, Hq, d] bf16 bits
    const void* k_pool;         // bf16 [pages, Hkv, ps, d] | nvfp4 codes [pages, Hkv, ps, d/2]
    const void* v_pool;
    const uint8_t* k_scales;    // nvfp4 e4m3 [pages, Hkv, ps, d/16]
    const uint8_t* v_scales;
    const int32_t* block_table; // [P, bt_stride]
    const int32_t* seq_lens;    // [P]
    const int32_t* q_indptr;    // [P + 1]
    uint16_t* o;                // [total_rows, Hq, d] bf16 bits
    float* lse;                 // [total_rows, Hq] or nullptr
    long long* trace;           // [total_rows, Hq, 2] or nullptr
    uint16_t* ws_o;             // split partials: per (row, head) pair, d fp16 values of O_s / scale_s
    float2* ws_ls;              // per pair: (lse_s in log2 units, scale_s = max |O_s|), same order
    unsigned int* status;       // sticky device-status word
    int always_partials;        // W-invariant mode: write split partials even for one split
    int num_reqs;
    int total_rows;
    int max_w;
    int num_q_heads;
    int num_kv_heads;
    int group;                  // Hq / Hkv
    int head_dim;
    int page_size;
    int num_pages;
    int bt_stride;
    int mask_mode;
    int keys_per_split;         // multiple of 64
    int max_splits;
    int row_groups;             // CTAs per (request, KV head, split)
    int rows_per_cta;           // query rows per CTA (tensor-core kernel: whole window rows x G)
    int window_rows_per_cta;    // tensor-core kernel: window rows of one row group
    long long max_seq_len;
    float score_scale_log2;     // sm_scale * log2(e) [* k_gscale for NVFP4]
    float out_scale;            // 1, or v_gscale for NVFP4
    int page_shift;             // log2(page_size / 16): 16-key units per page = 1 << page_shift
    long long kv_page_stride;   // bytes between pages of a K or V pool
    long long scale_page_stride;// bytes between pages of a scale pool (NVFP4)
    int window_left;            // causal sliding window (keys), 0 = none
    int split_align;            // first split of a request starts at a multiple of this (keys)
    int early_metadata;         // lengths, windows and block table are not written by the previous kernel
    int early_context_kv;       // nor the cached keys below ctx_r: the first K/V tile may be read before the wait
    int test_stall;             // testing: the K (NVFP4: raw) producer issues nothing
    int dense_block;            // the window's keys come from block_k / block_v (bf16 caches)
    int compact;                // tensor-core kernel: one-dimensional grid, blocks in order of work units
                                // (request, split, KV head, row group) that exist; the rest idle
    const uint16_t* block_k;    // [total_rows, Hkv, d] bf16 bits, or nullptr
    const uint16_t* block_v;
};



// Everything one KV-append launch needs (append_kv.cu).
struct AppendParams {
    const uint16_t* k_new;      // [total_rows, Hkv, d] bf16 bits, rows in q_indptr order
    const uint16_t* v_new;
    void* k_pool;               // bf16 [pages, Hkv, ps, d] | nvfp4 codes [pages, Hkv, ps, d/2]
    void* v_pool;
    uint8_t* k_scales;          // nvfp4 e4m3 [pages, Hkv, ps, d/16]
    uint8_t* v_scales;
    float k_gscale;             // nvfp4 decode scales (> 0)
    float v_gscale;
    const int32_t* block_table; // [P, bt_stride]
    const int32_t* seq_lens;    // [P]
    const int32_t* q_indptr;    // [P + 1]
    unsigned int* status;       // sticky device-status word
    int num_reqs;
    int total_rows;
    int max_w;
    int num_kv_heads;
    int head_dim;
    int num_pages;
    int bt_stride;
    int bt_capacity_keys;       // bt_stride * page_size
    long long max_seq_len;
    int page_size;
    long long kv_page_stride;   // bytes between pages of a K or V pool
    long long scale_page_stride;// bytes between pages of a scale pool (NVFP4)
};

// Split partials.  A split leaves, per (window row, query head) pair, its
// normalised partial output O_s (d values), lse_s and scale_s = max_e |O_s[e]|;
// O_s is stored as d fp16 values of O_s / scale_s (in [-1, 1]), so a stored
// value is off by at most scale_s * 2^-12, and the partials take half the bytes
// of fp32 for the split kernel to write and the merge to read.
//
// Order of the (window row, query head) pairs in the split partials: split-major,
// then KV head, then window row, then the G query heads of that KV head.  The
// W_r x G pairs of one (split, KV head, request) form one contiguous block;
// the (lse, scale) pairs follow this order directly.
__host__ __device__ __forceinline__ size_t partial_pair(int split, int total_rows, int num_q_heads, int group,
                                                        int kvh, int row, int g) {
    return (size_t)split * total_rows * num_q_heads + ((size_t)kvh * total_rows + row) * group + g;
}

// The fp16 values of such a block (rows x d, rows = W_r x G, row m = window row
// x G + head) are stored chunk-major: element offset, from the block's start
// (partial_pair of its first pair, times d), of the 8-element chunk c of row m.
// Consecutive rows of one chunk are adjacent, so a warp holding 32 rows writes
// (and the merge reads) 512 contiguous bytes per chunk.
__host__ __device__ __forceinline__ size_t partial_chunk(int c, int rows, int m) {
    return ((size_t)c * rows + m) * 8;
}

// Device-status bits (mirror the public SPEC_ATTN_DEV_* values).
constexpr unsigned int kDevBadPage = 0x1u;
constexpr unsigned int kDevBadSeqLen = 0x2u;
constexpr unsigned int kDevBadWindow = 0x4u;
constexpr unsigned int kDevWaitTimeout = 0x8u;

// ---- CUDA-core split-KV kernel (split_attn_cc.cu) ----
struct CcConfig {
    int rows_per_warp;   // 1, 2 or 4
    int stages;          // pages in the cp.async ring
    int smem_bytes;
    int threads;
};
CcConfig cc_config(int head_dim, int kv_dtype, int max_rows);
// Prepare (max dynamic smem attribute) the instance a config uses; returns a CUDA error code.
cudaError_t cc_prepare(int head_dim, int kv_dtype, const CcConfig& cfg);
// programmatic: launch as a programmatic dependent of the previous kernel in the
// stream (the kernel waits on griddepcontrol before its first global access).
cudaError_t cc_launch(const SplitParams& p, int kv_dtype, const CcConfig& cfg, bool traced,
                      dim3 grid, cudaStream_t stream, bool programmatic);

// ---- tcgen05 split-KV kernel (split_attn_tc.cu) ----
// TMA descriptors of one (Q, K pool, V pool) triple; opaque CUtensorMap storage.
// bf16 KV: K and V pools, and (dense block operand) the block K and V tensors
// in the ks / vs slots; NVFP4: K and V code pools, plus their scale pools.
struct TcMaps {
    alignas(64) unsigned char q[128];
    alignas(64) unsigned char k[128];
    alignas(64) unsigned char v[128];
    alignas(64) unsigned char ks[128];
    alignas(64) unsigned char vs[128];
};
bool tc_supported(int head_dim, int kv_dtype, int max_rows);
// window rows one CTA of the tensor-core kernel holds (its row group): Wg x G <= 128
int tc_window_rows_per_cta(int max_w, int group);
int tc_smem_bytes(int head_dim, int kv_dtype);
int tc_threads(int kv_dtype);
cudaError_t tc_prepare(int head_dim, int kv_dtype);
bool tc_encode_maps(const SplitParams& p, int kv_dtype, TcMaps* maps);
cudaError_t tc_launch(const SplitParams& p, int kv_dtype, const TcMaps& maps, bool traced, dim3 grid,
                      cudaStream_t stream, bool programmatic);

// ---- LSE merge (merge_lse.cu) ----
cudaError_t merge_launch(const MergeParams& p, cudaStream_t stream, bool programmatic);

// ---- no-alloc entry point (spec_attn_noalloc.cu) ----
// spec_attn_run that, once every host check has passed, first zeroes the
// workspace's device-status word on `stream` (the built-in scratch is shared
// by every call, so each call starts from a clean word).
int run_clearing_status(const ::spec_attn_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                        const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

// ---- KV append (append_kv.cu) ----
// Always a programmatic dependent of the previous kernel in the stream (the
// kernel waits on griddepcontrol before its first global access).
cudaError_t append_launch(const AppendParams& p, int kv_dtype, cudaStream_t stream);

}  // namespace spec_attn
