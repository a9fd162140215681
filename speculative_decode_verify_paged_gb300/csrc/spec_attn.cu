// Host side of the C ABI (include/spec_attn.h): validation, the split-count
// heuristic, workspace layout and the kernel launches.
//
// The split heuristic restates the key-splitting idea of the page
// "ChunkedSmallT re-streams full KV per query chunk (DFlash K>=8 verify at
// long context)" (section "Finding": keys are split across CTAs and a reduce
// kernel merges the partials) without its width cap: every CTA holds all
// W x G query rows of one KV head, so the K/V of a window is swept once for
// any W <= 16, and an unsupported width is an explicit error rather than a
// silent truncation (page "perf(dflash): widen the verify window past the
// compact graph's four-row limit", section "What changed").
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/spec_attn.h"
#include "spec_attn_internal.h"

using namespace spec_attn;

struct spec_attn_plan {
    spec_attn_problem prob;
    int device;
    int num_sms;
    int variant;
    int keys_per_split;
    int max_splits;
    int row_groups;
    int rows_per_cta;
    CcConfig cc;
    dim3 grid;
    int threads;
    int smem;
    bool uses_merge;
    bool w_invariant;
    bool compact;               // tensor-core kernel in compact block order (one-dimensional grid)
    int split_align;
    int64_t kv_page_stride;     // bytes, resolved (dense when the problem gives 0)
    int64_t scale_page_stride;
    size_t ws_bytes;
    size_t ws_ls_off;
    size_t ws_o_off;
    float sm_scale;
    cudaEvent_t ev_begin;
    cudaEvent_t ev_end;
    // TMA descriptors of the last (Q, K pool, V pool) pointers a run used: a
    // decode loop re-running a plan on the same buffers encodes them once.
    std::mutex maps_mutex;
    TcMaps maps;
    const void* maps_key[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
};

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return SPEC_ATTN_E_CUDA;
}

constexpr size_t kStatusBytes = 256;
constexpr int kSplitUnit = 64;  // keys; a multiple of the page size and of every kernel's key tile

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t bytes_per_token_head(int kv_dtype, int d) {
    return kv_dtype == SPEC_ATTN_KV_BF16 ? static_cast<size_t>(2 * d) : static_cast<size_t>(d / 2 + d / 16);
}

// Rough cost (microseconds) of one call with `c` keys per split.  Terms:
//   waves of CTAs, each paying a fixed start/finish cost plus its keys at the
//   per-CTA streaming (or compute) rate; the whole job can not beat HBM; and
//   the merge reads every partial once more.  Waves count the CTAs with work
//   when the kernel runs in compact block order (those come first in launch
//   order); otherwise the whole grid (max splits x KV heads x requests x row
//   groups): it is laid out for the longest request, and a CTA of a shorter one
//   past its last split still takes an SM for its prologue before it leaves, so
//   blocks past the first wave start late even when the CTAs with work would
//   fit in one.
struct CostModel {
    double hbm_bytes_per_us = 6.5e6;   // ~6.5 TB/s
    double l2_bytes_per_us = 2.0e7;    // partials stay in L2
    double cta_fixed_us = 3.0;
    double merge_fixed_us = 2.0;
    double key_us = 0.0;               // one CTA's time per key (set per variant)
};

int choose_keys_per_split(const std::vector<int64_t>& lens, int64_t max_seq, int hkv, int row_groups,
                          int slots, double total_bytes, double partial_bytes_per_split,
                          const CostModel& cm, bool compact) {
    const int64_t max_units = std::max<int64_t>(1, (max_seq + kSplitUnit - 1) / kSplitUnit);
    double best = 1e300;
    int best_c = static_cast<int>(max_units * kSplitUnit);
    for (int64_t u = 1; u <= max_units; ++u) {
        const int64_t c = u * kSplitUnit;
        const int64_t splits = (max_seq + c - 1) / c;
        int64_t ctas = static_cast<int64_t>(lens.size()) * hkv * row_groups * splits;
        if (compact) {
            ctas = 0;
            for (int64_t L : lens) ctas += static_cast<int64_t>(hkv) * row_groups * ((L + c - 1) / c);
        }
        const int64_t waves = (ctas + slots - 1) / slots;
        const double t_cta = cm.cta_fixed_us + static_cast<double>(c) * cm.key_us;
        const double t_waves = static_cast<double>(waves) * t_cta;
        const double t_bw = total_bytes / cm.hbm_bytes_per_us;
        const double t_merge = splits > 1
            ? cm.merge_fixed_us + static_cast<double>(splits) * partial_bytes_per_split / cm.l2_bytes_per_us
            : 0.0;
        const double cost = std::max(t_waves, t_bw) + t_merge;
        if (cost < best * (1.0 - 1e-9)) {
            best = cost;
            best_c = static_cast<int>(c);
        }
    }
    return best_c;
}

int validate_problem(const spec_attn_problem* p, const int32_t* h_seq_lens, const int32_t* h_q_indptr) {
    if (!p) return SPEC_ATTN_E_INVALID_ARG;
    if (p->num_reqs < 0 || p->total_q_rows < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->head_dim <= 0 || p->page_size <= 0 || p->max_w < 1 || p->max_seq_len < 0 ||
        p->block_table_stride < 0 || p->num_pages < 0 || p->force_splits < 0)
        return SPEC_ATTN_E_INVALID_ARG;
    if (p->w_invariant != 0 && p->w_invariant != 1) return SPEC_ATTN_E_INVALID_ARG;
    if (p->dense_block_kv != 0 && p->dense_block_kv != 1) return SPEC_ATTN_E_INVALID_ARG;
    if (p->early_metadata != 0 && p->early_metadata != 1) return SPEC_ATTN_E_INVALID_ARG;
    if (p->early_context_kv != 0 && p->early_context_kv != 1) return SPEC_ATTN_E_INVALID_ARG;
    if (p->early_context_kv && !p->early_metadata) return SPEC_ATTN_E_INVALID_ARG;   // its tiles need the metadata
    if (p->test_stall != 0 && p->test_stall != 1) return SPEC_ATTN_E_INVALID_ARG;
    // the stall exercises the tensor-core kernel's bounded waits
    if (p->test_stall && p->kernel_variant != SPEC_ATTN_VARIANT_TCGEN05) return SPEC_ATTN_E_INVALID_ARG;
    if (p->dense_block_kv && p->w_invariant) return SPEC_ATTN_E_INVALID_ARG;   // exactness is a cache-only rule
    if (p->dense_block_kv && p->kv_dtype != SPEC_ATTN_KV_BF16) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->w_invariant && (p->fixed_keys_per_split < 0 || p->fixed_keys_per_split % 64 != 0))
        return SPEC_ATTN_E_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return SPEC_ATTN_E_INVALID_ARG;
    if (p->mask_mode != SPEC_ATTN_MASK_CAUSAL_IN_BLOCK && p->mask_mode != SPEC_ATTN_MASK_NON_CAUSAL)
        return SPEC_ATTN_E_INVALID_ARG;
    if (p->kv_dtype != SPEC_ATTN_KV_BF16 && p->kv_dtype != SPEC_ATTN_KV_NVFP4) return SPEC_ATTN_E_INVALID_ARG;
    if (p->kernel_variant < SPEC_ATTN_VARIANT_AUTO || p->kernel_variant > SPEC_ATTN_VARIANT_TCGEN05)
        return SPEC_ATTN_E_INVALID_ARG;
    if (!(p->sm_scale >= 0.f) || std::isinf(p->sm_scale)) return SPEC_ATTN_E_INVALID_ARG;
    // limits of the library: fail loudly, never truncate a window
    if (p->max_w > SPEC_ATTN_MAX_W) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->num_q_heads / p->num_kv_heads > SPEC_ATTN_MAX_GROUP) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->page_size != 16 && p->page_size != 32 && p->page_size != 64) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->window_left < 0 || (p->window_left > 0 && p->mask_mode != SPEC_ATTN_MASK_CAUSAL_IN_BLOCK))
        return SPEC_ATTN_E_INVALID_ARG;
    {
        const int64_t row = static_cast<int64_t>(bytes_per_token_head(p->kv_dtype, p->head_dim) -
                                                 (p->kv_dtype == SPEC_ATTN_KV_NVFP4 ? p->head_dim / 16 : 0));
        const int64_t dense = static_cast<int64_t>(p->num_kv_heads) * p->page_size * row;
        if (p->kv_page_stride != 0 && (p->kv_page_stride < dense || p->kv_page_stride % 16 != 0))
            return SPEC_ATTN_E_INVALID_ARG;
        const int64_t dense_sc = static_cast<int64_t>(p->num_kv_heads) * p->page_size * (p->head_dim / 16);
        if (p->kv_dtype == SPEC_ATTN_KV_NVFP4 && p->scale_page_stride != 0 &&
            (p->scale_page_stride < dense_sc || p->scale_page_stride % 16 != 0))
            return SPEC_ATTN_E_INVALID_ARG;
    }
    if (p->max_seq_len > INT32_MAX) return SPEC_ATTN_E_UNSUPPORTED;
    // key positions, and a block-table row's capacity in keys, are 32-bit on the device
    if (static_cast<int64_t>(p->block_table_stride) * p->page_size > INT32_MAX) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->num_kv_heads > 65535 || p->num_reqs > 65535) return SPEC_ATTN_E_UNSUPPORTED;
    if (p->num_reqs > 0) {
        if (p->max_seq_len < 1 || p->num_pages < 1) return SPEC_ATTN_E_INVALID_ARG;
        // the cache holds every key (with the dense block operand only the
        // context: checked per request below when the host lengths are given,
        // and on the device always)
        const int64_t need_pages = (p->max_seq_len + p->page_size - 1) / p->page_size;
        if (!p->dense_block_kv && p->block_table_stride < need_pages) return SPEC_ATTN_E_INVALID_ARG;
    }
    if (h_q_indptr) {
        if (h_q_indptr[0] != 0) return SPEC_ATTN_E_INVALID_ARG;
        for (int r = 0; r < p->num_reqs; ++r) {
            const int w = h_q_indptr[r + 1] - h_q_indptr[r];
            if (w < 0) return SPEC_ATTN_E_INVALID_ARG;
            if (w > SPEC_ATTN_MAX_W) return SPEC_ATTN_E_UNSUPPORTED;
            if (w > p->max_w) return SPEC_ATTN_E_INVALID_ARG;
        }
        if (h_q_indptr[p->num_reqs] > p->total_q_rows) return SPEC_ATTN_E_INVALID_ARG;
    }
    if (h_seq_lens) {
        for (int r = 0; r < p->num_reqs; ++r) {
            if (h_seq_lens[r] < 0 || h_seq_lens[r] > p->max_seq_len) return SPEC_ATTN_E_INVALID_ARG;
            if (h_q_indptr && h_seq_lens[r] < h_q_indptr[r + 1] - h_q_indptr[r]) return SPEC_ATTN_E_INVALID_ARG;
            if (h_q_indptr && p->dense_block_kv &&
                h_seq_lens[r] - (h_q_indptr[r + 1] - h_q_indptr[r]) >
                    static_cast<int64_t>(p->block_table_stride) * p->page_size)
                return SPEC_ATTN_E_INVALID_ARG;
        }
    }
    return SPEC_ATTN_OK;
}

}  // namespace

extern "C" {

int spec_attn_version(void) { return 100; }

int spec_attn_last_cuda_error(void) { return g_last_cuda_error; }

const char* spec_attn_status_string(int status) {
    switch (status) {
        case SPEC_ATTN_OK: return "ok";
        case SPEC_ATTN_E_INVALID_ARG: return "invalid argument";
        case SPEC_ATTN_E_UNSUPPORTED: return "unsupported by the library (W > 16, head_dim not in {64,128,256}, page_size not in {16,32,64}, group > 16, ...)";
        case SPEC_ATTN_E_WORKSPACE_TOO_SMALL: return "workspace too small";
        case SPEC_ATTN_E_CUDA: return "CUDA runtime error";
        case SPEC_ATTN_E_DEVICE_CHECK: return "a device-side check tripped";
        default: return "unknown status";
    }
}

int spec_attn_plan_create(const spec_attn_problem* problem, const int32_t* h_seq_lens,
                          const int32_t* h_q_indptr, spec_attn_plan** out, size_t* workspace_bytes) {
    if (!out) return SPEC_ATTN_E_INVALID_ARG;
    *out = nullptr;
    int st = validate_problem(problem, h_seq_lens, h_q_indptr);
    if (st != SPEC_ATTN_OK) return st;
    const spec_attn_problem& p = *problem;

    spec_attn_plan* plan = new (std::nothrow) spec_attn_plan();
    if (!plan) return SPEC_ATTN_E_INVALID_ARG;
    plan->prob = p;
    plan->sm_scale = p.sm_scale > 0.f ? p.sm_scale : 1.0f / std::sqrt(static_cast<float>(p.head_dim));
    plan->ev_begin = nullptr;
    plan->ev_end = nullptr;

    cudaError_t e = cudaGetDevice(&plan->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, plan->device);
    if (e != cudaSuccess) {
        delete plan;
        return cuda_fail(e);
    }

    const int G = p.num_q_heads / p.num_kv_heads;
    const int max_rows = p.max_w * G;
    const bool tc_ok = tc_supported(p.head_dim, p.kv_dtype, max_rows);
    // W-invariant mode needs one kernel for every width: the tensor-core one
    if ((p.kernel_variant == SPEC_ATTN_VARIANT_TCGEN05 || p.w_invariant) && !tc_ok) {
        delete plan;
        return SPEC_ATTN_E_UNSUPPORTED;
    }
    if (p.w_invariant && p.kernel_variant == SPEC_ATTN_VARIANT_CUDA_CORE) {
        delete plan;
        return SPEC_ATTN_E_UNSUPPORTED;
    }
    plan->w_invariant = p.w_invariant != 0;
    // AUTO takes the tensor-core kernel wherever it applies (every supported
    // head_dim and KV dtype; windows of more than 128 rows per KV head in row groups).
    const bool use_tc = p.kernel_variant == SPEC_ATTN_VARIANT_TCGEN05 ||
                        (p.kernel_variant == SPEC_ATTN_VARIANT_AUTO && tc_ok);
    if (use_tc) {
        plan->variant = SPEC_ATTN_VARIANT_TCGEN05;
        const int wg = tc_window_rows_per_cta(p.max_w, G);
        plan->rows_per_cta = wg * G;
        plan->row_groups = (p.max_w + wg - 1) / wg;
        plan->threads = tc_threads(p.kv_dtype);
        plan->smem = tc_smem_bytes(p.head_dim, p.kv_dtype);
        e = tc_prepare(p.head_dim, p.kv_dtype);
    } else {
        plan->variant = SPEC_ATTN_VARIANT_CUDA_CORE;
        plan->cc = cc_config(p.head_dim, p.kv_dtype, max_rows);
        plan->rows_per_cta = 8 * plan->cc.rows_per_warp;
        plan->row_groups = (max_rows + plan->rows_per_cta - 1) / plan->rows_per_cta;
        plan->threads = plan->cc.threads;
        plan->smem = plan->cc.smem_bytes;
        e = cc_prepare(p.head_dim, p.kv_dtype, plan->cc);
    }
    if (e != cudaSuccess) {
        delete plan;
        return cuda_fail(e);
    }

    {
        const int64_t row = static_cast<int64_t>(p.kv_dtype == SPEC_ATTN_KV_NVFP4 ? p.head_dim / 2 : 2 * p.head_dim);
        plan->kv_page_stride = p.kv_page_stride ? p.kv_page_stride
                                                : static_cast<int64_t>(p.num_kv_heads) * p.page_size * row;
        plan->scale_page_stride = p.scale_page_stride
                                      ? p.scale_page_stride
                                      : static_cast<int64_t>(p.num_kv_heads) * p.page_size * (p.head_dim / 16);
    }

    // ---- split heuristic ----
    // With a sliding window a request's splits cover only [key_base, len),
    // key_base = its first visible key rounded down to split_align (the key
    // tile, or the fixed split length in W-invariant mode); the lengths the
    // heuristic weighs are those spans.
    // W-invariant default: about max_seq_len / 32 keys per split (a multiple of
    // 64, at least 512), so that one request of the longest length fills the
    // GPU with its KV heads' splits (512 at 16K keys, 2048 at 64K)
    const int fixed_kps =
        p.fixed_keys_per_split > 0
            ? p.fixed_keys_per_split
            : static_cast<int>(std::max<int64_t>(512, (p.max_seq_len + 2047) / 2048 * 64));
    plan->split_align = plan->w_invariant ? fixed_kps : kSplitUnit;
    // (dense block operand: the splits cover the cached context; the window's
    // own keys ride along in the last one)
    auto span = [&](int64_t len, int64_t w) {
        const int64_t cached = p.dense_block_kv ? len - w : len;
        if (p.window_left <= 0) return cached;
        const int64_t lo0 = std::max<int64_t>(0, len - w - p.window_left + 1);
        return cached - lo0 / plan->split_align * plan->split_align;
    };
    std::vector<int64_t> lens;
    lens.reserve(static_cast<size_t>(p.num_reqs));
    // without host lengths: the longest span any request can have
    const int64_t span_bound =
        p.window_left > 0
            ? std::min<int64_t>(p.max_seq_len, static_cast<int64_t>(p.max_w) + p.window_left - 1 + plan->split_align - 1)
            : p.max_seq_len;
    for (int r = 0; r < p.num_reqs; ++r) {
        int64_t L = span_bound;
        if (h_seq_lens && h_q_indptr) L = span(h_seq_lens[r], h_q_indptr[r + 1] - h_q_indptr[r]);
        else if (h_seq_lens) L = std::min<int64_t>(h_seq_lens[r], span_bound);
        if (h_q_indptr && h_q_indptr[r + 1] == h_q_indptr[r]) L = 0;  // empty window: no CTAs do work
        lens.push_back(L);
    }
    const int64_t max_seq = std::max<int64_t>(1, span_bound);
    // Compact block order (tensor-core kernel, 2 to 64 requests): the CTAs
    // with work come first in launch order.  It costs the CTAs one more round
    // trip for metadata, so it is used only where the (splits x KV heads x
    // requests) grid would hold idle slots: lengths unknown, or uneven spans or
    // windows.
    plan->compact = false;
    if (use_tc && p.num_reqs >= 2 && p.num_reqs <= 64) {
        plan->compact = !(h_seq_lens && h_q_indptr);
        for (int r = 1; r < p.num_reqs && !plan->compact; ++r)
            plan->compact = lens[r] != lens[0] ||
                            (h_q_indptr[r + 1] - h_q_indptr[r]) != (h_q_indptr[1] - h_q_indptr[0]);
    }
    const size_t bkh = bytes_per_token_head(p.kv_dtype, p.head_dim);
    double total_bytes = 0;
    for (int64_t L : lens) total_bytes += static_cast<double>(L) * p.num_kv_heads * 2.0 * bkh;
    int occ = 1;
    {
        // CTAs the split kernel fits per SM (smem bound for the CUDA-core variant)
        int max_smem = 0;
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, plan->device);
        occ = std::max(1, std::min(max_smem / std::max(1, plan->smem + 1024), 2048 / plan->threads));
    }
    CostModel cm;
    if (use_tc) {
        // tensor cores keep up with HBM: a CTA streams its keys at roughly
        // its SM's share of HBM bandwidth (one CTA per SM).
        occ = 1;
        cm.key_us = 2.0 * bkh / (6.5e6 / plan->num_sms);
    } else {
        // CUDA cores: ~2 FMA per element per row (QK and PV) at ~128 FMA/clk/SM,
        // ~1.9 GHz, shared by `occ` CTAs, times an instruction-overhead factor.
        const double fma_per_us = 128.0 * 1.9e3 / occ;
        const double rows = std::min(max_rows, plan->rows_per_cta);
        const double t_compute = rows * 2.0 * p.head_dim * 2.0 / fma_per_us;
        const double t_stream = 2.0 * bkh / (6.5e6 / (plan->num_sms * occ));
        cm.key_us = std::max(t_compute, t_stream);
    }
    // per split: fp16 partial rows + (lse, scale), written once and read once
    const double partial_bytes = static_cast<double>(p.total_q_rows) * p.num_q_heads * (p.head_dim * 2.0 + 8.0) * 2.0;
    if (plan->w_invariant) {
        // split boundaries fixed by key position alone (never by W, P or lengths)
        plan->keys_per_split = fixed_kps;
    } else if (p.force_splits > 0) {
        int64_t c = (max_seq + p.force_splits - 1) / p.force_splits;
        c = (c + kSplitUnit - 1) / kSplitUnit * kSplitUnit;
        plan->keys_per_split = static_cast<int>(std::max<int64_t>(c, kSplitUnit));
    } else {
        plan->keys_per_split = choose_keys_per_split(lens, max_seq, p.num_kv_heads, plan->row_groups,
                                                     plan->num_sms * occ, total_bytes, partial_bytes, cm,
                                                     plan->compact);
    }
    plan->max_splits = static_cast<int>((max_seq + plan->keys_per_split - 1) / plan->keys_per_split);
    plan->uses_merge = plan->max_splits > 1 || plan->w_invariant;

    if (plan->compact && static_cast<int64_t>(plan->max_splits) * plan->row_groups * p.num_kv_heads *
                                 p.num_reqs > INT32_MAX)
        plan->compact = false;   // the one-dimensional grid would not fit
    if (plan->compact)
        plan->grid = dim3(static_cast<unsigned>(static_cast<int64_t>(plan->max_splits) * plan->row_groups *
                                                p.num_kv_heads * p.num_reqs));
    else
        plan->grid = dim3(static_cast<unsigned>(plan->max_splits * plan->row_groups),
                          static_cast<unsigned>(p.num_kv_heads), static_cast<unsigned>(std::max(1, p.num_reqs)));

    // ---- workspace layout: [status region][(lse, scale) partials][fp16 O partials] ----
    size_t ws = kStatusBytes;
    plan->ws_ls_off = ws;
    if (plan->uses_merge) {
        const size_t pairs = static_cast<size_t>(p.total_q_rows) * p.num_q_heads;
        ws = align_up(ws + static_cast<size_t>(plan->max_splits) * pairs * 2 * sizeof(float), 256);
        plan->ws_o_off = ws;
        ws += static_cast<size_t>(plan->max_splits) * pairs * p.head_dim * sizeof(uint16_t);
    } else {
        plan->ws_o_off = kStatusBytes;
    }
    plan->ws_bytes = align_up(ws, 256);
    if (workspace_bytes) *workspace_bytes = plan->ws_bytes;
    *out = plan;
    return SPEC_ATTN_OK;
}

int spec_attn_plan_destroy(spec_attn_plan* plan) {
    delete plan;
    return SPEC_ATTN_OK;
}

int spec_attn_plan_get_info(const spec_attn_plan* plan, spec_attn_plan_info* info) {
    if (!plan || !info) return SPEC_ATTN_E_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    info->kernel_variant = plan->variant;
    info->keys_per_split = plan->keys_per_split;
    info->max_splits = plan->max_splits;
    info->row_groups = plan->row_groups;
    info->grid_x = static_cast<int32_t>(plan->grid.x);
    info->grid_y = static_cast<int32_t>(plan->grid.y);
    info->grid_z = static_cast<int32_t>(plan->grid.z);
    info->block_threads = plan->threads;
    info->smem_bytes = plan->smem;
    info->uses_merge = plan->uses_merge ? 1 : 0;
    info->num_sms = plan->num_sms;
    info->workspace_bytes = plan->ws_bytes;
    return SPEC_ATTN_OK;
}

int spec_attn_plan_set_timing_events(spec_attn_plan* plan, void* split_begin, void* split_end) {
    if (!plan) return SPEC_ATTN_E_INVALID_ARG;
    if ((split_begin == nullptr) != (split_end == nullptr)) return SPEC_ATTN_E_INVALID_ARG;
    plan->ev_begin = static_cast<cudaEvent_t>(split_begin);
    plan->ev_end = static_cast<cudaEvent_t>(split_end);
    return SPEC_ATTN_OK;
}

// Host-side checks shared by every entry point that reads or writes the cache:
// the pools, their scales (NVFP4), the request arrays, the workspace and the
// current device.  min_ws is the workspace the entry point needs.
static int check_cache_args(const spec_attn_plan* plan, const void* k_pool, const void* v_pool,
                            const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                            const void* workspace, size_t workspace_bytes, size_t min_ws) {
    const spec_attn_problem& p = plan->prob;
    if (!k_pool || !v_pool || !block_table || !seq_lens || !q_indptr || !workspace) return SPEC_ATTN_E_INVALID_ARG;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        !aligned(q_indptr, 4) || !aligned(workspace, 256))
        return SPEC_ATTN_E_INVALID_ARG;
    if (p.kv_dtype == SPEC_ATTN_KV_NVFP4) {
        if (!k_scales || !v_scales || !aligned(k_scales, 16) || !aligned(v_scales, 16))
            return SPEC_ATTN_E_INVALID_ARG;
        if (!(k_gscale > 0.f) || !(v_gscale > 0.f) || std::isinf(k_gscale) || std::isinf(v_gscale))
            return SPEC_ATTN_E_INVALID_ARG;
    }
    if (workspace_bytes < min_ws) return SPEC_ATTN_E_WORKSPACE_TOO_SMALL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev != plan->device) return SPEC_ATTN_E_INVALID_ARG;
    return SPEC_ATTN_OK;
}

static int check_run_args(const spec_attn_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                          const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                          const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                          const void* o, const float* lse, const int64_t* trace, const void* workspace,
                          size_t workspace_bytes) {
    if (!q || !o || !aligned(q, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
        (trace && !aligned(trace, 8)))
        return SPEC_ATTN_E_INVALID_ARG;
    return check_cache_args(plan, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                            q_indptr, workspace, workspace_bytes, plan->ws_bytes);
}

static int check_append_args(const spec_attn_plan* plan, const void* k_new, const void* v_new,
                             const void* k_pool, const void* v_pool, const void* k_scales, const void* v_scales,
                             float k_gscale, float v_gscale, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* q_indptr, const void* workspace,
                             size_t workspace_bytes) {
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return SPEC_ATTN_E_INVALID_ARG;
    return check_cache_args(plan, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                            q_indptr, workspace, workspace_bytes, kStatusBytes);
}

static int append_launch_checked(const spec_attn_plan* plan, const void* k_new, const void* v_new, void* k_pool,
                                 void* v_pool, void* k_scales, void* v_scales, float k_gscale, float v_gscale,
                                 const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                                 void* workspace, cudaStream_t stream) {
    const spec_attn_problem& p = plan->prob;
    AppendParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.k_new = static_cast<const uint16_t*>(k_new);
    ap.v_new = static_cast<const uint16_t*>(v_new);
    ap.k_pool = k_pool;
    ap.v_pool = v_pool;
    ap.k_scales = static_cast<uint8_t*>(k_scales);
    ap.v_scales = static_cast<uint8_t*>(v_scales);
    ap.k_gscale = k_gscale;
    ap.v_gscale = v_gscale;
    ap.block_table = block_table;
    ap.seq_lens = seq_lens;
    ap.q_indptr = q_indptr;
    ap.status = static_cast<unsigned int*>(workspace);
    ap.num_reqs = p.num_reqs;
    ap.total_rows = p.total_q_rows;
    ap.max_w = p.max_w;
    ap.num_kv_heads = p.num_kv_heads;
    ap.head_dim = p.head_dim;
    ap.num_pages = p.num_pages;
    ap.bt_stride = p.block_table_stride;
    ap.bt_capacity_keys = p.block_table_stride * p.page_size;
    ap.max_seq_len = p.max_seq_len;
    ap.page_size = p.page_size;
    ap.kv_page_stride = plan->kv_page_stride;
    ap.scale_page_stride = plan->scale_page_stride;
    const cudaError_t e = append_launch(ap, p.kv_dtype, stream);
    return e == cudaSuccess ? SPEC_ATTN_OK : cuda_fail(e);
}

static int run_impl(const spec_attn_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                    const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                    void* o, float* lse, int64_t* trace, void* workspace, size_t workspace_bytes,
                    spec_attn_stream_t stream_handle, const void* block_k = nullptr,
                    const void* block_v = nullptr, bool clear_status = false) {
    if (!plan) return SPEC_ATTN_E_INVALID_ARG;
    const spec_attn_problem& p = plan->prob;
    // a dense-block plan runs only with its block tensors, and they need such a plan
    if ((p.dense_block_kv != 0) != (block_k != nullptr) || (block_k == nullptr) != (block_v == nullptr))
        return SPEC_ATTN_E_INVALID_ARG;
    if (block_k && (!aligned(block_k, 16) || !aligned(block_v, 16))) return SPEC_ATTN_E_INVALID_ARG;
    if (p.num_reqs == 0 || p.total_q_rows == 0) return SPEC_ATTN_OK;
    const int chk = check_run_args(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table,
                                   seq_lens, q_indptr, o, lse, trace, workspace, workspace_bytes);
    if (chk != SPEC_ATTN_OK) return chk;
    cudaError_t e = cudaSuccess;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    if (clear_status) {
        // only once every host check has passed: a rejected call writes nothing
        e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    SplitParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.q = static_cast<const uint16_t*>(q);
    sp.k_pool = k_pool;
    sp.v_pool = v_pool;
    sp.k_scales = static_cast<const uint8_t*>(k_scales);
    sp.v_scales = static_cast<const uint8_t*>(v_scales);
    sp.block_table = block_table;
    sp.seq_lens = seq_lens;
    sp.q_indptr = q_indptr;
    sp.o = static_cast<uint16_t*>(o);
    sp.lse = lse;
    sp.trace = reinterpret_cast<long long*>(trace);
    sp.status = reinterpret_cast<unsigned int*>(ws);
    sp.always_partials = plan->w_invariant ? 1 : 0;
    sp.ws_ls = reinterpret_cast<float2*>(ws + plan->ws_ls_off);
    sp.ws_o = reinterpret_cast<uint16_t*>(ws + plan->ws_o_off);
    sp.num_reqs = p.num_reqs;
    sp.total_rows = p.total_q_rows;
    sp.max_w = p.max_w;
    sp.num_q_heads = p.num_q_heads;
    sp.num_kv_heads = p.num_kv_heads;
    sp.group = p.num_q_heads / p.num_kv_heads;
    sp.head_dim = p.head_dim;
    sp.page_size = p.page_size;
    sp.num_pages = p.num_pages;
    sp.bt_stride = p.block_table_stride;
    sp.mask_mode = p.mask_mode;
    sp.keys_per_split = plan->keys_per_split;
    sp.max_splits = plan->max_splits;
    sp.row_groups = plan->row_groups;
    sp.rows_per_cta = plan->rows_per_cta;
    sp.window_rows_per_cta = plan->rows_per_cta / sp.group;
    sp.max_seq_len = p.max_seq_len;
    const float log2e = 1.4426950408889634f;
    const bool fp4 = p.kv_dtype == SPEC_ATTN_KV_NVFP4;
    sp.score_scale_log2 = plan->sm_scale * log2e * (fp4 ? k_gscale : 1.0f);
    sp.out_scale = fp4 ? v_gscale : 1.0f;
    sp.page_shift = p.page_size == 64 ? 2 : p.page_size == 32 ? 1 : 0;
    sp.kv_page_stride = plan->kv_page_stride;
    sp.scale_page_stride = plan->scale_page_stride;
    sp.window_left = p.window_left;
    sp.split_align = plan->split_align;
    sp.dense_block = p.dense_block_kv;
    sp.compact = plan->compact ? 1 : 0;
    sp.early_metadata = p.early_metadata;
    sp.early_context_kv = p.early_context_kv;
    sp.test_stall = p.test_stall;
    sp.block_k = static_cast<const uint16_t*>(block_k);
    sp.block_v = static_cast<const uint16_t*>(block_v);

    MergeParams mprm;
    std::memset(&mprm, 0, sizeof(mprm));
    mprm.seq_lens = seq_lens;
    mprm.q_indptr = q_indptr;
    mprm.ws_o = sp.ws_o;
    mprm.ws_ls = sp.ws_ls;
    mprm.o = sp.o;
    mprm.lse = lse;
    mprm.num_reqs = p.num_reqs;
    mprm.total_rows = p.total_q_rows;
    mprm.max_w = p.max_w;
    mprm.num_q_heads = p.num_q_heads;
    mprm.num_kv_heads = p.num_kv_heads;
    mprm.group = p.num_q_heads / p.num_kv_heads;
    mprm.head_dim = p.head_dim;
    mprm.keys_per_split = plan->keys_per_split;
    mprm.max_splits = plan->max_splits;
    mprm.max_seq_len = p.max_seq_len;
    mprm.bt_capacity_keys = p.block_table_stride * p.page_size;
    mprm.w_invariant = plan->w_invariant ? 1 : 0;
    mprm.window_left = p.window_left;
    mprm.split_align = plan->split_align;
    mprm.dense_block = p.dense_block_kv;

    spec_attn_plan* mp = const_cast<spec_attn_plan*>(plan);
    std::unique_lock<std::mutex> maps_lock(mp->maps_mutex, std::defer_lock);
    if (plan->variant == SPEC_ATTN_VARIANT_TCGEN05) {
        maps_lock.lock();
        // (dense block operand: the block tensors take the scale pools' places)
        const void* key3 = p.dense_block_kv ? block_k : k_scales;
        const void* key4 = p.dense_block_kv ? block_v : v_scales;
        if (mp->maps_key[0] != q || mp->maps_key[1] != k_pool || mp->maps_key[2] != v_pool ||
            mp->maps_key[3] != key3 || mp->maps_key[4] != key4) {
            if (!tc_encode_maps(sp, p.kv_dtype, &mp->maps)) {
                for (auto& k : mp->maps_key) k = nullptr;
                return SPEC_ATTN_E_INVALID_ARG;
            }
            mp->maps_key[0] = q;
            mp->maps_key[1] = k_pool;
            mp->maps_key[2] = v_pool;
            mp->maps_key[3] = key3;
            mp->maps_key[4] = key4;
        }
    }
    if (plan->ev_begin) {
        e = cudaEventRecord(plan->ev_begin, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (plan->variant == SPEC_ATTN_VARIANT_TCGEN05) {
        e = tc_launch(sp, p.kv_dtype, mp->maps, trace != nullptr, plan->grid, stream, plan->ev_begin == nullptr);
        maps_lock.unlock();
    } else
        e = cc_launch(sp, p.kv_dtype, plan->cc, trace != nullptr, plan->grid, stream, plan->ev_begin == nullptr);
    if (e != cudaSuccess) return cuda_fail(e);
    if (plan->ev_end) {
        e = cudaEventRecord(plan->ev_end, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (plan->uses_merge) {
        // programmatic launch lets the merge's CTAs become resident while the
        // split kernel drains; it is skipped when a timing event sits between.
        e = merge_launch(mprm, stream, plan->ev_end == nullptr);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return SPEC_ATTN_OK;
}

}  // extern "C"

namespace spec_attn {
int run_clearing_status(const spec_attn_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                        const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return run_impl(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                    q_indptr, o, lse, nullptr, workspace, workspace_bytes, stream, nullptr, nullptr, true);
}
}  // namespace spec_attn

extern "C" {

int spec_attn_run(const spec_attn_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                  const void* k_scales, const void* v_scales, float k_gscale, float v_gscale,
                  const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                  void* o, float* lse, void* workspace, size_t workspace_bytes,
                  spec_attn_stream_t stream) {
    return run_impl(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table,
                    seq_lens, q_indptr, o, lse, nullptr, workspace, workspace_bytes, stream);
}

int spec_attn_run_dense_block(const spec_attn_plan* plan, const void* q, const void* block_k,
                              const void* block_v, const void* k_pool, const void* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                              void* o, float* lse, int64_t* trace, void* workspace, size_t workspace_bytes,
                              spec_attn_stream_t stream) {
    if (!plan || !plan->prob.dense_block_kv || !block_k || !block_v) return SPEC_ATTN_E_INVALID_ARG;
    return run_impl(plan, q, k_pool, v_pool, nullptr, nullptr, 1.0f, 1.0f, block_table, seq_lens, q_indptr, o,
                    lse, trace, workspace, workspace_bytes, stream, block_k, block_v);
}

int spec_attn_append_kv(const spec_attn_plan* plan, const void* k_new, const void* v_new, void* k_pool,
                        void* v_pool, void* k_scales, void* v_scales, float k_gscale, float v_gscale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                        void* workspace, size_t workspace_bytes, spec_attn_stream_t stream) {
    // (a dense-block plan keeps the window's keys out of the cache: nothing to append)
    if (!plan || plan->prob.dense_block_kv) return SPEC_ATTN_E_INVALID_ARG;
    const spec_attn_problem& p = plan->prob;
    if (p.num_reqs == 0 || p.total_q_rows == 0) return SPEC_ATTN_OK;
    const int chk = check_append_args(plan, k_new, v_new, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                      block_table, seq_lens, q_indptr, workspace, workspace_bytes);
    if (chk != SPEC_ATTN_OK) return chk;
    return append_launch_checked(plan, k_new, v_new, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                 block_table, seq_lens, q_indptr, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int spec_attn_run_append(const spec_attn_plan* plan, const void* q, const void* k_new, const void* v_new,
                         void* k_pool, void* v_pool, void* k_scales, void* v_scales, float k_gscale,
                         float v_gscale, const int32_t* block_table, const int32_t* seq_lens,
                         const int32_t* q_indptr, void* o, float* lse, void* workspace, size_t workspace_bytes,
                         spec_attn_stream_t stream) {
    if (!plan || plan->prob.dense_block_kv) return SPEC_ATTN_E_INVALID_ARG;
    const spec_attn_problem& p = plan->prob;
    if (p.num_reqs == 0 || p.total_q_rows == 0) return SPEC_ATTN_OK;
    // every check before the first launch: a rejected call changes nothing
    int chk = check_append_args(plan, k_new, v_new, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                block_table, seq_lens, q_indptr, workspace, workspace_bytes);
    if (chk == SPEC_ATTN_OK)
        chk = check_run_args(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                             q_indptr, o, lse, nullptr, workspace, workspace_bytes);
    if (chk != SPEC_ATTN_OK) return chk;
    chk = append_launch_checked(plan, k_new, v_new, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                block_table, seq_lens, q_indptr, workspace, reinterpret_cast<cudaStream_t>(stream));
    if (chk != SPEC_ATTN_OK) return chk;
    return run_impl(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                    q_indptr, o, lse, nullptr, workspace, workspace_bytes, stream);
}

int spec_attn_run_traced(const spec_attn_plan* plan, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scales, const void* v_scales,
                         float k_gscale, float v_gscale, const int32_t* block_table,
                         const int32_t* seq_lens, const int32_t* q_indptr, void* o, float* lse,
                         int64_t* trace, void* workspace, size_t workspace_bytes,
                         spec_attn_stream_t stream) {
    if (!trace) return SPEC_ATTN_E_INVALID_ARG;
    return run_impl(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table,
                    seq_lens, q_indptr, o, lse, trace, workspace, workspace_bytes, stream);
}

int spec_attn_reset_device_status(void* workspace, spec_attn_stream_t stream) {
    if (!workspace) return SPEC_ATTN_E_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, kStatusBytes, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_ATTN_OK : cuda_fail(e);
}

int spec_attn_check_device_status(void* workspace, spec_attn_stream_t stream_handle, uint32_t* bits) {
    if (!workspace) return SPEC_ATTN_E_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(v), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (bits) *bits = v;
    return v ? SPEC_ATTN_E_DEVICE_CHECK : SPEC_ATTN_OK;
}

}  // extern "C"
