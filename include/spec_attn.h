/*
 * spec_attn.h -- C ABI of a GB300 (sm_103a) library for the attention of
 * speculative-decoding windows against a paged KV cache.
 *
 * The operation.  A batch holds P requests.  Request r brings a window of
 * W_r = q_indptr[r+1] - q_indptr[r] query rows (0 <= W_r <= 16: the seed
 * token plus k proposed tokens) and owns seq_len[r] keys in a paged K/V cache
 * shared by all requests.  The window's own W_r keys are already in the
 * cache as its last W_r keys, so ctx_r = seq_len[r] - W_r keys precede it.
 * Every window row attends to its request's cache under one of two masks:
 *
 *   causal-in-block: window row i sees keys 0 .. ctx_r + i (inclusive)
 *   non-causal:      every window row sees all seq_len[r] keys
 *
 * optionally narrowed, for causal calls, by a sliding window: with
 * window_left = n > 0, row i sees only keys max(0, ctx_r + i - n + 1) ..
 * ctx_r + i.  (The first page below names an attention window that its
 * non-causal draft layers leave unapplied, without defining it; this is the
 * plainest reading, and non-causal calls take no window.)
 *
 * and outputs are produced for window rows only, never for context rows.
 * Sources (titles of the pages this library restates):
 *   - "DFlash2 leaves the paged graph fast path at every c>1 and re-attends
 *     the whole batch context every decode step", sections "The route
 *     change" (paged store, Tq = 1+k rows, graph-captured), "The cost" (no
 *     outputs for context rows; non-causal draft layers see their request's
 *     whole span) and "Scope" (one shared paged pool, a batched block table,
 *     per-request seq_lens, P x (1+k) query rows).
 *   - "ChunkedSmallT re-streams full KV per query chunk (DFlash K>=8 verify
 *     at long context)", sections "Finding" (key-splitting plus a reduce
 *     kernel; the K/V sweep must not repeat per query chunk) and
 *     "Measurement" (q24 verify windows W = 8 and 16, bf16 and nvfp4 KV).
 *   - "perf(dflash): widen the verify window past the compact graph's
 *     four-row limit", section "What changed" (an unsupported width must not
 *     silently truncate; attention reads only seq_len entries).
 *
 * For each query row and head h (KV head h / (Hq/Hkv)):
 *   s_j = sm_scale * <q, k_j>,  O = sum_j softmax(s)_j v_j,
 *   LSE = max_j s_j + ln(sum_j exp(s_j - max_j s_j))     (natural log)
 * with fp32 accumulation; O is written as bf16 (round to nearest even),
 * LSE as fp32.
 *
 * Layouts (row-major; the pools may have a page stride, everything else is
 * dense):
 *   Q, O       [total_q_rows, Hq, head_dim] bf16; the rows of request r are
 *              q_indptr[r] .. q_indptr[r+1]-1, in window order.
 *   LSE        [total_q_rows, Hq] fp32.
 *   K/V pools  num_pages pages, page p at byte offset p * kv_page_stride
 *              (default: dense), each page [Hkv, page_size, row] with
 *              bf16:  row = head_dim bf16 values;
 *              NVFP4: row = head_dim/2 code bytes (two e2m1 codes per byte,
 *                     low nibble = even element), and scale pools laid out
 *                     the same way with page stride scale_page_stride and
 *                     row = head_dim/16 bytes (one OCP e4m3 scale per 16
 *                     contiguous elements), plus one fp32 global scale per
 *                     tensor: value = e2m1(code) * e4m3(scale) * gscale.
 *              A page stride lets K and V (and their scales) share one
 *              allocation, e.g. [num_pages, 2, Hkv, page_size, row].
 *   block_table [P, block_table_stride] int32: key j of request r lives in
 *              page block_table[r][j / page_size], slot j % page_size.
 *              Entries past ceil(seq_len[r] / page_size) are never read.
 *   seq_lens   [P] int32;  q_indptr [P+1] int32 (q_indptr[0] == 0).
 *
 * Ownership: every buffer is allocated and owned by the caller.  The library
 * allocates no device memory, makes no host<->device copy and never
 * synchronises inside spec_attn_run / spec_attn_run_traced, so both may be
 * captured into a CUDA graph.  A plan is a host object owned by the library
 * between spec_attn_plan_create() and spec_attn_plan_destroy().
 *
 * Errors: every function returns a spec_attn_status.  Host-side checks run
 * in spec_attn_plan_create() (shapes, limits, host copies of seq_lens and
 * q_indptr when given) and spec_attn_run() (null or misaligned pointers,
 * workspace size).  Device-side checks (a page id outside [0, num_pages), a
 * seq_len above the plan's max_seq_len or below its window, a window wider
 * than max_w) never fault: the kernels clamp the access, set a sticky error
 * word in the workspace and go on; spec_attn_check_device_status() reads and
 * clears it.
 */
#ifndef SPEC_ATTN_H
#define SPEC_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA
 * include.  NULL means the legacy default stream. */
typedef struct CUstream_st* spec_attn_stream_t;

typedef enum spec_attn_status {
    SPEC_ATTN_OK = 0,
    SPEC_ATTN_E_INVALID_ARG = -1,          /* bad shape, pointer, alignment or value */
    SPEC_ATTN_E_UNSUPPORTED = -2,          /* valid but outside the library's limits */
    SPEC_ATTN_E_WORKSPACE_TOO_SMALL = -3,  /* workspace_bytes below the plan's need */
    SPEC_ATTN_E_CUDA = -4,                 /* a CUDA runtime call failed; see spec_attn_last_cuda_error */
    SPEC_ATTN_E_DEVICE_CHECK = -5          /* a device-side check tripped (check_device_status) */
} spec_attn_status;

typedef enum spec_attn_mask_mode {
    SPEC_ATTN_MASK_CAUSAL_IN_BLOCK = 0,
    SPEC_ATTN_MASK_NON_CAUSAL = 1
} spec_attn_mask_mode;

typedef enum spec_attn_kv_dtype {
    SPEC_ATTN_KV_BF16 = 0,
    SPEC_ATTN_KV_NVFP4 = 1
} spec_attn_kv_dtype;

typedef enum spec_attn_kernel_variant {
    SPEC_ATTN_VARIANT_AUTO = 0,       /* the library's choice for the shape */
    SPEC_ATTN_VARIANT_CUDA_CORE = 1,  /* fp32 FMA on CUDA cores */
    SPEC_ATTN_VARIANT_TCGEN05 = 2     /* 5th-generation tensor cores, TMEM accumulators */
} spec_attn_kernel_variant;

/* Device-status bits set by the kernels (spec_attn_check_device_status). */
#define SPEC_ATTN_DEV_BAD_PAGE      0x1u  /* block-table entry outside [0, num_pages) */
#define SPEC_ATTN_DEV_BAD_SEQ_LEN   0x2u  /* seq_len > max_seq_len or table capacity, or < W_r */
#define SPEC_ATTN_DEV_BAD_WINDOW    0x4u  /* W_r < 0, W_r > max_w, or rows past total_q_rows */
#define SPEC_ATTN_DEV_WAIT_TIMEOUT  0x8u  /* a pipeline wait gave up (bounded spin) */

/* Limits of the library. */
#define SPEC_ATTN_MAX_W 16
#define SPEC_ATTN_MAX_GROUP 16       /* Hq / Hkv */
#define SPEC_ATTN_MIN_PAGE_SIZE 16   /* page_size is 16, 32 or 64 */
#define SPEC_ATTN_MAX_PAGE_SIZE 64

typedef struct spec_attn_problem {
    int32_t num_reqs;            /* P >= 0 */
    int32_t total_q_rows;        /* rows of Q and O (sum of all W_r) */
    int32_t max_w;               /* upper bound on every W_r, 1..16 */
    int32_t num_q_heads;         /* Hq */
    int32_t num_kv_heads;        /* Hkv; Hq % Hkv == 0, Hq / Hkv <= 16 */
    int32_t head_dim;            /* 64, 128 or 256 */
    int32_t page_size;           /* keys per page: 16, 32 or 64 */
    int32_t num_pages;           /* pages in each pool (device bounds check); >= 1 when
                                    num_reqs > 0, even if no key is cached */
    int32_t block_table_stride;  /* int32 entries per block-table row; a row's capacity,
                                    stride x page_size keys, at most 2^31 - 1 */
    int32_t mask_mode;           /* spec_attn_mask_mode */
    int32_t kv_dtype;            /* spec_attn_kv_dtype */
    float sm_scale;              /* softmax scale; 0 selects 1/sqrt(head_dim) */
    int64_t max_seq_len;         /* upper bound on every seq_len the plan will see,
                                    at most 2^31 - 1 */
    int32_t force_splits;        /* 0: heuristic; n > 0: split the longest request's keys n ways */
    int32_t kernel_variant;      /* spec_attn_kernel_variant */
    int32_t w_invariant;         /* 1: W-invariant mode (below); 0: off */
    int32_t fixed_keys_per_split;/* W-invariant mode: keys per split, a multiple of 64
                                    (0 selects 64 x ceil(max_seq_len / 2048), at least
                                    512); ignored otherwise */
    int32_t window_left;         /* causal sliding window in keys; 0 = none (required
                                    for the non-causal mask) */
    int64_t kv_page_stride;      /* bytes from a K (or V) page to the next: 0 = dense
                                    (Hkv * page_size * row bytes); else a multiple of 16
                                    and at least the dense size */
    int64_t scale_page_stride;   /* NVFP4 scale pools, likewise (dense: Hkv * page_size
                                    * head_dim/16 bytes); ignored for bf16 */
    int32_t dense_block_kv;      /* 1: the window's own keys come from dense block
                                    tensors (spec_attn_run_dense_block), not the cache;
                                    bf16 caches only, not with w_invariant */
    int32_t early_metadata;      /* 1: the caller vouches that no kernel still running
                                    when a run starts in its stream (the one launched
                                    just before it, and any earlier one that kernel
                                    overlaps through a programmatic launch) writes
                                    seq_lens, q_indptr or block_table (true of every
                                    layer of a decode step that fills them once per
                                    step); the attention kernel then reads them while
                                    that kernel drains.  0: it waits first (safe). */
    int32_t test_stall;          /* testing only (needs kernel_variant TCGEN05): 1 makes
                                    the K producer issue nothing, so its consumers'
                                    bounded waits run out after about a second; the
                                    call then sets SPEC_ATTN_DEV_WAIT_TIMEOUT, frees its
                                    tensor memory and returns, leaving O undefined and
                                    the context usable.  0 in every real call. */
    int32_t early_context_kv;    /* 1 (needs early_metadata = 1): the caller also
                                    vouches that no such kernel writes a cached key
                                    below its request's ctx_r (the window's own keys
                                    may be written, e.g. by spec_attn_append_kv just
                                    before); the bf16 tensor-core kernel then starts
                                    the copies of each split's first K and V tile
                                    (when it holds context keys only, and with no
                                    sliding window or dense block operand) while that
                                    kernel drains.  Results are bit-identical either
                                    way.  0: it waits first (safe). */
} spec_attn_problem;

/*
 * W-invariant mode (w_invariant = 1).  Every output row comes out bit-identical
 * to the same row computed alone: window row i of request r equals the W = 1
 * call on the same cache with seq_len = ctx_r + i + 1, whatever W, P or the
 * other rows are -- the exactness rule of the page "perf(dflash): widen the
 * verify window past the compact graph's four-row limit" (section
 * "Exactness"), which greedy speculative decoding needs for its output to
 * match plain decoding.  The plan then uses split boundaries that depend only
 * on key positions (every fixed_keys_per_split keys), always writes split
 * partials and always merges them in a fold order fixed by the split index
 * alone (split s in group s mod G, G a constant of head_dim).  It
 * needs the tensor-core kernel (E_UNSUPPORTED if the CUDA-core one is
 * forced) and ignores force_splits.  Rows computed in W-invariant mode match
 * rows computed in W-invariant mode with the same fixed_keys_per_split; the
 * default mode's splits are chosen for speed and may round differently.  The
 * cost is the split count this fixes: one CTA per (split, KV head, request),
 * so the call is fastest when fixed_keys_per_split is near the typical
 * context length x P x Hkv / (number of SMs), e.g. 512 for one request with
 * 4 KV heads at 16K keys, 2048 at 64K.  The default (0) derives it from
 * max_seq_len (512 up to 16K keys, 2048 at 64K): plans that must agree
 * bitwise with each other pass the same explicit value, or have max_seq_len
 * values that round up to the same multiple of 2048 (or are both at most
 * 16384).
 */

typedef struct spec_attn_plan spec_attn_plan;   /* opaque */

/* What a plan decided; for tests, benches and logs. */
typedef struct spec_attn_plan_info {
    int32_t kernel_variant;      /* the variant that will run (never AUTO) */
    int32_t keys_per_split;      /* keys of one request one CTA sweeps (multiple of 64) */
    int32_t max_splits;          /* splits of the longest request */
    int32_t row_groups;          /* CTAs sharing one (request, KV head, split), each with
                                    its own rows; tcgen05: > 1 only above 128 query rows
                                    per KV head (groups of whole window rows) */
    int32_t grid_x, grid_y, grid_z;
    int32_t block_threads;
    int32_t smem_bytes;          /* dynamic shared memory of the split kernel */
    int32_t uses_merge;          /* 1 when a second (LSE-merge) kernel runs */
    int32_t num_sms;
    size_t workspace_bytes;
} spec_attn_plan_info;

/*
 * Validate a problem and choose the split count (keys per split) and the
 * kernel variant (the plan step of the scope table; its spec_attn_plan).
 * The split count restates the key-splitting of the page "ChunkedSmallT
 * re-streams full KV per query chunk (DFlash K>=8 verify at long context)",
 * section "Finding", without its width cap: every CTA holds all W x G rows of
 * one KV head, so widths up to 16 keep one sweep; wider ones fail here
 * rather than truncate (page "perf(dflash): widen the verify window past the
 * compact graph's four-row limit", section "What changed").  Host only; no
 * device allocation.  h_seq_lens [P] and
 * h_q_indptr [P+1] are optional host copies: when given they are checked
 * and used by the split heuristic; otherwise max_seq_len and max_w stand in
 * for every request.  A plan may be reused for every layer of a step and
 * replayed inside a CUDA graph while every device seq_len stays at or below
 * max_seq_len.  *out receives the plan; *workspace_bytes (nullable) receives
 * the bytes spec_attn_run needs.  The CUDA device current at this call is
 * the one the plan targets.
 */
int spec_attn_plan_create(const spec_attn_problem* problem, const int32_t* h_seq_lens,
                          const int32_t* h_q_indptr, spec_attn_plan** out,
                          size_t* workspace_bytes);

/* Free a plan (host memory only).  NULL is accepted. */
int spec_attn_plan_destroy(spec_attn_plan* plan);

int spec_attn_plan_get_info(const spec_attn_plan* plan, spec_attn_plan_info* info);

/*
 * Run one attention call asynchronously on `stream`: the block attention of
 * the page "DFlash2 leaves the paged graph fast path at every c>1 and
 * re-attends the whole batch context every decode step" (sections "The
 * route change" and "Scope": P x W rows over a shared paged pool through a
 * batched block table, outputs for window rows only), swept once over each
 * request's keys however wide its window (page "ChunkedSmallT re-streams full
 * KV per query chunk (DFlash K>=8 verify at long context)", section
 * "Finding"), reading only seq_len entries (page "perf(dflash): widen the
 * verify window past the compact graph's four-row limit", section "What
 * changed").
 *   q         [total_q_rows, Hq, d] bf16, 16-byte aligned
 *   k_pool, v_pool   pools as above, 16-byte aligned (NVFP4: code pools)
 *   k_scales, v_scales  NVFP4 scale pools, 16-byte aligned; NULL for bf16
 *   k_gscale, v_gscale  NVFP4 global scales; ignored for bf16
 *   block_table [P, block_table_stride] int32, seq_lens [P], q_indptr [P+1]
 *   o         [total_q_rows, Hq, d] bf16 output, 16-byte aligned
 *   lse       [total_q_rows, Hq] fp32 output, or NULL
 *   workspace caller-owned device scratch of at least the plan's
 *             workspace_bytes, 256-byte aligned; its first 256 bytes hold the
 *             sticky device-status word, which the caller zeroes once after
 *             allocating it (spec_attn_reset_device_status).  One workspace
 *             must not be shared by runs that may overlap on the GPU.
 * All device pointers must belong to the plan's device.  Returns
 * SPEC_ATTN_E_CUDA if a launch fails.
 */
int spec_attn_run(const spec_attn_plan* plan, const void* q, const void* k_pool,
                  const void* v_pool, const void* k_scales, const void* v_scales,
                  float k_gscale, float v_gscale, const int32_t* block_table,
                  const int32_t* seq_lens, const int32_t* q_indptr, void* o, float* lse,
                  void* workspace, size_t workspace_bytes, spec_attn_stream_t stream);

/*
 * spec_attn_run plus an index/mask trace: trace [total_q_rows, Hq, 2] int64
 * (zeroed by the caller) receives, for every output (row, head), the number
 * of keys the kernels let into its softmax and the sum of their physical
 * slot ids (page * page_size + slot), accumulated over all splits.  This is
 * the floating-point-free check that every row saw exactly its mask's keys
 * through the block table.  Slower than spec_attn_run; for validation.
 */
int spec_attn_run_traced(const spec_attn_plan* plan, const void* q, const void* k_pool,
                         const void* v_pool, const void* k_scales, const void* v_scales,
                         float k_gscale, float v_gscale, const int32_t* block_table,
                         const int32_t* seq_lens, const int32_t* q_indptr, void* o,
                         float* lse, int64_t* trace, void* workspace,
                         size_t workspace_bytes, spec_attn_stream_t stream);

/*
 * Dense block operand (dense_block_kv = 1).  The window's own W_r keys are
 * not in the cache: they come from dense tensors block_k, block_v
 * [total_q_rows, Hkv, head_dim] bf16 (16-byte aligned), row q_indptr[r] + i
 * holding key ctx_r + i = seq_len[r] - W_r + i.  The cache holds the context
 * keys 0 .. ctx_r - 1 only, and the block table need cover just those.  This
 * is the "Narrow" shape of the page "DFlash2 leaves the paged graph fast path
 * at every c>1 and re-attends the whole batch context every decode step"
 * (section "Scope"): the draft's block K/V are discarded after the step, so
 * they are kept apart from the paged context.  Masks, window and outputs are
 * as for spec_attn_run, over the keys 0 .. seq_len[r] - 1 so formed.  trace
 * (nullable, as spec_attn_run_traced) counts a block key with slot id
 * -(1 + its row).  A plan made with dense_block_kv = 1 runs only here, and
 * this entry point needs such a plan (else SPEC_ATTN_E_INVALID_ARG).
 */
int spec_attn_run_dense_block(const spec_attn_plan* plan, const void* q, const void* block_k,
                              const void* block_v, const void* k_pool, const void* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* q_indptr, void* o, float* lse, int64_t* trace,
                              void* workspace, size_t workspace_bytes, spec_attn_stream_t stream);

/*
 * KV append: write the window's new key and value rows into their cache slots
 * (page "perf(dflash): widen the verify window past the compact graph's
 * four-row limit", section "What changed": the window's rows go into the
 * cache, later steps overwrite the rows a rejected tail leaves stale, and
 * attention reads only seq_len entries).  seq_len_r already counts the
 * window, so window row i of request r is written at key position
 * pos = seq_len_r - W_r + i: page block_table[r][pos / page_size], slot
 * pos % page_size, for every KV head.
 *   k_new, v_new  [total_q_rows, Hkv, d] bf16, rows in q_indptr order,
 *                 16-byte aligned; read only
 *   k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table,
 *   seq_lens, q_indptr   as for spec_attn_run; the pools (and, for NVFP4,
 *                 the scale pools) are written at the window's slots only
 *   workspace     as for spec_attn_run; spec_attn_append_kv uses only its
 *                 device-status word (workspace_bytes >= 256)
 * bf16 caches receive the bits unchanged.  NVFP4 caches receive each run of
 * 16 head_dim elements quantised against the cache's decode scale g (k_gscale
 * or v_gscale): amax = max |x|; scale byte = E4M3(amax / (6 g)); den =
 * scale * g; code = E2M1(x / den), or +0 throughout when den = 0; every
 * product and quotient in binary32 rounded to nearest even in that order, the
 * conversions to nearest even, saturating at 448 and 6 and keeping the sign.
 * Values beyond 6 * 448 * g clip.  NaN or infinite inputs give unspecified
 * codes.  Device-side checks (bad window, seq_len or page id) set the same
 * status bits as spec_attn_run and skip the row; nothing else is written.
 * Asynchronous on `stream`, allocation-free, graph capturable.
 */
int spec_attn_append_kv(const spec_attn_plan* plan, const void* k_new, const void* v_new, void* k_pool,
                        void* v_pool, void* k_scales, void* v_scales, float k_gscale, float v_gscale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_indptr,
                        void* workspace, size_t workspace_bytes, spec_attn_stream_t stream);

/*
 * spec_attn_append_kv followed by spec_attn_run on the same stream: the step
 * a verify layer takes once it has the window's K and V.  Every argument is
 * checked before either kernel is launched, so a rejected call writes
 * nothing.  The attention kernel is launched as a programmatic dependent of
 * the append and reads the cache only after the append has completed.
 * workspace as for spec_attn_run (the plan's workspace_bytes).
 */
int spec_attn_run_append(const spec_attn_plan* plan, const void* q, const void* k_new, const void* v_new,
                         void* k_pool, void* v_pool, void* k_scales, void* v_scales, float k_gscale,
                         float v_gscale, const int32_t* block_table, const int32_t* seq_lens,
                         const int32_t* q_indptr, void* o, float* lse, void* workspace, size_t workspace_bytes,
                         spec_attn_stream_t stream);

/*
 * Optional timing hooks: when set (both non-NULL; cudaEvent_t values), every
 * later run records `split_begin` on its stream just before the split-KV
 * kernel launch and `split_end` just after it, so a caller can time that
 * kernel alone with cudaEventElapsedTime.  Pass NULLs to clear.
 */
int spec_attn_plan_set_timing_events(spec_attn_plan* plan, void* split_begin, void* split_end);

/* Zero the workspace's device-status word (asynchronous on `stream`). */
int spec_attn_reset_device_status(void* workspace, spec_attn_stream_t stream);

/* Synchronise `stream`, read the device-status word into *bits (nullable)
 * and clear it.  Returns SPEC_ATTN_E_DEVICE_CHECK when any bit was set. */
int spec_attn_check_device_status(void* workspace, spec_attn_stream_t stream, uint32_t* bits);

/* Name of a status code; never NULL. */
const char* spec_attn_status_string(int status);

/* The last CUDA error code this thread saw inside the library (0 if none). */
int spec_attn_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int spec_attn_version(void);

/*
 * spec_attn_run without a workspace argument, for callers that cannot
 * allocate device memory (code running where cudaMalloc is not allowed, such
 * as inside an allocator hook or a host callback, or a plugin handed only its
 * input and output buffers).  No counterpart on the pages this library
 * restates: it is a convenience of this library.
 *
 * Scratch comes from one array of SPEC_ATTN_NOALLOC_SCRATCH_BYTES (32 MiB) in
 * the library's own device memory; every GPU that loads the library holds it
 * until the process exits.  A plan whose workspace_bytes exceeds that size is
 * rejected with SPEC_ATTN_E_WORKSPACE_TOO_SMALL.  Every call on a device
 * shares the array, so calls that may overlap on the GPU race and must be
 * serialised by the caller; each call clears the device-status word at the
 * head of the array once its host checks have passed (a rejected call writes
 * nothing), and spec_attn_noalloc_check_device_status reads what the last
 * call left.  The first call on each device looks up the array's device
 * address (with that device current) and caches it with the id of the
 * context it belongs to; make that first call before any stream capture.  A
 * call made in another context of the device (after cudaDeviceReset, which
 * creates the primary context anew) looks the address up again, so make the
 * first call after a reset outside stream capture too.  Allocates nothing;
 * other arguments and errors as spec_attn_run.
 */
#define SPEC_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int spec_attn_run_noalloc(const spec_attn_plan* plan, const void* q, const void* k_pool,
                          const void* v_pool, const void* k_scales, const void* v_scales,
                          float k_gscale, float v_gscale, const int32_t* block_table,
                          const int32_t* seq_lens, const int32_t* q_indptr, void* o, float* lse,
                          spec_attn_stream_t stream);

/*
 * Device-status bits of the last spec_attn_run_noalloc call on the current
 * device (read and cleared, synchronising `stream` like
 * spec_attn_check_device_status); 0 in *bits, and SPEC_ATTN_OK, before any
 * such call.  Returns SPEC_ATTN_E_DEVICE_CHECK when a bit is set.  Also no
 * counterpart on the pages: it completes the no-alloc entry point.
 */
int spec_attn_noalloc_check_device_status(spec_attn_stream_t stream, uint32_t* bits);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_ATTN_H */
