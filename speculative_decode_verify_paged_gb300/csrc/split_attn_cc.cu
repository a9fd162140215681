// Split-KV block attention on CUDA cores (fp32 FMA), bf16 or NVFP4 KV.
//
// One CTA = (split s of request r's keys) x (KV head kvh) x (row group).
// A row group holds up to 8 * RPW of the request's W x G query rows that
// share KV head kvh (row m = window row m / G, query head kvh * G + m % G),
// so the K/V pages of a split are read once for all those rows: the single
// sweep per window the page "ChunkedSmallT re-streams full KV per query
// chunk (DFlash K>=8 verify at long context)" (section "Finding") asks for,
// for every W up to 16.  Keys are fetched in 16-key units (a whole page of 16
// keys, or a half or quarter of a 32- or 64-key page) through the block table
// with 16-byte cp.async copies into a ring of shared-memory stages.
//
// Each warp owns RPW rows; lane l owns head_dim elements [l*D/32, (l+1)*D/32).
// Per unit: partial dot products per lane, a transposing butterfly reduction
// (16 shuffles for 16 keys), the causal-in-block / non-causal mask and the
// sliding window by key index, an online softmax in base 2 (scores
// pre-scaled by sm_scale * log2 e), and O += p * V.  A split's result is
// written as the final bf16 output when the request has one split, else as
// the split partial (fp16 O / l over its scale, the log2-sum-exp and the
// scale) for the LSE merge.
//
// NVFP4 pages are decoded in registers: e2m1 code * e4m3 block scale; the
// per-tensor global scales are folded into the score scale (K) and the
// output scale (V) by the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace spec_attn {
namespace {

constexpr int kUnit = 16;   // keys per unit
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int D, int KV>
struct CcStage {
    static constexpr int kCodeBytes = (KV == 0) ? kUnit * D * 2 : kUnit * D / 2;  // per K or V page
    static constexpr int kScaleBytes = (KV == 0) ? 0 : kUnit * D / 16;
    static constexpr int kHalf = kCodeBytes + kScaleBytes;
    static constexpr int kBytes = 2 * kHalf;  // K then V
    static_assert(kCodeBytes % 16 == 0 && kScaleBytes % 16 == 0, "16-byte chunks");
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
    // wait_group needs an immediate; the ring depth is at most 8.
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}

// Load the lane's DPL elements of one K or V row (key j) of a staged page as floats.
template <int D, int KV>
__device__ __forceinline__ void load_row_slice(const unsigned char* half, int j, int lane,
                                               float (&x)[D / 32]) {
    constexpr int DPL = D / 32;
    if constexpr (KV == 0) {
        const uint16_t* row = reinterpret_cast<const uint16_t*>(half) + j * D + lane * DPL;
        if constexpr (DPL == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(row);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else if constexpr (DPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(row);
            x[0] = __uint_as_float(u.x << 16);
            x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16);
            x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(row);
            x[0] = __uint_as_float(u << 16);
            x[1] = __uint_as_float(u & 0xffff0000u);
        }
    } else {
        const unsigned char* codes = half + j * (D / 2) + lane * (DPL / 2);
        const unsigned char* scales = half + CcStage<D, KV>::kCodeBytes + j * (D / 16);
        const float sc = e4m3_to_float(scales[(lane * DPL) / 16]);
        uint32_t packed;
        if constexpr (DPL == 8)
            packed = *reinterpret_cast<const uint32_t*>(codes);
        else if constexpr (DPL == 4)
            packed = *reinterpret_cast<const uint16_t*>(codes);
        else
            packed = *codes;
#pragma unroll
        for (int i = 0; i < DPL; ++i) x[i] = e2m1_to_float((packed >> (4 * i)) & 0xfu) * sc;
    }
}

// Sum 16 per-lane partial values over the warp so that lanes 2k and 2k+1
// both end up with the full sum of value k.
__device__ __forceinline__ float transpose_reduce16(const float (&x)[16], int lane) {
    float y8[8], y4[4], y2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float send = b4 ? x[v] : x[v + 8];
        const float keep = b4 ? x[v + 8] : x[v];
        y8[v] = keep + __shfl_xor_sync(kFullMask, send, 16);
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float send = b3 ? y8[v] : y8[v + 4];
        const float keep = b3 ? y8[v + 4] : y8[v];
        y4[v] = keep + __shfl_xor_sync(kFullMask, send, 8);
    }
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        const float send = b2 ? y4[v] : y4[v + 2];
        const float keep = b2 ? y4[v + 2] : y4[v];
        y2[v] = keep + __shfl_xor_sync(kFullMask, send, 4);
    }
    const float send = b1 ? y2[0] : y2[1];
    const float keep = b1 ? y2[1] : y2[0];
    const float y1 = keep + __shfl_xor_sync(kFullMask, send, 2);
    return y1 + __shfl_xor_sync(kFullMask, y1, 1);
}

template <int D, int KV, int RPW, bool TRACE>
__global__ void __launch_bounds__(kThreads)
split_attn_cc_kernel(const SplitParams p, const int stages) {
    constexpr int DPL = D / 32;
    using Stage = CcStage<D, KV>;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = blockIdx.x % p.row_groups;
    const int split = blockIdx.x / p.row_groups;
    const int kvh = blockIdx.y;
    const int r = blockIdx.z;

    // launched as a programmatic dependent: nothing global is touched before
    // the previous kernel in the stream has completed (with early_metadata,
    // nothing but the lengths and windows, which that kernel does not write)
    if (!p.early_metadata) pdl_wait_primary();
    ReqInfo ri;
    const bool reporter = (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0);
    if (!load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                      p.bt_stride << (4 + p.page_shift), p.keys_per_split, reporter ? p.status : nullptr, ri,
                      p.window_left, p.split_align, p.dense_block))
        return;
    if (split >= ri.nsplits) return;
    if (p.early_metadata) pdl_wait_primary();
    const int G = p.group;
    const int R = ri.w * G;
    const int row_lo = rg * p.rows_per_cta;
    if (row_lo >= R) return;

    const int key_lo = ri.key_base + split * p.keys_per_split;
    const int key_hi = min(key_lo + p.keys_per_split, ri.cache_len);
    // the loop runs over 16-key units: unit u is slots (u & sub_mask) * 16 .. +15
    // of page block_table[r][u >> page_shift]; with the dense block operand the
    // request's last split ends with one more unit, rows row0 .. row0 + W - 1 of
    // block_k / block_v (keys ctx .. len - 1)
    const int page_first = key_lo / kUnit;
    const int npages = key_hi > key_lo ? (key_hi - 1) / kUnit - page_first + 1 : 0;
    const bool has_block = p.dense_block && split == ri.nsplits - 1;
    const int nunits = npages + (has_block ? 1 : 0);
    const int32_t* bt_row = p.block_table + (size_t)r * p.bt_stride;
    const int page_keys = kUnit << p.page_shift;
    const int sub_mask = (1 << p.page_shift) - 1;

    // ---- this warp's rows ----
    int m_row[RPW], hq[RPW], qrow[RPW], hi_key[RPW], lo_key[RPW];
    bool valid[RPW];
    float q[RPW][DPL];
    float o_acc[RPW][DPL];
    float m_run[RPW], l_run[RPW];
    long long tr_cnt[RPW], tr_sum[RPW];
    bool any_valid = false;
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        m_row[t] = row_lo + warp * RPW + t;
        valid[t] = m_row[t] < R;
        any_valid |= valid[t];
        const int i = valid[t] ? m_row[t] / G : 0;
        hq[t] = kvh * G + (valid[t] ? m_row[t] % G : 0);
        qrow[t] = ri.row0 + i;
        hi_key[t] = (p.mask_mode == 0) ? (ri.ctx + i) : (ri.len - 1);
        lo_key[t] = (p.window_left > 0) ? max(0, hi_key[t] - p.window_left + 1) : 0;
        m_run[t] = -INFINITY;
        l_run[t] = 0.f;
        tr_cnt[t] = 0;
        tr_sum[t] = 0;
        const uint16_t* qp = p.q + ((size_t)qrow[t] * p.num_q_heads + hq[t]) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            q[t][e] = valid[t] ? bf16_bits_to_float(qp[e]) * p.score_scale_log2 : 0.f;
            o_acc[t][e] = 0.f;
        }
    }

    // ---- page loader (all threads) ----
    auto issue_page = [&](int pi) {
        if (pi < npages) {
            const int u = page_first + pi;
            int phys = bt_row[u >> p.page_shift];
            if (phys < 0 || phys >= p.num_pages) {
                if (tid == 0) atomicOr(p.status, kDevBadPage);
                phys = 0;
            }
            unsigned char* st = smem + (size_t)(pi % stages) * Stage::kBytes;
            // first slot of the unit within its page-head
            const size_t slot0 = (size_t)kvh * page_keys + (u & sub_mask) * kUnit;
            const size_t kv_off = (size_t)phys * p.kv_page_stride + slot0 * (Stage::kCodeBytes / kUnit);
            const unsigned char* ksrc = static_cast<const unsigned char*>(p.k_pool) + kv_off;
            const unsigned char* vsrc = static_cast<const unsigned char*>(p.v_pool) + kv_off;
            for (int c = tid; c < Stage::kCodeBytes / 16; c += kThreads) {
                cp_async16(st + c * 16, ksrc + c * 16);
                cp_async16(st + Stage::kHalf + c * 16, vsrc + c * 16);
            }
            if constexpr (KV == 1) {
                const size_t sc_off = (size_t)phys * p.scale_page_stride + slot0 * (D / 16);
                const unsigned char* kss = p.k_scales + sc_off;
                const unsigned char* vss = p.v_scales + sc_off;
                for (int c = tid; c < Stage::kScaleBytes / 16; c += kThreads) {
                    cp_async16(st + Stage::kCodeBytes + c * 16, kss + c * 16);
                    cp_async16(st + Stage::kHalf + Stage::kCodeBytes + c * 16, vss + c * 16);
                }
            }
        } else if (KV == 0 && pi == npages && has_block) {   // (bf16 caches only)
            // the window's own rows (bf16): row j of the unit is block row row0 + j;
            // rows past W are zeros (never read from another window)
            unsigned char* st = smem + (size_t)(pi % stages) * Stage::kBytes;
            constexpr int kRowPieces = D * 2 / 16;
            for (int c = tid; c < kUnit * kRowPieces; c += kThreads) {
                const int j = c / kRowPieces, piece = c % kRowPieces;
                unsigned char* kd = st + j * (D * 2) + piece * 16;
                unsigned char* vd = st + Stage::kHalf + j * (D * 2) + piece * 16;
                if (j < ri.w) {
                    const size_t off = (((size_t)(ri.row0 + j) * p.num_kv_heads + kvh) * D) * 2 + piece * 16;
                    cp_async16(kd, reinterpret_cast<const unsigned char*>(p.block_k) + off);
                    cp_async16(vd, reinterpret_cast<const unsigned char*>(p.block_v) + off);
                } else {
                    *reinterpret_cast<uint4*>(kd) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(vd) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        cp_async_commit();
    };

    for (int pi = 0; pi < stages - 1; ++pi) issue_page(pi);

    for (int pi = 0; pi < nunits; ++pi) {
        issue_page(pi + stages - 1);
        cp_async_wait_dyn(stages - 1);
        __syncthreads();
        const unsigned char* st = smem + (size_t)(pi % stages) * Stage::kBytes;
        const bool blk = pi == npages;   // the dense block unit
        const int kbase = blk ? ri.ctx : (page_first + pi) * kUnit;
        const int kend = blk ? ri.len : key_hi;
        if (any_valid) {
            // scores for the 16 keys of this page
            float part[RPW][16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float kx[DPL];
                load_row_slice<D, KV>(st, j, lane, kx);
#pragma unroll
                for (int t = 0; t < RPW; ++t) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc = fmaf(q[t][e], kx[e], acc);
                    part[t][j] = acc;
                }
            }
            const int key = kbase + (lane >> 1);
            float pj[RPW];
#pragma unroll
            for (int t = 0; t < RPW; ++t) {
                const float sc = transpose_reduce16(part[t], lane);
                const bool vis = (key < kend) && (key <= hi_key[t]) && (key >= lo_key[t]);
                float mx = vis ? sc : -INFINITY;
#pragma unroll
                for (int off = 2; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
                const float m_new = fmaxf(m_run[t], mx);
                const float alpha = (m_run[t] == -INFINITY) ? 0.f : fast_exp2(m_run[t] - m_new);
                const float pv = vis ? fast_exp2(sc - m_new) : 0.f;
                float ps = pv;
#pragma unroll
                for (int off = 2; off < 32; off <<= 1) ps += __shfl_xor_sync(kFullMask, ps, off);
                l_run[t] = l_run[t] * alpha + ps;
                m_run[t] = m_new;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o_acc[t][e] *= alpha;
                pj[t] = pv;
                if constexpr (TRACE) {
                    if (vis && (lane & 1) == 0) {
                        tr_cnt[t] += 1;
                        if (blk) {   // a dense block key has no cache slot: -(1 + its row)
                            tr_sum[t] += -1 - (long long)(ri.row0 + key - ri.ctx);
                        } else {
                            int phys = bt_row[(page_first + pi) >> p.page_shift];
                            if (phys < 0 || phys >= p.num_pages) phys = 0;
                            tr_sum[t] += (long long)phys * page_keys + (key & (page_keys - 1));
                        }
                    }
                }
            }
            // O += P V
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float vx[DPL];
                load_row_slice<D, KV>(st + Stage::kHalf, j, lane, vx);
                // Slots past seq_len hold stale data (possibly non-finite);
                // their weight is 0, but 0 * NaN is NaN, so drop the values.
                if (kbase + j >= kend) {
#pragma unroll
                    for (int e = 0; e < DPL; ++e) vx[e] = 0.f;
                }
#pragma unroll
                for (int t = 0; t < RPW; ++t) {
                    const float w = __shfl_sync(kFullMask, pj[t], 2 * j);
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o_acc[t][e] = fmaf(w, vx[e], o_acc[t][e]);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    pdl_launch_dependents();

    // ---- epilogue ----
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        if constexpr (TRACE) {
            long long c = tr_cnt[t], s = tr_sum[t];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                c += __shfl_xor_sync(kFullMask, c, off);
                s += __shfl_xor_sync(kFullMask, s, off);
            }
            if (valid[t] && lane == 0 && p.trace) {
                unsigned long long* tp = reinterpret_cast<unsigned long long*>(
                    p.trace + ((size_t)qrow[t] * p.num_q_heads + hq[t]) * 2);
                atomicAdd(tp, (unsigned long long)c);
                atomicAdd(tp + 1, (unsigned long long)s);
            }
        }
        if (!valid[t]) continue;
        const float inv_l = (l_run[t] > 0.f) ? (p.out_scale / l_run[t]) : 0.f;
        const float lse2 = (l_run[t] > 0.f) ? (m_run[t] + log2f(l_run[t])) : -INFINITY;
        const size_t oi = ((size_t)qrow[t] * p.num_q_heads + hq[t]);
        if (ri.nsplits == 1 && !p.always_partials) {
            uint16_t* op = p.o + oi * D + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; e += 2) {
                const uint32_t lo = float_to_bf16_bits(o_acc[t][e] * inv_l);
                const uint32_t hi = float_to_bf16_bits(o_acc[t][e + 1] * inv_l);
                *reinterpret_cast<uint32_t*>(op + e) = lo | (hi << 16);
            }
            if (p.lse && lane == 0) p.lse[oi] = lse2 * kLn2;
        } else {
            // fp16 of value / scale, scale = the row's largest magnitude
            const size_t pi = partial_pair(split, p.total_rows, p.num_q_heads, G, kvh, qrow[t], hq[t] - kvh * G);
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) amax = fmaxf(amax, fabsf(o_acc[t][e] * inv_l));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
            const float sc = amax > 0.f ? inv_l / amax : 0.f;
            // this lane's DPL values: elements lane * DPL .. of the row, inside
            // chunk lane * DPL / 8 of the request's chunk-major block
            const int rtot = ri.w * G, mg = (qrow[t] - ri.row0) * G + (hq[t] - kvh * G);
            uint32_t* wp = reinterpret_cast<uint32_t*>(
                p.ws_o + partial_pair(split, p.total_rows, p.num_q_heads, G, kvh, ri.row0, 0) * D +
                partial_chunk(lane * DPL / 8, rtot, mg) + (lane * DPL) % 8);
#pragma unroll
            for (int e = 0; e < DPL; e += 2) wp[e / 2] = pack_half2(o_acc[t][e] * sc, o_acc[t][e + 1] * sc);
            if (lane == 0) p.ws_ls[pi] = make_float2(lse2, amax);
        }
    }
}

template <int D, int KV, int RPW, bool TRACE>
constexpr auto cc_kernel_ptr() {
    return &split_attn_cc_kernel<D, KV, RPW, TRACE>;
}

using CcKernel = void (*)(const SplitParams, const int);

template <int D, int KV, bool TRACE>
CcKernel pick_rpw(int rpw) {
    switch (rpw) {
        case 1: return cc_kernel_ptr<D, KV, 1, TRACE>();
        case 2: return cc_kernel_ptr<D, KV, 2, TRACE>();
        default: return cc_kernel_ptr<D, KV, 4, TRACE>();
    }
}

template <int D>
CcKernel pick_kv(int kv, int rpw, bool traced) {
    if (kv == 0) return traced ? pick_rpw<D, 0, true>(rpw) : pick_rpw<D, 0, false>(rpw);
    return traced ? pick_rpw<D, 1, true>(rpw) : pick_rpw<D, 1, false>(rpw);
}

CcKernel pick(int d, int kv, int rpw, bool traced) {
    switch (d) {
        case 64: return pick_kv<64>(kv, rpw, traced);
        case 128: return pick_kv<128>(kv, rpw, traced);
        case 256: return pick_kv<256>(kv, rpw, traced);
        default: return nullptr;
    }
}

int stage_bytes(int d, int kv) {
    const int code = (kv == 0) ? kUnit * d * 2 : kUnit * d / 2;
    const int scale = (kv == 0) ? 0 : kUnit * d / 16;
    return 2 * (code + scale);
}

}  // namespace

CcConfig cc_config(int head_dim, int kv_dtype, int max_rows) {
    CcConfig c;
    c.rows_per_warp = (max_rows <= kWarps) ? 1 : (max_rows <= 2 * kWarps) ? 2 : 4;
    const int sb = stage_bytes(head_dim, kv_dtype);
    int st = (96 * 1024) / sb;
    st = st < 2 ? 2 : (st > 8 ? 8 : st);
    c.stages = st;
    c.smem_bytes = st * sb;
    c.threads = kThreads;
    return c;
}

cudaError_t cc_prepare(int head_dim, int kv_dtype, const CcConfig& cfg) {
    for (int traced = 0; traced < 2; ++traced) {
        CcKernel k = pick(head_dim, kv_dtype, cfg.rows_per_warp, traced != 0);
        if (!k) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t cc_launch(const SplitParams& p, int kv_dtype, const CcConfig& cfg, bool traced,
                      dim3 grid, cudaStream_t stream, bool programmatic) {
    CcKernel k = pick(p.head_dim, kv_dtype, cfg.rows_per_warp, traced);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(cfg.threads, 1, 1);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k, p, cfg.stages);
}

}  // namespace spec_attn
