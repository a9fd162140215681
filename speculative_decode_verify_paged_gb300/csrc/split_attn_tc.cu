// Split-KV block attention on 5th-generation tensor cores (tcgen05 + TMEM),
// bf16 KV, for sm_103a.
//
// One CTA = (split s of request r's keys) x (KV head kvh).  Its query tile is
// all W x G rows of the request that read KV head kvh (row m = window row
// m / G, query head kvh * G + m % G), padded to the MMA's M = 128, so every
// K/V page of the split is streamed from HBM exactly once whatever W is --
// the single sweep per window that the page "ChunkedSmallT re-streams full
// KV per query chunk (DFlash K>=8 verify at long context)" (section
// "Finding") finds missing for W > 8.  No output is produced for context
// rows (page "DFlash2 leaves the paged graph fast path at every c>1 ...",
// section "The cost").
//
// Warp roles (256 threads):
//   warp 0      TMA producer: reads the block table, loads 64-key K and V
//               tiles (four 16-key pages, one 2 KB box per 64 head_dim
//               elements) into a ring of shared-memory stages, 128-byte
//               swizzled so the MMA reads them directly.
//   warp 1      allocates TMEM; one lane issues the MMAs:
//                 S_t = Q K_t^T   (M 128, N 64, bf16 -> fp32 in TMEM, double-buffered)
//                 O  += P_t V_t   (M 128, N head_dim, P from shared memory, V MN-major)
//   warps 2-7   load the query tile once (warps 4-7 then switch roles).
//   warps 4-7   softmax: thread m owns row m (TMEM lane m).  Per tile it reads
//               its 64 scores, applies the causal-in-block / non-causal mask by
//               key index, updates a base-2 online softmax whose reference
//               maximum moves only when a score exceeds it by more than 2^8
//               (then the row of O in TMEM is rescaled), writes P as bf16 into
//               the swizzled A-operand tile, and at the end normalises O and
//               writes the output (or an fp32 partial for the LSE merge).
//
// Every wait on an mbarrier is bounded: on time-out the CTA raises the
// device-status bit, stops issuing, drains its in-flight copies and MMAs,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec_attn {

namespace {

using namespace sm100;

constexpr int kBN = 64;        // keys per tile
constexpr int kM = 128;        // MMA rows (query tile, padded)
constexpr int kTcThreads = 256;
constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM cycles
constexpr long long kDrainLimit = 200000000LL;
constexpr float kRescaleThreshold = 8.0f;        // log2 units: rescale when max grows by > 2^8

template <int D>
struct TcLayout {
    static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along head_dim
    static constexpr int kQBytes = kM * D * 2;
    static constexpr int kTileBytes = kBN * D * 2;         // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPBytes = kM * kBN * 2;
    static constexpr int kAuxBytes = 1024;
    static constexpr int kMaxDyn = 232448;                  // 227 KB opt-in limit
    static constexpr int kFit = (kMaxDyn - 1024 - kQBytes - kPBytes - kAuxBytes) / kStageBytes;
    static constexpr int kStages = kFit > 4 ? 4 : kFit;
    static constexpr int kSmem = 1024 + kQBytes + kStages * kStageBytes + kPBytes + kAuxBytes;
    static constexpr uint32_t kTmemCols = (D + 2 * kBN) <= 256 ? 256u : 512u;
    static_assert(kStages >= 2, "need at least two stages");
};

struct TcAux {
    uint64_t k_full[4];
    uint64_t v_full[4];
    uint64_t kv_empty[4];
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t q_full;
    uint64_t drain;
    int32_t pages[4][4];
    uint32_t tmem_base;
    int abort;
};

// Warp-uniform bounded wait (all 32 lanes leave together).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const long long t0 = clock64();
    while (true) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(kFullMask, ok)) return true;
        const bool give_up = (*abort != 0) || (clock64() - t0 > kWaitLimit);
        if (__any_sync(kFullMask, give_up)) {
            *abort = 1;
            return false;
        }
    }
}

template <int D, bool TRACE>
__global__ void __launch_bounds__(kTcThreads, 1)
split_attn_tc_kernel(const SplitParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    using L = TcLayout<D>;
    constexpr int S = L::kStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;

    ReqInfo ri;
    const bool reporter = (tid == 0 && split == 0 && kvh == 0);
    if (!load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                      p.bt_stride * 16, p.keys_per_split, reporter ? p.status : nullptr, ri))
        return;
    if (split >= ri.nsplits) return;
    const int G = p.group;
    const int R = ri.w * G;  // <= 128: the plan admits this kernel only when max_w * G <= 128
    const int key_lo = split * p.keys_per_split;
    const int key_hi = min(key_lo + p.keys_per_split, ri.len);
    const int T = (key_hi - key_lo + kBN - 1) / kBN;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sQ = smem;
    unsigned char* sStage = smem + L::kQBytes;
    unsigned char* sP = sStage + S * L::kStageBytes;
    TcAux* aux = reinterpret_cast<TcAux*>(sP + L::kPBytes);
    volatile int* abort = &aux->abort;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&aux->k_full[s], 1);
            mbar_init(&aux->v_full[s], 1);
            mbar_init(&aux->kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&aux->s_full[b], 1);
            mbar_init(&aux->s_empty[b], 4);
        }
        mbar_init(&aux->p_full, 4);
        mbar_init(&aux->o_done, 1);
        mbar_init(&aux->q_full, 6);
        mbar_init(&aux->drain, 1);
        aux->abort = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    if (warp == 1) tmem_alloc(&aux->tmem_base, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = aux->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int32_t* bt = p.block_table + (size_t)r * p.bt_stride;
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int s = t % S;
                if (t >= S && !mbar_wait(&aux->kv_empty[s], ((t / S) - 1) & 1, abort, kWaitLimit)) break;
                const int key0 = key_lo + t * kBN;
                const int np = min(4, (key_hi - key0 + 15) / 16);
                unsigned char* kt = sStage + s * L::kStageBytes;
                unsigned char* vt = kt + L::kTileBytes;
                int phys[4];
                for (int pp = 0; pp < np; ++pp) {
                    int pg = bt[key0 / 16 + pp];
                    if (pg < 0 || pg >= p.num_pages) {
                        atomicOr(p.status, kDevBadPage);
                        pg = 0;
                    }
                    phys[pp] = pg;
                    if (TRACE) aux->pages[s][pp] = pg;
                }
                const uint32_t bytes = static_cast<uint32_t>(np * L::kChunks * 2048);
                mbar_arrive_expect_tx(&aux->k_full[s], bytes);
                for (int pp = 0; pp < np; ++pp)
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_4d(kt + c * (kBN * 128) + pp * 2048, &tmk, c * 64, 0, kvh, phys[pp],
                                    &aux->k_full[s]);
                mbar_arrive_expect_tx(&aux->v_full[s], bytes);
                for (int pp = 0; pp < np; ++pp)
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_4d(vt + c * (kBN * 128) + pp * 2048, &tmv, c * 64, 0, kvh, phys[pp],
                                    &aux->v_full[s]);
                issued = t + 1;
            }
            if (*abort) {
                // let every copy still in flight land before the CTA's shared memory goes away
                for (int t = max(0, issued - S); t < issued; ++t) {
                    volatile int no_abort = 0;
                    mbar_wait(&aux->k_full[t % S], (t / S) & 1, &no_abort, kDrainLimit);
                    mbar_wait(&aux->v_full[t % S], (t / S) & 1, &no_abort, kDrainLimit);
                }
                atomicOr(p.status, kDevWaitTimeout);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kBN, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kM, D, 0, 1);
            const uint32_t q_addr = smem_addr(sQ);
            const uint32_t p_addr = smem_addr(sP);
            bool ok = mbar_wait(&aux->q_full, 0, abort, kWaitLimit);
            tc_fence_after();
            auto issue_s = [&](int t) -> bool {
                const int s = t % S, b = t & 1;
                if (!mbar_wait(&aux->k_full[s], (t / S) & 1, abort, kWaitLimit)) return false;
                if (t >= 2 && !mbar_wait(&aux->s_empty[b], ((t >> 1) - 1) & 1, abort, kWaitLimit)) return false;
                tc_fence_after();
                const uint32_t k_addr = smem_addr(sStage + s * L::kStageBytes);
                const uint32_t d_tmem = tmem + D + b * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c = kk >> 2, sub = kk & 3;
                    const uint64_t a = smem_desc_sw128(q_addr + c * (kM * 128) + sub * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(k_addr + c * (kBN * 128) + sub * 32, 16, 1024);
                    mma_bf16_ss(d_tmem, a, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&aux->s_full[b]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int t = 0; ok && t < T; ++t) {
                if (t + 1 < T && !(ok = issue_s(t + 1))) break;
                const int s = t % S;
                if (!(ok = mbar_wait(&aux->p_full, t & 1, abort, kWaitLimit))) break;
                if (!(ok = mbar_wait(&aux->v_full[s], (t / S) & 1, abort, kWaitLimit))) break;
                tc_fence_after();
                const int key0 = key_lo + t * kBN;
                const int np = min(4, (key_hi - key0 + 15) / 16);
                const uint32_t v_addr = smem_addr(sStage + s * L::kStageBytes + L::kTileBytes);
                for (int kk = 0; kk < np; ++kk) {
                    const uint64_t a = smem_desc_sw128(p_addr + kk * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(v_addr + kk * 2048, kBN * 128, 1024);
                    mma_bf16_ss(tmem, a, bd, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&aux->kv_empty[s]);
                mma_commit(&aux->o_done);
            }
            // every MMA this thread issued completes before TMEM is released
            mma_commit(&aux->drain);
            volatile int no_abort = 0;
            mbar_wait(&aux->drain, 0, &no_abort, kDrainLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ query tile (warps 2-7)
        {
            const int qt = tid - 64;  // 0..191
            constexpr int kPieces = D / 8;  // 16-byte pieces per row
            for (int u = qt; u < kM * kPieces; u += 192) {
                const int m = u / kPieces, q = u % kPieces;
                const int c = q >> 3, j = q & 7;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (m < R) {
                    const size_t row = (size_t)(ri.row0 + m / G) * p.num_q_heads + kvh * G + (m % G);
                    val = *reinterpret_cast<const uint4*>(p.q + row * D + q * 8);
                }
                *reinterpret_cast<uint4*>(sQ + c * (kM * 128) + m * 128 + ((j ^ (m & 7)) << 4)) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aux->q_full);
        }
        if (warp >= 4) {
            // -------------------------------------------------------- softmax + epilogue
            const int wq = warp - 4;
            const int m = wq * 32 + lane;
            const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(wq * 32) << 16);
            const bool valid = m < R;
            const int i = valid ? m / G : 0;
            const int hq = kvh * G + (valid ? m % G : 0);
            const int qrow = ri.row0 + i;
            const int hi = (p.mask_mode == 0) ? (ri.ctx + i) : (ri.len - 1);
            const float sc = p.score_scale_log2;
            float m_ref = -INFINITY, l_sum = 0.f;
            long long tr_cnt = 0, tr_sum = 0;
            bool ok = true;
            for (int t = 0; t < T; ++t) {
                const int b = t & 1, s = t % S;
                if (!(ok = warp_wait(&aux->s_full[b], (t >> 1) & 1, abort))) break;
                tc_fence_after();
                float sv[64];
                {
                    float* lo = sv;
                    float* hi32 = sv + 32;
                    tmem_ld32(lane_tmem + D + b * kBN, *reinterpret_cast<float(*)[32]>(lo));
                    tmem_ld32(lane_tmem + D + b * kBN + 32, *reinterpret_cast<float(*)[32]>(hi32));
                }
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aux->s_empty[b]);

                const int key0 = key_lo + t * kBN;
                const int lim = valid ? (min(key_hi - 1, hi) - key0) : -1;  // visible iff c <= lim
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float x = (c <= lim) ? sv[c] * sc : -INFINITY;
                    sv[c] = x;
                    mx = fmaxf(mx, x);
                }
                const bool need = (m_ref != -INFINITY) && (mx > m_ref + kRescaleThreshold);
                const bool first = (m_ref == -INFINITY) && (mx != -INFINITY);
                const float ref = (need || first) ? mx : m_ref;
                const float alpha = need ? fast_exp2(m_ref - ref) : 1.f;
                uint32_t pk[32];
                float psum = 0.f;
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float p0 = (c <= lim) ? fast_exp2(sv[c] - ref) : 0.f;
                    const float p1 = (c + 1 <= lim) ? fast_exp2(sv[c + 1] - ref) : 0.f;
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    // the normaliser sums the fp32 weights: rounding P to bf16 for
                    // the PV MMA must not leak into l (and so into LSE) on rows
                    // that see only a few keys
                    psum += p0 + p1;
                    pk[c >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                l_sum = l_sum * alpha + psum;
                m_ref = ref;

                // P_t overwrites P_{t-1} and O may need rescaling: PV_{t-1} must be done.
                if (t > 0 && !(ok = warp_wait(&aux->o_done, (t - 1) & 1, abort))) break;
                if (__any_sync(kFullMask, need) && t > 0) {
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        float ov[32];
                        tmem_ld32(lane_tmem + ch * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                        tmem_st32(lane_tmem + ch * 32, ov);
                    }
                    tmem_wait_st();
                }
                // The request's last page may end mid-page: its stale slots hold
                // arbitrary (even non-finite) values and 0 * NaN is NaN, so zero them.
                const int np = min(4, (key_hi - key0 + 15) / 16);
                if (key_hi == ri.len && t == T - 1 && (ri.len & 15) != 0) {
                    if (!(ok = warp_wait(&aux->v_full[s], (t / S) & 1, abort))) break;
                    const int row_first = ri.len - key0, row_end = np * 16;
                    unsigned char* vt = sStage + s * L::kStageBytes + L::kTileBytes;
                    const int pieces = (row_end - row_first) * L::kChunks * 8;
                    for (int u = m; u < pieces; u += 128) {
                        const int rr = row_first + u / (L::kChunks * 8);
                        const int rem = u % (L::kChunks * 8);
                        const int c = rem >> 3, j = rem & 7;
                        *reinterpret_cast<uint4*>(vt + c * (kBN * 128) + rr * 128 + (j << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (TRACE) {
                    for (int c = 0; c <= lim && c < 64; ++c) {
                        const int key = key0 + c;
                        tr_cnt += 1;
                        tr_sum += (long long)aux->pages[s][c >> 4] * 16 + (key & 15);
                    }
                }
                // P row m into the 128-byte-swizzled K-major A tile
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(sP + m * 128 + ((j ^ (m & 7)) << 4)) =
                        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aux->p_full);
            }
            pdl_launch_dependents();
            if (ok) ok = warp_wait(&aux->o_done, (T - 1) & 1, abort);
            tc_fence_after();
            if (ok) {
                const float inv = (valid && l_sum > 0.f) ? (p.out_scale / l_sum) : 0.f;
                const float lse2 = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) : -INFINITY;
                const size_t oi = (size_t)qrow * p.num_q_heads + hq;
                const bool final_out = (ri.nsplits == 1);
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    float ov[32];
                    tmem_ld32(lane_tmem + ch * 32, ov);
                    tmem_wait_ld();
                    if (!valid) continue;
                    if (final_out) {
                        uint16_t* op = p.o + oi * D + ch * 32;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 =
                                    __floats2bfloat162_rn(ov[q4 * 8 + 2 * e] * inv, ov[q4 * 8 + 2 * e + 1] * inv);
                                w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                            }
                            *reinterpret_cast<uint4*>(op + q4 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float* wp = p.ws_o + ((size_t)split * p.total_rows * p.num_q_heads + oi) * D + ch * 32;
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            *reinterpret_cast<float4*>(wp + q4 * 4) =
                                make_float4(ov[q4 * 4] * inv, ov[q4 * 4 + 1] * inv, ov[q4 * 4 + 2] * inv,
                                            ov[q4 * 4 + 3] * inv);
                    }
                }
                if (valid) {
                    if (final_out) {
                        if (p.lse) p.lse[oi] = lse2 * kLn2;
                    } else {
                        p.ws_lse[(size_t)split * p.total_rows * p.num_q_heads + oi] = lse2;
                    }
                    if (TRACE && p.trace) {
                        unsigned long long* tp = reinterpret_cast<unsigned long long*>(p.trace + oi * 2);
                        atomicAdd(tp, (unsigned long long)tr_cnt);
                        atomicAdd(tp + 1, (unsigned long long)tr_sum);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

using TcKernel = void (*)(const SplitParams, const CUtensorMap, const CUtensorMap);

template <int D>
TcKernel pick_trace(bool traced) {
    return traced ? &split_attn_tc_kernel<D, true> : &split_attn_tc_kernel<D, false>;
}

TcKernel pick(int d, bool traced) {
    switch (d) {
        case 64: return pick_trace<64>(traced);
        case 128: return pick_trace<128>(traced);
        case 256: return pick_trace<256>(traced);
        default: return nullptr;
    }
}

int smem_for(int d) {
    switch (d) {
        case 64: return TcLayout<64>::kSmem;
        case 128: return TcLayout<128>::kSmem;
        case 256: return TcLayout<256>::kSmem;
        default: return 0;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Pool [num_pages, Hkv, 16, d] bf16 viewed as a 4-D tensor (d, slot, kv head, page);
// box = 64 head_dim elements x 16 slots of one page and head, 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int num_pages, int hkv, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * 16, (cuuint64_t)d * 2 * 16 * hkv};
    cuuint32_t box[4] = {64, 16, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(int head_dim, int kv_dtype, int max_rows) {
    return kv_dtype == 0 && max_rows <= kM && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

int tc_smem_bytes(int head_dim) { return smem_for(head_dim); }
int tc_threads() { return kTcThreads; }

cudaError_t tc_prepare(int head_dim) {
    for (int traced = 0; traced < 2; ++traced) {
        TcKernel k = pick(head_dim, traced != 0);
        if (!k) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_for(head_dim));
        if (e != cudaSuccess) return e;
    }
    return encode_fn() ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t tc_launch(const SplitParams& p, bool traced, dim3 grid, cudaStream_t stream) {
    TcKernel k = pick(p.head_dim, traced);
    if (!k) return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, p.k_pool, p.num_pages, p.num_kv_heads, p.head_dim) ||
        !encode_pool_map(&mv, p.v_pool, p.num_pages, p.num_kv_heads, p.head_dim))
        return cudaErrorInvalidValue;
    k<<<grid, kTcThreads, smem_for(p.head_dim), stream>>>(p, mk, mv);
    return cudaGetLastError();
}

}  // namespace spec_attn
