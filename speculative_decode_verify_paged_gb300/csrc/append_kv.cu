// KV append: the W_r new key and value rows of every request's window are
// written into their paged-cache slots before the window attends (page
// "perf(dflash): widen the verify window past the compact graph's four-row
// limit", section "What changed": the window's rows go into the cache, later
// steps overwrite the rows a rejection leaves stale, and attention reads only
// seq_len entries).  seq_len_r already counts the window, so window row i of
// request r is key ctx_r + i = seq_len_r - W_r + i: page
// block_table[r][pos / page_size], slot pos % page_size, for K, V and every
// KV head.
//
// bf16 caches take the bits as they are.  NVFP4 caches quantise each run of
// 16 head_dim elements against the tensor's decode scale g (one g per cache,
// so an append cannot re-derive it from a global maximum):
//   amax = max |x|,  scale = E4M3(amax / (6 g)),  den = scale * g,
//   code = den == 0 ? 0 : E2M1(x / den)
// each product and quotient in binary32 rounded to nearest even, the
// conversions to nearest even and saturating (cvt ... satfinite), codes two
// to a byte with the even element in the low nibble.
//
// Work layout: one thread per 8 bf16 elements (a 16-byte copy) or per
// 16-element NVFP4 block of one (window row, KV head, K or V); consecutive
// threads cover consecutive pieces of a row, so loads and stores coalesce.
// Grid: x over max_w * Hkv * 2 * pieces-per-row, y over requests.
//
// Ordering: the kernel is launched as a programmatic dependent of whatever
// precedes it in the stream and waits on griddepcontrol before its first
// global access (an earlier attention call may still be reading the slots it
// overwrites).  It then lets the next kernel -- the split-KV attention, which
// itself waits on griddepcontrol before touching the cache -- launch at once,
// so that kernel's CTA setup overlaps this one.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec_attn {
namespace {

constexpr int kAppendThreads = 256;

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global_v2(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// binary32 -> E4M3 byte, nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float x) {
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x), "f"(x));
    return d & 0xFFu;
}

// Four pairs (t[2k] even element, t[2k+1] odd) -> four E2M1 code bytes, the
// even element in each low nibble; nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(const float (&t)[8]) {
    uint32_t d;
    asm("{ .reg .b8 c0, c1, c2, c3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"   // first operand -> high nibble
        "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
        "mov.b32 %0, {c0, c1, c2, c3}; }"
        : "=r"(d)
        : "f"(t[0]), "f"(t[1]), "f"(t[2]), "f"(t[3]), "f"(t[4]), "f"(t[5]), "f"(t[6]), "f"(t[7]));
    return d;
}

template <int D, bool FP4>
__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const AppendParams p) {
    constexpr int kUnit = FP4 ? 16 : 8;     // elements per thread
    constexpr int kPieces = D / kUnit;      // per (row, KV head)
    pdl_wait_primary();
    pdl_launch_dependents();
    const int r = blockIdx.y;
    const int idx = blockIdx.x * kAppendThreads + threadIdx.x;
    ReqInfo ri;
    // one thread per CTA reports a bad window or length
    if (!load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len, p.bt_capacity_keys,
                      p.page_size, threadIdx.x == 0 ? p.status : nullptr, ri))
        return;
    const int piece = idx % kPieces;
    int t = idx / kPieces;
    const int is_v = t & 1;
    t >>= 1;
    const int h = t % p.num_kv_heads;
    const int i = t / p.num_kv_heads;
    if (i >= ri.w) return;
    const int pos = ri.ctx + i;
    // the new row and the block-table entry are independent: one memory round trip
    const uint16_t* src = (is_v ? p.v_new : p.k_new) + ((size_t)(ri.row0 + i) * p.num_kv_heads + h) * D +
                          piece * kUnit;
    const uint4 a = ld_global_nc_v4(src);
    uint4 b = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (FP4) b = ld_global_nc_v4(src + 8);
    const int page = p.block_table[(size_t)r * p.bt_stride + pos / p.page_size];
    if (page < 0 || page >= p.num_pages) {
        atomicOr(p.status, kDevBadPage);
        return;
    }
    // the destination row within its page: KV head h, slot pos % page_size
    const size_t slot = (size_t)h * p.page_size + (pos % p.page_size);
    if constexpr (!FP4) {
        unsigned char* dst = static_cast<unsigned char*>(is_v ? p.v_pool : p.k_pool) +
                             (size_t)page * p.kv_page_stride + slot * (D * 2) + piece * (kUnit * 2);
        sm100::st_global_v4(dst, a);
    } else {
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float x[16];
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            amax = fmaxf(amax, fmaxf(fabsf(x[2 * k]), fabsf(x[2 * k + 1])));
        }
        const float g = is_v ? p.v_gscale : p.k_gscale;
        const uint32_t sb = e4m3_rn_sat(__fdiv_rn(amax, __fmul_rn(6.0f, g)));
        const float den = __fmul_rn(e4m3_to_float(sb), g);
        uint32_t c0 = 0u, c1 = 0u;
        if (den != 0.f) {
            float t0[8], t1[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                t0[e] = __fdiv_rn(x[e], den);
                t1[e] = __fdiv_rn(x[8 + e], den);
            }
            c0 = e2m1x8_rn_sat(t0);
            c1 = e2m1x8_rn_sat(t1);
        }
        uint8_t* codes = static_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool) + (size_t)page * p.kv_page_stride +
                         slot * (D / 2) + piece * 8;
        uint8_t* scales = (is_v ? p.v_scales : p.k_scales) + (size_t)page * p.scale_page_stride + slot * (D / 16) +
                          piece;
        st_global_v2(codes, c0, c1);
        *scales = static_cast<uint8_t>(sb);
    }
}

template <int D>
cudaError_t launch_d(const AppendParams& p, bool fp4, cudaStream_t stream) {
    const int pieces = fp4 ? D / 16 : D / 8;
    const long long threads = (long long)p.max_w * p.num_kv_heads * 2 * pieces;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((threads + kAppendThreads - 1) / kAppendThreads),
                       static_cast<unsigned>(p.num_reqs), 1);
    cfg.blockDim = dim3(kAppendThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return fp4 ? cudaLaunchKernelEx(&cfg, &append_kv_kernel<D, true>, p)
               : cudaLaunchKernelEx(&cfg, &append_kv_kernel<D, false>, p);
}

}  // namespace

cudaError_t append_launch(const AppendParams& p, int kv_dtype, cudaStream_t stream) {
    const bool fp4 = kv_dtype != 0;
    switch (p.head_dim) {
        case 64: return launch_d<64>(p, fp4, stream);
        case 128: return launch_d<128>(p, fp4, stream);
        case 256: return launch_d<256>(p, fp4, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace spec_attn
