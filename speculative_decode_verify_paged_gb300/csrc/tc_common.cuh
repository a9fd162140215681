// Device helpers of the tensor-core split kernel (split_attn_tc.cu): bounded
// mbarrier waits, the block-table load, NVFP4 decode by the hardware converts,
// and the drain of copies in flight.
#pragma once

#include <limits.h>
#include <stdint.h>

#include <cuda_fp16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec_attn {
namespace tcc {

using namespace sm100;

// A 32-bit global load the compiler keeps in program order (not sunk past later loads).
__device__ __forceinline__ int ld_volatile_i32(const int32_t* p) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM cycles
constexpr long long kDrainLimit = 200000000LL;
constexpr int kPageListCap = 64;                 // page ids staged in shared memory at a time (2 per lane)
constexpr int kNoPrefetch = INT_MIN;             // the producer fetches its first page ids itself

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

// Position of 16-byte code chunk ch (of D / 32) within key sl's row of a page's
// codes in the raw ring.  The TMA copies them with the 128/64/32-byte swizzle
// of d = 256/128/64 (16-byte chunk index XOR address bits 7..9), which places
// one chunk of 8 consecutive keys in 8 different 16-byte bank groups.
template <int D>
__device__ __forceinline__ int raw_code_chunk(int sl, int ch) {
    return D == 256 ? (ch ^ (sl & 7)) : D == 128 ? (ch ^ ((sl >> 1) & 3)) : (ch ^ ((sl >> 2) & 1));
}

// Decode of NVFP4 K/V into fp16 MMA operands.  cvt.rn.f16x2.e2m1x2 turns one
// code byte (two e2m1 values, the low nibble into the low half) into an fp16
// pair and cvt.rn.f16x2.e4m3x2 one scale byte into (s, s); the products (at most
// 5 significant bits, magnitudes 2^-10 .. 2688) are exact in fp16.
__device__ __forceinline__ uint32_t e4m3_pair_f16x2(uint32_t byte) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(byte * 0x0101u)));
    return d;
}
// 8 e2m1 codes (one 32-bit word) times the fp16 scale pair s2, as 4 fp16 pairs.
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t s2, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                           uint32_t& o3) {
    uint32_t a0, a1, a2, a3;
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4; "
        "cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1; "
        "cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
        : "r"(w));
    const __half2 s = *reinterpret_cast<const __half2*>(&s2);
    __half2 h;
    h = __hmul2(*reinterpret_cast<const __half2*>(&a0), s); o0 = *reinterpret_cast<const uint32_t*>(&h);
    h = __hmul2(*reinterpret_cast<const __half2*>(&a1), s); o1 = *reinterpret_cast<const uint32_t*>(&h);
    h = __hmul2(*reinterpret_cast<const __half2*>(&a2), s); o2 = *reinterpret_cast<const uint32_t*>(&h);
    h = __hmul2(*reinterpret_cast<const __half2*>(&a3), s); o3 = *reinterpret_cast<const uint32_t*>(&h);
}

template <int NSLOT>
__device__ __forceinline__ void drain_copies(uint64_t* full, int issued) {
    // let every copy still in flight land before the CTA's shared memory goes away
    for (int t = max(0, issued - NSLOT); t < issued; ++t) {
        volatile int no_abort = 0;
        mbar_wait(&full[t % NSLOT], (t / NSLOT) & 1, &no_abort, kDrainLimit);
    }
}

}  // namespace tcc
}  // namespace spec_attn
