// Split-KV block attention on 5th-generation tensor cores (tcgen05 + TMEM),
// bf16 or NVFP4 KV, for sm_103a.
//
// One CTA = (split s of request r's keys) x (KV head kvh).  Its query tile is
// all W x G rows of the request that read KV head kvh (row m = window row
// m / G, query head kvh * G + m % G), padded to the MMA's M = 128, so every
// K/V page of the split is streamed from HBM exactly once whatever W is
// (above 128 rows per KV head, in row groups of whole window rows, one CTA
// each; the template flag RG marks such launches) --
// the single sweep per window that the page "ChunkedSmallT re-streams full
// KV per query chunk (DFlash K>=8 verify at long context)" (section
// "Finding") finds missing for W > 8.  No output is produced for context
// rows (page "DFlash2 leaves the paged graph fast path at every c>1 ...",
// section "The cost").
//
// Warp roles, bf16 KV (256 threads):
//   warp 0      loads the query tile once (one TMA box: every 64-element
//               chunk of G heads x the group's window rows, into the V
//               slots), then streams the K tiles: 64 keys (four 16-key units,
//               a unit being a 16-key page or a quarter/half of a 64/32-key
//               page; one 2 KB box per unit and 64 head_dim elements, issued
//               from 16 lanes), 128-byte swizzled, chunk-major, into a ring.
//   warp 2      streams the V tiles into a second ring, one box per unit of a
//               page-head, once the query tile has left the V slots.
//   warp 1      allocates TMEM and issues S_t = Q K_t^T (M 128, N 64, query
//               tile from TMEM, -> fp32 in TMEM, double-buffered).
//   warp 3      issues O += P_t V_t (M 128, N head_dim, one MMA per unit, P
//               from TMEM, V MN-major), then frees the S buffer P sat in.  Each
//               issuer waits only on its own inputs, in tile order.
//   warps 4-7   softmax: thread m owns row m (TMEM lane m).  First it moves its
//               query row into TMEM.  Per tile it reads its 64 scores, applies
//               the causal-in-block / non-causal mask and the sliding window
//               by key index (rows past W x G run unmasked), updates a
//               base-2 online softmax whose reference maximum moves only when a
//               score exceeds it by more than 2^8 (then the row of O in TMEM is
//               rescaled), and writes P (16-bit) over the first half of its S
//               buffer in TMEM.  At the end a request finished by this split
//               has its rows normalised, staged and copied out by every warp;
//               a split partial goes straight from TMEM to global memory
//               (warps 0-7, chunk-major fp16 of O / its row maximum).
//   (multi-request batches of uneven lengths: the grid is one-dimensional,
//   each block taking the next existing (request, split, KV head, row group)
//   unit, so the CTAs with work come first in launch order)
// With the dense block operand, the request's last split ends with one more
// tile: the window's own keys, one unit loaded from the block tensors.
// NVFP4 KV (512 threads): warp 0 streams the tiles' codes and scales by TMA
// into a raw ring; warps 8-11 decode K and 12-15 decode V into fp16 operand
// tiles; the query row is converted to fp16 on its way into TMEM, and P is
// fp16; the rest as for bf16.
//
// Every wait on an mbarrier is bounded: on time-out the CTA raises the
// device-status bit, stops issuing, drains its in-flight copies and MMAs,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace spec_attn {

namespace {

using namespace sm100;
using namespace tcc;

constexpr int kBN = 64;        // keys per tile (a multiple of the 16-key unit; 32 or 64)
constexpr int kPPT = kBN / 16;  // pages per tile
static_assert(kBN == 32 || kBN == 64, "tile");
constexpr int kM = 128;        // MMA rows (query tile, padded)
constexpr int kTcThreadsBf16 = 256;   // warps 0-7
constexpr int kTcThreadsFp4 = 512;    // + warps 8-11 (K dequant) and 12-15 (V dequant)
constexpr float kRescaleThreshold = 8.0f;        // log2 units: rescale when max grows by > 2^8
constexpr int kMaxNR = 8;                        // NVFP4 raw (codes + scales) ring slots
constexpr int kMaxNK = 8, kMaxNV = 16;

// Shared memory: K ring | V ring | [NVFP4 raw ring] | barriers.
// The query tile lands (bf16, by TMA) in the V slots before any V does; the
// softmax warps move it into TMEM (NVFP4: converted to fp16), where the
// S = Q K^T MMA reads its A operand.  An MMA with its A operand in TMEM issues
// at about twice the rate of one reading it from shared memory, and the
// 128-row tile costs no shared memory or shared-memory bandwidth.  P goes to
// TMEM as well, where the P V MMA reads it as its A operand: P (16-bit) takes
// the first half of the S buffer it was computed from, and S is double
// buffered, so the S MMA of tile t + 1 runs while the softmax works on tile t.
// bf16 KV: K and V arrive by TMA into rings of kNK / kNV slots.  The CTA keeps
// below 200 KB of shared memory, so that a CTA of the kernel that follows in
// the stream (the LSE merge: 10 KB) can become resident beside it.
// NVFP4 KV: codes and scales arrive by TMA into a ring of kNR raw slots and are
// decoded into fp16 K and V operand tiles (two slots each).
// NVFP4 raw slot: the codes and scales of a tile's 16-key units, K then V.
// Every TMA tile copy lands on a 128-byte boundary (the tensor copy's
// shared-memory alignment), so a unit's scales (d bytes: 64 at d = 64) take at
// least 128.
template <int D>
struct RawLayout {
    static constexpr int kCodePage = 16 * D / 2;           // codes of one 16-key unit
    static constexpr int kScaleBox = 16 * D / 16;          // scales of one unit (bytes copied)
    static constexpr int kScalePage = kScaleBox < 128 ? 128 : kScaleBox;   // their spacing
    static constexpr int kKS = kPPT * kCodePage;           // offsets inside a raw slot
    static constexpr int kVC = kKS + kPPT * kScalePage;
    static constexpr int kVS = kVC + kPPT * kCodePage;
    static constexpr int kTile = 2 * kPPT * (kCodePage + kScalePage);
    static_assert(kCodePage % 128 == 0 && kScalePage % 128 == 0, "TMA destinations on 128 B");
};

template <int D, int KV>
struct TcLayout {
    static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along head_dim
    static constexpr int kQBytes = kM * D * 2;             // the query tile (16-bit elements)
    static constexpr int kQSmem = 0;                       // no region of its own: it lands in the V slots
    static constexpr int kPBytes = 0;                      // P lives in TMEM
    static constexpr int kTileBytes = kBN * D * 2;         // one K or V tile (16-bit elements)
    static constexpr int kPageBytes = 16 * D * 2;          // one 16-key unit of V (16-bit elements)
    static constexpr int kRawTile = RawLayout<D>::kTile;   // one NVFP4 raw slot
    static constexpr int kAuxBytes = 1664;
    static constexpr int kMaxDyn = KV ? 232448 : 204800;    // 227 KB opt-in limit; bf16: 200 KB
    static constexpr int kFixed = 1024 + kQSmem + kPBytes + kAuxBytes;
    static constexpr int kRing = (kMaxDyn - kFixed) / kTileBytes;
    // bf16: the ring is split evenly: every tile needs its K and its V, and
    // loads land in about the order they are issued, so a V ring running far
    // ahead of a short K ring only delays the K tiles the next S waits for.
    static constexpr int kNK = KV ? 2 : ((kRing / 2) > kMaxNK ? kMaxNK : ((kRing / 2) < 2 ? 2 : (kRing / 2)));
    static constexpr int kNV = KV ? 2 : ((kRing - kNK) > kMaxNV ? kMaxNV : (kRing - kNK));
    static constexpr int kRawFit = (kMaxDyn - kFixed - (kNK + kNV) * kTileBytes) / kRawTile;
    static constexpr int kNR = KV ? (kRawFit > kMaxNR ? kMaxNR : kRawFit) : 0;
    static constexpr int kSmem = kFixed + (kNK + kNV) * kTileBytes + kNR * kRawTile;
    // TMEM columns: O [0, D), S double buffer [D, D + 2 BN) with P_b (16-bit
    // pairs: bf16, NVFP4 fp16) in the first BN / 2 columns of S buffer b, query
    // tile (16-bit pairs) [D + 2 BN, D + 2 BN + D / 2).
    static constexpr int kSBufs = 2;
    __host__ __device__ static constexpr int p_col(int b) { return D + b * kBN; }
    static constexpr int kQCol = D + 2 * kBN;
    static constexpr int kTmemNeed = D + 2 * kBN + D / 2;
    static constexpr uint32_t kTmemCols = kTmemNeed <= 128 ? 128u : (kTmemNeed <= 256 ? 256u : 512u);
    static_assert(KV ? (kNR >= 2) : (kNK >= 2 && kNV >= 2), "ring too small");
    static_assert(kSmem <= kMaxDyn, "shared memory");
    static_assert(kTmemNeed <= 512, "tensor memory");
    static_assert(kQBytes <= kNV * kTileBytes, "the query tile lands in the V slots");
    // With early_context_kv it lands in the last V slots instead, so that the
    // first V tile may be copied while it is still there (only the first: more
    // V copies ahead of the query tile would delay it, and the first scores
    // wait for it).
    static constexpr int kQOff = kNV * kTileBytes - kQBytes;
    static_assert(KV || kQOff >= kTileBytes, "a V slot free of the query tile (bf16)");
    static_assert(kQOff % 1024 == 0, "the query tile's box lands on 1024-byte swizzle atoms");
    // the final-output epilogue stages kM rows of bf16 O (+16 B padding), the
    // partials epilogue 3 x kM floats, over the operand/raw buffers (idle by then)
    static_assert(kM * (D * 2 + 16) <= (kNK + kNV) * kTileBytes + kNR * kRawTile, "epilogue staging");
};

struct TcAux {
    uint64_t k_full[kMaxNK];
    uint64_t k_empty[kMaxNK];
    uint64_t v_full[kMaxNV];
    uint64_t v_empty[kMaxNV];
    uint64_t s_full[2];
    uint64_t s_empty[2];   // the P V of the buffer's tile has read its P (committed by the MMA)
    uint64_t p_full[2];
    uint64_t o_done;     // one phase per P V (rescale waits: at most one phase behind)
    uint64_t o_final;    // one phase after the last P V (the epilogue's wait)
    uint64_t q_full;     // the query tile landed in the V slots (TMA bytes)
    uint64_t q_ready;    // the query tile moved into TMEM (NVFP4: as fp16), its V slots free
                         // (one arrival per softmax warp)
    uint64_t drain;
    uint64_t drain_pv;   // the P V issuer's own MMAs
    uint64_t raw_full[kMaxNR];             // NVFP4: codes/scales of a tile landed (32 lane arrivals)
    uint64_t raw_empty[kMaxNR];            // NVFP4: both dequant warpgroups are done with a raw slot
    int32_t pages_v[kMaxNV][kPPT];         // physical pages of each V slot (index trace)
    int32_t raw_pages[kMaxNR][kPPT];       // NVFP4: physical pages of each raw slot
    uint32_t tmem_base;
    int abort;
    int32_t list_k[kPageListCap];          // the split's page ids, one list per producer
    int32_t list_v[kPageListCap];
    int32_t item[4];                       // compact block order: request (-1: none), split, KV head, row group
    ReqInfo item_ri;                       // and that request's metadata
};
static_assert(sizeof(TcAux) <= TcLayout<64, 0>::kAuxBytes, "aux region");

// One producer warp streams one of K or V: block-table entries are fetched by
// all 32 lanes at once (coalesced) into a shared-memory list, then lane 0
// issues one 2 KB TMA box per (page, 64 head_dim elements) into the ring slot.
// With the dense block operand, tile Tc (the last of the request's last
// split) holds the window's own keys: one 16-key unit of rows row0 .. row0 + 15
// of the block tensor (tm_block), laid out like a page unit.
// V: the slots from q_gate on hold the query tile until it is in TMEM, so the
// producer waits for that before it first fills one.  after_first() runs once
// the first tile's copies are issued (or, if the loop stops before, at its end).
template <int D, int NSLOT, bool IS_V, bool TRACE, class F>
__device__ __forceinline__ int produce(const SplitParams& p, int r, int kvh, int key_lo, int key_hi, int T,
                                       unsigned char* ring, uint64_t* full, uint64_t* empty, int32_t* list,
                                       TcAux* aux, const CUtensorMap* tm, volatile int* abort, int lane,
                                       int pre0, int pre1, int Tc, int row0, const CUtensorMap* tm_block,
                                       int q_gate, const F& after_first) {
    using L = TcLayout<D, 0>;
    const int32_t* bt = p.block_table + (size_t)r * p.bt_stride;
    const int u_lo = key_lo / 16;                    // first 16-key unit of the split
    const int n_pages = (key_hi - key_lo + 15) / 16;  // 16-key units
    const int sub_mask = (1 << p.page_shift) - 1;
    int list_base = 0;
    // list entries are 16-key units: (page << page_shift) | unit within the page
    auto unit = [&](int pg, int u) {
        if (pg < 0 || pg >= p.num_pages) {
            if (!IS_V) atomicOr(p.status, kDevBadPage);
            pg = 0;
        }
        return (pg << p.page_shift) | (u & sub_mask);
    };
    auto fill_list = [&](int base) {
        for (int i = lane; i < kPageListCap && base + i < n_pages; i += 32) {
            const int u = u_lo + base + i;
            list[i] = unit(bt[u >> p.page_shift], u);
        }
        __syncwarp();
    };
    // the first 64 entries were fetched by the caller (unless it could not know where)
    if (pre0 == kNoPrefetch) {
        fill_list(0);
    } else {
        if (lane < n_pages) list[lane] = unit(pre0, u_lo + lane);
        if (lane + 32 < n_pages) list[lane + 32] = unit(pre1, u_lo + lane + 32);
        __syncwarp();
    }
    int issued = 0;
    for (int t = 0; t < T; ++t) {
        const int slot = t % NSLOT;
        if (t >= NSLOT && !warp_wait(&empty[slot], ((t / NSLOT) - 1) & 1, abort)) break;
        if (IS_V && t == q_gate && !warp_wait(&aux->q_ready, 0, abort)) break;
        unsigned char* dst = ring + slot * L::kTileBytes;
        if (t >= Tc) {   // the dense block unit
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(L::kChunks * 2048));
            __syncwarp();
            if (IS_V) {
                if (lane == 0) tma_load_4d(dst, tm_block, 0, row0, 0, kvh, &full[slot]);
            } else if (lane < L::kChunks) {
                tma_load_3d(dst + lane * (kBN * 128), tm_block, lane * 64, row0, kvh, &full[slot]);
            }
            __syncwarp();
            issued = t + 1;
            if (t == 0) after_first();
            continue;
        }
        const int rel = t * kPPT;  // first page of the tile, relative to the split
        if (rel >= list_base + kPageListCap) {
            __syncwarp();
            list_base = rel;
            fill_list(list_base);
        }
        // The copies of a tile are issued by several lanes at once (a copy's
        // issue takes a while; one lane issuing them all in turn would add
        // that time to every tile's latency).
        const int np = min(kPPT, (key_hi - (key_lo + t * kBN) + 15) / 16);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(np * L::kChunks * 2048));
        __syncwarp();
        if (IS_V) {
            // lane pp: all of unit pp in one copy, [chunk][16 slots][128 B]
            if (lane < np) {
                const int pg = list[rel - list_base + lane];
                if (TRACE) aux->pages_v[slot][lane] = pg;
                tma_load_5d(dst + lane * L::kPageBytes, tm, 0, (pg & sub_mask) * 16, 0, kvh, pg >> p.page_shift,
                            &full[slot]);
            }
        } else if (lane < np * L::kChunks) {
            // lane (pp, c): chunk c of unit pp, chunk-major across the tile's
            // units so that S = Q K^T spans the tile in one MMA
            const int pp = lane / L::kChunks, c = lane % L::kChunks;
            const int pg = list[rel - list_base + pp];
            tma_load_4d(dst + c * (kBN * 128) + pp * 2048, tm, c * 64, (pg & sub_mask) * 16, kvh,
                        pg >> p.page_shift, &full[slot]);
        }
        __syncwarp();
        issued = t + 1;
        if (t == 0) after_first();
    }
    if (issued == 0) after_first();
    return issued;
}

// NVFP4: one warp streams each tile's e2m1 codes and e4m3 scales, K and V, into
// a raw ring slot by TMA: per 16-key unit one box of codes (16 keys x d/2
// bytes, swizzled) and one of scales (d bytes), issued from 4 lanes per unit.
template <int D>
__device__ __forceinline__ int produce_raw(const SplitParams& p, int r, int kvh, int key_lo, int key_hi, int T,
                                           unsigned char* raw, TcAux* aux, const CUtensorMap* tkc,
                                           const CUtensorMap* tvc, const CUtensorMap* tks, const CUtensorMap* tvs,
                                           volatile int* abort, int lane, int pre0, int pre1) {
    using L = TcLayout<D, 1>;
    using RL = RawLayout<D>;
    constexpr int NR = L::kNR;
    const int32_t* bt = p.block_table + (size_t)r * p.bt_stride;
    const int u_lo = key_lo / 16;
    const int n_pages = (key_hi - key_lo + 15) / 16;   // 16-key units
    const int sub_mask = (1 << p.page_shift) - 1;
    int32_t* list = aux->list_k;
    int list_base = 0;
    auto unit = [&](int pg, int u) {
        if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.status, kDevBadPage);
            pg = 0;
        }
        return (pg << p.page_shift) | (u & sub_mask);
    };
    auto fill_list = [&](int base) {
        for (int i = lane; i < kPageListCap && base + i < n_pages; i += 32) {
            const int u = u_lo + base + i;
            list[i] = unit(bt[u >> p.page_shift], u);
        }
        __syncwarp();
    };
    // the first 64 entries were fetched by the caller (unless it could not know where)
    if (pre0 == kNoPrefetch) {
        fill_list(0);
    } else {
        if (lane < n_pages) list[lane] = unit(pre0, u_lo + lane);
        if (lane + 32 < n_pages) list[lane + 32] = unit(pre1, u_lo + lane + 32);
        __syncwarp();
    }
    int issued = 0;
    for (int t = 0; t < T; ++t) {
        const int slot = t % NR;
        if (t >= NR && !warp_wait(&aux->raw_empty[slot], ((t / NR) - 1) & 1, abort)) break;
        const int rel = t * kPPT;
        if (rel >= list_base + kPageListCap) {
            __syncwarp();
            list_base = rel;
            fill_list(list_base);
        }
        const int np = min(kPPT, (key_hi - (key_lo + t * kBN) + 15) / 16);
        unsigned char* dst = raw + slot * RL::kTile;
        // the slot's page ids (index trace) are published by the arrival below
        if (lane < np) aux->raw_pages[slot][lane] = list[rel - list_base + lane];
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(&aux->raw_full[slot],
                                  static_cast<uint32_t>(np * 2 * (RL::kCodePage + RL::kScaleBox)));
        __syncwarp();
        if (lane < 4 * np) {
            const int pp = lane >> 2, kind = lane & 3;
            const int pg = list[rel - list_base + pp];
            const int page = pg >> p.page_shift, sub = pg & sub_mask;
            uint64_t* bar = &aux->raw_full[slot];
            if (kind == 0) tma_load_4d(dst + pp * RL::kCodePage, tkc, 0, sub * 16, kvh, page, bar);
            else if (kind == 1) tma_load_4d(dst + RL::kVC + pp * RL::kCodePage, tvc, 0, sub * 16, kvh, page, bar);
            else if (kind == 2) tma_load_3d(dst + RL::kKS + pp * RL::kScalePage, tks, sub * D, kvh, page, bar);
            else tma_load_3d(dst + RL::kVS + pp * RL::kScalePage, tvs, sub * D, kvh, page, bar);
        }
        __syncwarp();
        issued = t + 1;
    }
    return issued;
}

// One dequant warpgroup (128 threads) decodes the K (IS_V false) or V codes of
// each tile from the raw ring into the fp16 operand tile the MMA reads: K
// chunk-major across the tile's keys, V page by page, 128-byte swizzled like
// the TMA-loaded bf16 tiles.  A unit is one key's 64-element chunk (32 code
// bytes, 4 scales, one 128-byte swizzle row of the tile); eight consecutive
// keys of one chunk run side by side, so the row stores hit distinct banks.
// Keys at or past key_hi are written as zeros.
template <int D, bool IS_V, bool TRACE>
__device__ __forceinline__ void dequant(const SplitParams& p, int key_lo, int key_hi, int T, const unsigned char* raw,
                                        unsigned char* tile_ring, TcAux* aux, volatile int* abort, int dt) {
    using L = TcLayout<D, 1>;
    using RL = RawLayout<D>;
    constexpr int NR = L::kNR;
    constexpr int NS = IS_V ? L::kNV : L::kNK;   // operand tile slots
    constexpr int CPK = D / 64;                  // 64-element chunks per key
    constexpr int kUnits = kBN * CPK;
    const int lane = dt & 31;
    uint64_t* full = IS_V ? aux->v_full : aux->k_full;
    uint64_t* empty = IS_V ? aux->v_empty : aux->k_empty;
    // the query tile lands in the V slots: they are free once it is in TMEM
    if (IS_V && !warp_wait(&aux->q_ready, 0, abort)) return;
    for (int t = 0; t < T; ++t) {
        const int slot = t % NR, ts = t % NS;
        if (!warp_wait(&aux->raw_full[slot], (t / NR) & 1, abort)) break;
        if (t >= NS && !warp_wait(&empty[ts], ((t / NS) - 1) & 1, abort)) break;
        const int nvalid = key_hi - (key_lo + t * kBN);
        const unsigned char* src = raw + slot * RL::kTile;
        const unsigned char* codes = src + (IS_V ? RL::kVC : 0);
        const unsigned char* scales = src + (IS_V ? RL::kVS : RL::kKS);
        unsigned char* tile = tile_ring + ts * L::kTileBytes;
        for (int u = dt; u < kUnits; u += 128) {
            // u -> (group of 8 keys, chunk c, key within the group)
            const int j = (u / (8 * CPK)) * 8 + (u & 7);
            const int c = (u >> 3) % CPK;
            const int pg = j >> 4, sl = j & 15;
            uint4 outp[8];
            if (j < nvalid) {
                const unsigned char* kr = codes + pg * RL::kCodePage + sl * (D / 2);
                const uint4 w0 = *reinterpret_cast<const uint4*>(kr + raw_code_chunk<D>(sl, 2 * c) * 16);
                const uint4 w1 = *reinterpret_cast<const uint4*>(kr + raw_code_chunk<D>(sl, 2 * c + 1) * 16);
                const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(scales + pg * RL::kScalePage +
                                                                        sl * (D / 16) + c * 4);
                const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    // word q holds elements 8q .. 8q + 7 of the chunk; block scale q / 2
                    const uint32_t s2 = e4m3_pair_f16x2((sc4 >> (8 * (q >> 1))) & 0xFFu);
                    e2m1x8_f16(words[q], s2, outp[q].x, outp[q].y, outp[q].z, outp[q].w);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) outp[q] = make_uint4(0u, 0u, 0u, 0u);
            }
            unsigned char* row = IS_V ? tile + pg * L::kPageBytes + c * 2048 + sl * 128
                                      : tile + c * (kBN * 128) + j * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(row + ((q ^ (j & 7)) << 4)) = outp[q];
        }
        if (TRACE && IS_V && dt < kPPT) aux->pages_v[ts][dt] = aux->raw_pages[slot][dt];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&full[ts]);
            mbar_arrive(&aux->raw_empty[slot]);
        }
    }
}

// Compact block order (p.compact): block L of a one-dimensional grid takes the
// L-th unit of work -- (request, split, KV head, row group), requests in
// order, and within one split-major, then KV head, then row group -- counting
// only the splits and row groups each request's length and window give it.
// Blocks past the last unit have none.  The blocks with work thus come first
// in launch order, so in a batch of uneven lengths they all start in the
// first wave, instead of waiting behind the blocks of short requests' missing
// splits that the (splits x KV heads x requests) grid lays out for the longest.
// One warp: requests in chunks of 32, one lane each (their metadata in one
// memory round trip a chunk), and a warp scan of the unit counts.  Writes
// the unit and its request's metadata to item / item_ri.  Block 0 reports
// the device status of requests with bad lengths or windows (which get no
// work).
template <bool RG>
__device__ __forceinline__ void compact_item(const SplitParams& p, TcAux* aux, int lane) {
    const int L = blockIdx.x;
    int base = 0;
    int found = 0;
    // (block 0 scans every request, for the status report)
    for (int r0 = 0; r0 < p.num_reqs && (!found || L == 0); r0 += 32) {
        const int r = r0 + lane;
        ReqInfo ri;
        int cnt = 0, groups = 1;
        if (r < p.num_reqs &&
            load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                         p.bt_stride << (4 + p.page_shift), p.keys_per_split, blockIdx.x == 0 ? p.status : nullptr,
                         ri, p.window_left, p.split_align, p.dense_block)) {
            groups = RG ? (ri.w + p.window_rows_per_cta - 1) / p.window_rows_per_cta : 1;
            cnt = ri.nsplits * p.num_kv_heads * groups;
        }
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFullMask, inc, o);
            if (lane >= o) inc += v;
        }
        const int lo = base + inc - cnt;
        const bool mine = cnt > 0 && L >= lo && L < base + inc;
        if (mine) {
            const int local = L - lo;
            aux->item[0] = r;
            aux->item[1] = local / (groups * p.num_kv_heads);
            aux->item[2] = (local / groups) % p.num_kv_heads;
            aux->item[3] = local % groups;
            aux->item_ri = ri;
        }
        found |= __any_sync(kFullMask, mine);
        base += __shfl_sync(kFullMask, inc, 31);
    }
    if (!found && lane == 0) aux->item[0] = -1;
}

template <int D, int KV, bool TRACE, bool RG>
__global__ void __launch_bounds__(KV ? kTcThreadsFp4 : kTcThreadsBf16, 1)
split_attn_tc_kernel(const SplitParams p, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmks, const __grid_constant__ CUtensorMap tmvs) {
    using L = TcLayout<D, KV>;
    constexpr int NK = L::kNK, NV = L::kNV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // RG: blockIdx.x = split x row groups.  A row group is up to 128 / G whole
    // window rows (all G heads of each), so windows of more than 128 rows per KV
    // head take several CTAs, each streaming the split's K/V once.  Without RG
    // (one group) the row offsets below are compile-time zeros.
    // (compact block order: replaced below by the block's unit of work)
    int rg = RG ? blockIdx.x % p.row_groups : 0;
    int split = RG ? blockIdx.x / p.row_groups : blockIdx.x;
    int kvh = blockIdx.y, r = blockIdx.z;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sK = smem + L::kQSmem;
    unsigned char* sV = sK + NK * L::kTileBytes;
    // early_context_kv (bf16, no sliding window, no dense block operand): the K
    // and V producers issue each split's first tile, if it holds context keys
    // only, before the programmatic wait; the query tile then lands in the last
    // V slots (it is issued after the wait), so the first V tile need not wait
    // for it to move to TMEM
    const bool early_kv = !KV && p.early_context_kv && p.early_metadata && p.window_left == 0 && !p.dense_block;
    // the query tile lands in the V slots, then moves to TMEM
    unsigned char* sQ = sV + (early_kv ? L::kQOff : 0);
    unsigned char* sRaw = sV + NV * L::kTileBytes;   // NVFP4 only
    TcAux* aux = reinterpret_cast<TcAux*>(sRaw + L::kNR * L::kRawTile);
    volatile int* abort = &aux->abort;

    if (tid == 0) {
        // bf16: a full barrier completes on its TMA bytes (one expect_tx arrival);
        // NVFP4: on the four warps of the dequant warpgroup
        for (int s = 0; s < NK; ++s) {
            mbar_init(&aux->k_full[s], KV ? 4 : 1);
            mbar_init(&aux->k_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&aux->v_full[s], KV ? 4 : 1);
            mbar_init(&aux->v_empty[s], 1);
        }
        for (int s = 0; s < L::kNR; ++s) {
            mbar_init(&aux->raw_full[s], 1);
            mbar_init(&aux->raw_empty[s], 8);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&aux->s_full[b], 1);
            mbar_init(&aux->s_empty[b], 1);
            mbar_init(&aux->p_full[b], 4);
        }
        mbar_init(&aux->o_done, 1);
        mbar_init(&aux->o_final, 1);
        mbar_init(&aux->q_full, 1);
        mbar_init(&aux->q_ready, 4);
        mbar_init(&aux->drain, 1);
        mbar_init(&aux->drain_pv, 1);
        aux->abort = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        if (KV) {
            tma_prefetch_desc(&tmks);
            tma_prefetch_desc(&tmvs);
        }
    }
    if (warp == 1) tmem_alloc(&aux->tmem_base, L::kTmemCols);
    if (p.compact && warp == 3) {
        if (!p.early_metadata) pdl_wait_primary();
        compact_item<RG>(p, aux, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = aux->tmem_base;
    if (p.compact) {
        r = aux->item[0];
        split = aux->item[1];
        kvh = aux->item[2];
        rg = aux->item[3];
    }

    // Up to here the CTA touched only its own resources (and the kernel
    // parameters), which lets it start while the previous kernel in the stream
    // drains; from here on it reads what that kernel may have written -- except
    // that with early_metadata the caller vouches that the lengths, windows and
    // block table are not among it, and they are read before the wait.
    if (!p.early_metadata) pdl_wait_primary();
    // Without a sliding window the split's first block-table entries sit at a
    // fixed place, so the producers fetch them in the same memory round trip
    // as the request's window and length (entries past the request's pages
    // are never used).  The loads are volatile so that they stay ahead of the
    // request's.  With a window the split starts at a key that depends on the
    // length: those entries are dropped and the producers fetch their own.
    int key_lo = split * p.keys_per_split;
    int pre0 = -1, pre1 = -1;
    if ((warp == 0 || (!KV && warp == 2)) && r >= 0 && r < p.num_reqs) {
        const int32_t* bt = p.block_table + (size_t)r * p.bt_stride;
        const int u0 = key_lo / 16 + lane;
        if ((u0 >> p.page_shift) < p.bt_stride) pre0 = ld_volatile_i32(bt + (u0 >> p.page_shift));
        if (((u0 + 32) >> p.page_shift) < p.bt_stride) pre1 = ld_volatile_i32(bt + ((u0 + 32) >> p.page_shift));
    }
    ReqInfo ri;
    bool active;
    if (p.compact) {
        // the unit of work and its request's metadata (checked) came with the block order
        active = r >= 0;
        ri = aux->item_ri;
    } else {
        const bool reporter = (tid == 0 && blockIdx.x == 0 && kvh == 0);
        active = load_request(p.seq_lens, p.q_indptr, r, p.max_w, p.total_rows, p.max_seq_len,
                              p.bt_stride << (4 + p.page_shift), p.keys_per_split, reporter ? p.status : nullptr,
                              ri, p.window_left, p.split_align, p.dense_block) &&
                 split < ri.nsplits && (!RG || rg * p.window_rows_per_cta < ri.w);
    }
    if (!active) {   // uniform across the CTA
        if (warp == 1) tmem_dealloc(tmem, L::kTmemCols);
        return;
    }
    if (p.early_metadata && !(early_kv && (warp == 0 || warp == 2))) pdl_wait_primary();
    if (p.window_left > 0) {
        key_lo = ri.key_base + split * p.keys_per_split;
        pre0 = pre1 = kNoPrefetch;
    }
    const int G = p.group;
    const int Wg = RG ? p.window_rows_per_cta : p.max_w;   // window rows per row group (Wg x G <= 128)
    const int w_lo = RG ? rg * Wg : 0;                       // this CTA's first window row
    const int R = (RG ? min(ri.w - w_lo, Wg) : ri.w) * G;   // its query rows
    const int key_hi = min(key_lo + p.keys_per_split, ri.cache_len);
    const int Tc = (key_hi - key_lo + kBN - 1) / kBN;   // cache tiles
    // with the dense block operand the request's last split ends with one more
    // tile: the window's own keys (ctx .. len - 1, from the block tensors)
    const int T = Tc + ((p.dense_block && split == ri.nsplits - 1) ? 1 : 0);

    // the request is finished by this kernel (one split), or leaves split partials
    const bool final_out = (ri.nsplits == 1) && !p.always_partials;
    float ep_inv = 0.f, ep_lse2 = -INFINITY;   // softmax threads: 1 / l and log2-sum-exp of their row

    // the split's first tile holds context keys only (its copies may start early)
    const bool first_early = early_kv && key_lo + kBN <= ri.ctx;
    if (warp == 0) {
        // ------------------------------------------------------------ query tile + K producer
        auto issue_q = [&]() {
            if (lane == 0) {
                // one box: 64 head_dim elements x G heads x Wg window rows x the
                // d / 64 chunks, landing chunk-major ([chunk][row][head][128 B]);
                // rows past total_q_rows are zero-filled by TMA, rows past the
                // group's share of W_r x G belong to no output.
                const uint32_t qbytes = static_cast<uint32_t>(L::kChunks * 128 * G * Wg);
                mbar_arrive_expect_tx(&aux->q_full, qbytes);
                tma_load_4d(sQ, &tmq, 0, kvh * G, ri.row0 + w_lo, 0, &aux->q_full);
            }
            __syncwarp();
        };
        // early: the first K tile, then the wait, then the query tile
        if (early_kv && !first_early) pdl_wait_primary();
        if (!first_early) issue_q();
        auto after_first_k = [&]() {
            if (first_early) {
                pdl_wait_primary();
                issue_q();
            }
        };
        if constexpr (KV) {
            // testing (test_stall): nothing arrives, the decoders' waits run out
            const int issued = p.test_stall ? 0
                                            : produce_raw<D>(p, r, kvh, key_lo, key_hi, T, sRaw, aux, &tmk, &tmv,
                                                             &tmks, &tmvs, abort, lane, pre0, pre1);
            if (*abort && lane == 0) {
                drain_copies<L::kNR>(aux->raw_full, issued);
                atomicOr(p.status, kDevWaitTimeout);
            }
        } else {
            // testing (test_stall): K never arrives, its consumers' waits run out
            const int issued = p.test_stall ? 0
                                            : produce<D, NK, false, TRACE>(p, r, kvh, key_lo, key_hi, T, sK,
                                                                           aux->k_full, aux->k_empty, aux->list_k,
                                                                           aux, &tmk, abort, lane, pre0, pre1, Tc,
                                                                           ri.row0, &tmks, 0, after_first_k);
            if (p.test_stall) after_first_k();
            if (*abort && lane == 0) {
                drain_copies<NK>(aux->k_full, issued);
                atomicOr(p.status, kDevWaitTimeout);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ V producer (bf16)
        if constexpr (!KV) {
            // the query tile sits in V slots until the softmax warps have moved
            // it into TMEM: the producer waits for that before its first tile,
            // or (early_kv) before its second
            if (early_kv && !first_early) pdl_wait_primary();
            auto after_first_v = [&]() {
                if (first_early) pdl_wait_primary();
            };
            const int issued = produce<D, NV, true, TRACE>(p, r, kvh, key_lo, key_hi, T, sV, aux->v_full,
                                                           aux->v_empty, aux->list_v, aux, &tmv, abort, lane,
                                                           pre0, pre1, Tc, ri.row0, &tmvs,
                                                           early_kv ? 1 : 0, after_first_v);
            if (*abort && lane == 0) drain_copies<NV>(aux->v_full, issued);
        }
        __syncwarp();
    } else if (KV && warp >= 8) {
        // ------------------------------------------------------------ NVFP4 dequant (K: 8-11, V: 12-15)
        if (warp < 12)
            dequant<D, false, TRACE>(p, key_lo, key_hi, T, sRaw, sK, aux, abort, tid - 256);
        else
            dequant<D, true, TRACE>(p, key_lo, key_hi, T, sRaw, sV, aux, abort, tid - 384);
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues S_t = Q K_t^T and warp 3 O += P_t V_t, each in tile order
        // with blocking (bounded) waits on its own inputs only: a late K tile
        // never holds back a P V, nor a P not yet written the next S.
        if (lane == 0) {
            // NVFP4: fp16 operands (query tile in TMEM, K / V decoded, P fp16);
            // bf16 KV: bf16 operands
            constexpr uint32_t idesc_s = KV ? idesc_f16_f32(kM, kBN, 0, 0) : idesc_bf16_f32(kM, kBN, 0, 0);
            constexpr uint32_t idesc_o = KV ? idesc_f16_f32(kM, D, 0, 1) : idesc_bf16_f32(kM, D, 0, 1);
            const bool pv_issuer = (warp == 3);
            bool ok = pv_issuer || mbar_wait(&aux->q_ready, 0, abort, kWaitLimit);
            tc_fence_after();
            constexpr int NSB = L::kSBufs;
            // S_n = Q K_n^T into S buffer n % NSB
            auto issue_s = [&](int n) {
                const int ks = n % NK, b = n % NSB;
                tc_fence_after();
                const uint32_t k_addr = smem_addr(sK + ks * L::kTileBytes);
                const uint32_t d_tmem = tmem + D + b * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c = kk >> 2, sub = kk & 3;
                    const uint64_t bd = smem_desc_sw128(k_addr + c * (kBN * 128) + sub * 32, 16, 1024);
                    // query elements 16 kk .. 16 kk + 15: TMEM columns 8 kk .. 8 kk + 7
                    mma_ts(d_tmem, tmem + L::kQCol + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&aux->k_empty[ks]);
                mma_commit(&aux->s_full[b]);
            };
            // O += P_n V_n, one MMA per 16-key unit
            auto issue_pv = [&](int n) {
                const int vs = n % NV, b = n & 1;
                tc_fence_after();
                const int np = n >= Tc ? 1 : min(kPPT, (key_hi - (key_lo + n * kBN) + 15) / 16);
                const uint32_t v_addr = smem_addr(sV + vs * L::kTileBytes);
                for (int kk = 0; kk < np; ++kk) {
                    // V page kk: [chunk][16 keys][128 B]; MN atoms (64 head_dim
                    // elements) 2 KB apart, 8-key groups 1 KB apart
                    const uint64_t bd = smem_desc_sw128(v_addr + kk * L::kPageBytes, 2048, 1024);
                    // P keys 16 kk .. 16 kk + 15: TMEM columns 8 kk .. 8 kk + 7 of buffer b
                    mma_ts(tmem, tmem + L::p_col(b) + kk * 8, bd, idesc_o, (n > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&aux->v_empty[vs]);
                // bf16: P sat in S buffer b, which the S MMA of tile n + 2 may now overwrite
                mma_commit(&aux->s_empty[b]);
                mma_commit(&aux->o_done);
            };
            long long t_idle = clock64();
            if (!pv_issuer) {
                for (int t = 0; t < T && ok; ++t) {
                    ok = mbar_wait(&aux->k_full[t % NK], (t / NK) & 1, abort, kWaitLimit) &&
                         (t < NSB || mbar_wait(&aux->s_empty[t % NSB], ((t / NSB) - 1) & 1, abort, kWaitLimit));
                    if (ok) issue_s(t);
                }
            } else {
                for (int t = 0; t < T && ok; ++t) {
                    ok = mbar_wait(&aux->p_full[t & 1], (t >> 1) & 1, abort, kWaitLimit) &&
                         mbar_wait(&aux->v_full[t % NV], (t / NV) & 1, abort, kWaitLimit);
                    if (ok) issue_pv(t);
                }
            }
            // O is final once every P V is done.  A separate barrier: the softmax
            // warps can finish their loop while two P V are still pending, and a
            // parity wait on o_done would then match an older phase.
            if (ok && pv_issuer) mma_commit(&aux->o_final);
            // every MMA this thread issued completes before TMEM is released
            uint64_t* drain = pv_issuer ? &aux->drain_pv : &aux->drain;
            mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, kDrainLimit);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        const int wq = warp - 4;
        const int m = wq * 32 + lane;
        const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const bool valid = m < R;
        const int i = w_lo + (valid ? m / G : 0);      // window row
        const int hq = kvh * G + (valid ? m % G : 0);
        const int qrow = ri.row0 + i;
        const int hi = (p.mask_mode == 0) ? (ri.ctx + i) : (ri.len - 1);
        const bool has_window = p.window_left > 0;
        const int lo = has_window ? max(0, hi - p.window_left + 1) : 0;   // first visible key
        const float sc = p.score_scale_log2;
        float m_ref = -INFINITY, l_sum = 0.f;
        long long tr_cnt = 0, tr_sum = 0;
        bool ok = true;
        {
            // The query tile arrives as bf16 in the V slots.  Thread m moves its
            // row into the TMEM columns the S = Q K^T MMA reads as its A operand,
            // two elements per column, the lower one in the low half.  NVFP4:
            // its MMAs take fp16, so the row is converted on the way (saturating
            // at +-65504; exact for every bf16 value of magnitude 2^-14 .. 65504).
            // Rows past R (padding) are zero: their scores are exactly 0.
            if ((ok = warp_wait(&aux->q_full, 0, abort))) {
                const uint32_t qb = smem_addr(sQ);
                const int box_rows = G * Wg;   // rows per chunk of the landed box
#pragma unroll 1
                for (int c = 0; c < L::kChunks; ++c) {
                    uint32_t w[32];
                    // the box's row (c, m) is 128-byte row c * box_rows + m of the
                    // landing area, its 16-byte pieces swizzled by that row's index
                    const int lr = c * box_rows + m;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (valid) v = ld_shared_v4(qb + lr * 128 + ((q ^ (lr & 7)) << 4));
                        if constexpr (KV) {
                            w[4 * q + 0] = bf16x2_to_f16x2_sat(v.x);
                            w[4 * q + 1] = bf16x2_to_f16x2_sat(v.y);
                            w[4 * q + 2] = bf16x2_to_f16x2_sat(v.z);
                            w[4 * q + 3] = bf16x2_to_f16x2_sat(v.w);
                        } else {
                            w[4 * q + 0] = v.x;
                            w[4 * q + 1] = v.y;
                            w[4 * q + 2] = v.z;
                            w[4 * q + 3] = v.w;
                        }
                    }
                    tmem_st32u(lane_tmem + L::kQCol + c * 32, w);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aux->q_ready);
            }
        }
        for (int t = 0; t < T && ok; ++t) {
            const int b = t & 1;                      // P buffer
            constexpr int NSB = L::kSBufs;
            const int sb = t % NSB;                   // S buffer
            if (!(ok = warp_wait(&aux->s_full[sb], (t / NSB) & 1, abort))) break;
            tc_fence_after();
            float sv[kBN];
#pragma unroll
            for (int h = 0; h < kBN / 32; ++h)
                tmem_ld32(lane_tmem + D + sb * kBN + h * 32, *reinterpret_cast<float(*)[32]>(sv + h * 32));
            tmem_wait_ld();
            // P goes where S was, and the P V MMA frees the buffer

            // tile t covers keys key0 .. key0 + 63 (the dense block tile: ctx .. ctx + W - 1)
            const bool block_tile = t >= Tc;
            const int key0 = block_tile ? ri.ctx : key_lo + t * kBN;
            const int kend = block_tile ? ri.len : key_hi;
            const int lim = valid ? (min(kend - 1, hi) - key0) : -1;  // visible iff lim_lo <= c <= lim
            const int lim_lo = lo - key0;
            // Scores stay unscaled: the maximum is taken on raw scores (sc > 0) and
            // the scale is folded into one FFMA per exponent.  Tiles whose keys
            // are all visible to every output row of the warp skip the mask.
            // Padding rows (past W x G) never reach an output; their scores are
            // finite (zero-filled or another window's rows), so they may run
            // unmasked, and they never ask for a rescale.
            float mraw = -INFINITY;
            // no row's window starts inside this tile (always so without a window)
            const bool no_lower = !has_window || __all_sync(kFullMask, lim_lo <= 0);
            if (no_lower && __all_sync(kFullMask, !valid || lim >= kBN - 1)) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) mraw = fmaxf(mraw, sv[c]);
            } else if (no_lower) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    if (c > lim) sv[c] = -INFINITY;
                    mraw = fmaxf(mraw, sv[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    if (c > lim || c < lim_lo) sv[c] = -INFINITY;
                    mraw = fmaxf(mraw, sv[c]);
                }
            }
            const float mx = mraw * sc;
            const bool need = valid && (m_ref != -INFINITY) && (mx > m_ref + kRescaleThreshold);
            const bool first = (m_ref == -INFINITY) && (mx != -INFINITY);
            const float ref = (need || first) ? mx : m_ref;
            const float alpha = need ? fast_exp2(m_ref - ref) : 1.f;
            uint32_t pk[kBN / 2];
            float psum = 0.f;
            const float nref = (ref == -INFINITY) ? 0.f : -ref;   // masked scores are -inf -> p = 0
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                const float p0 = fast_exp2(fmaf(sv[c], sc, nref));
                const float p1 = fast_exp2(fmaf(sv[c + 1], sc, nref));
                // the normaliser sums the fp32 weights: rounding P to 16 bits for
                // the PV MMA must not leak into l (and so into LSE) on rows
                // that see only a few keys
                psum += p0 + p1;
                if constexpr (KV) {
                    pk[c >> 1] = pack_half2(p0, p1);
                } else {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[c >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
                }
            }
            l_sum = l_sum * alpha + psum;
            m_ref = ref;

            // (S_t, and so P_t, could only be written to buffer b once PV_{t-2}
            // had finished with it)
            if (__any_sync(kFullMask, need) && t > 0) {
                // rescaling O needs every earlier P V finished
                if (!(ok = warp_wait(&aux->o_done, (t - 1) & 1, abort))) break;
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
            const int vs = t % NV;
            // The request's last page may end mid-page: its stale slots hold
            // arbitrary (even non-finite) values and 0 * NaN is NaN, so zero them.
            // (NVFP4 tiles come out of the dequant already zeroed past key_hi)
            // (the dense block unit holds other windows' rows past W: zeroed likewise)
            const bool ragged_tail =
                !KV && (block_tile || (key_hi == ri.cache_len && t == Tc - 1 && (ri.cache_len & 15) != 0));
            if (ragged_tail || TRACE) {
                if (!(ok = warp_wait(&aux->v_full[vs], (t / NV) & 1, abort))) break;
            }
            if (ragged_tail) {
                const int np = block_tile ? 1 : min(kPPT, (key_hi - key0 + 15) / 16);
                const int row_first = block_tile ? ri.w : ri.cache_len - key0, row_end = np * 16;
                unsigned char* vt = sV + vs * L::kTileBytes;
                const int pieces = (row_end - row_first) * L::kChunks * 8;
                for (int u = m; u < pieces; u += 128) {
                    const int rr = row_first + u / (L::kChunks * 8);
                    const int rem = u % (L::kChunks * 8);
                    const int c = rem >> 3, j = rem & 7;
                    *reinterpret_cast<uint4*>(vt + (rr >> 4) * L::kPageBytes + c * 2048 + (rr & 15) * 128 + (j << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (TRACE) {
                for (int c = max(0, lim_lo); c <= lim && c < kBN; ++c) {
                    const int key = key0 + c;
                    tr_cnt += 1;
                    // a dense block key has no cache slot: it counts -(1 + its row)
                    tr_sum += block_tile ? -1 - (long long)(ri.row0 + c)
                                         : (long long)aux->pages_v[vs][c >> 4] * 16 + (key & 15);
                }
            }
            // P row m (16-bit pairs, key 2c in the low half) into TMEM buffer b
            static_assert(kBN == 64, "one 32-column store per P row");
            tmem_st32u(lane_tmem + L::p_col(b), pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aux->p_full[b]);
        }
        pdl_launch_dependents();
        if (ok) ok = warp_wait(&aux->o_final, 0, abort);
        tc_fence_after();
        if (ok) {
            // Every MMA and copy has completed (o_final), so the ring buffers
            // are free.  The row's normaliser and log-sum-exp go to the
            // epilogue below; a request with a single split is finished here:
            // each thread stages its row of bf16 O (row stride padded by 16
            // bytes so the 16-byte stores of a warp hit distinct banks), which
            // every warp then copies out.
            ep_inv = (valid && l_sum > 0.f) ? (p.out_scale / l_sum) : 0.f;
            ep_lse2 = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) : -INFINITY;
            if (final_out && wq * 32 < R) {   // warps holding output rows only
                unsigned char* myrow = smem + m * (D * 2 + 16);
                // two 32-column TMEM loads in flight per wait
#pragma unroll 1
                for (int ch0 = 0; ch0 < D / 32; ch0 += 2) {
                    float ov[2][32];
                    tmem_ld32(lane_tmem + ch0 * 32, ov[0]);
                    tmem_ld32(lane_tmem + (ch0 + 1) * 32, ov[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                    ov[hh][q4 * 8 + 2 * e] * ep_inv, ov[hh][q4 * 8 + 2 * e + 1] * ep_inv);
                                w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                            }
                            *reinterpret_cast<uint4*>(myrow + (ch0 + hh) * 64 + q4 * 16) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
            if (valid) {
                if (final_out && p.lse) p.lse[(size_t)qrow * p.num_q_heads + hq] = ep_lse2 * kLn2;
                if (TRACE && p.trace) {
                    unsigned long long* tp =
                        reinterpret_cast<unsigned long long*>(p.trace + ((size_t)qrow * p.num_q_heads + hq) * 2);
                    atomicAdd(tp, (unsigned long long)tr_cnt);
                    atomicAdd(tp + 1, (unsigned long long)tr_sum);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // Every role has finished, so the abort flag is final.  Nothing is written
    // if any role gave up.
    const bool ep_ok = (*abort == 0);
    if (ep_ok && !final_out && warp < 8) {
        // ------------------------------------------------------------ split partial (warps 0-7)
        // Straight from TMEM to global memory, no staging: warp w reads TMEM
        // lanes 32 (w % 4) .. + 31 (query rows), warps 4-7 the first half of
        // the head_dim columns and warps 0-3 the second.  A partial is fp16 of
        // O_s / scale_s with scale_s = max_e |O_s[e]| (the halves exchange
        // their maxima through shared memory), stored chunk-major within the
        // request's block of W_r x G rows (see partial_chunk), so that the 32
        // rows of a warp fill 512 contiguous bytes per chunk.
        tc_fence_after();
        float* ep = reinterpret_cast<float*>(smem);   // [0, kM) 1 / l;  [kM, 3 kM) max |O| per half
        const int mrow = (warp & 3) * 32 + lane;
        const int half = warp < 4 ? 1 : 0;
        if (warp >= 4) ep[mrow] = ep_inv;
        named_barrier_sync(1, 256);
        const bool rows_here = (warp & 3) * 32 < R;   // warp-uniform
        const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + half * (D / 2);
        const float inv = ep[mrow];
        float amax = 0.f;
        if (rows_here) {
#pragma unroll 1
            for (int ch = 0; ch < D / 64; ++ch) {
                float ov[32];
                tmem_ld32(taddr + ch * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(ov[e]));
            }
            amax *= inv;
        }
        ep[kM * (1 + half) + mrow] = amax;
        named_barrier_sync(1, 256);
        if (rows_here) {
            amax = fmaxf(ep[kM + mrow], ep[2 * kM + mrow]);
            const float rsc = amax > 0.f ? inv / amax : 0.f;
            const bool row_ok = mrow < R;
            if (warp >= 4 && row_ok)
                p.ws_ls[partial_pair(split, p.total_rows, p.num_q_heads, G, kvh, ri.row0 + w_lo + mrow / G,
                                     mrow % G)] = make_float2(ep_lse2, amax);
            uint16_t* blk = p.ws_o + partial_pair(split, p.total_rows, p.num_q_heads, G, kvh, ri.row0, 0) * D;
            const int rtot = ri.w * G, mg = w_lo * G + mrow;   // the request's rows; this row among them
#pragma unroll 1
            for (int ch = 0; ch < D / 64; ++ch) {
                float ov[32];
                tmem_ld32(taddr + ch * 32, ov);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 h;
                        h.x = pack_half2(ov[q4 * 8 + 0] * rsc, ov[q4 * 8 + 1] * rsc);
                        h.y = pack_half2(ov[q4 * 8 + 2] * rsc, ov[q4 * 8 + 3] * rsc);
                        h.z = pack_half2(ov[q4 * 8 + 4] * rsc, ov[q4 * 8 + 5] * rsc);
                        h.w = pack_half2(ov[q4 * 8 + 6] * rsc, ov[q4 * 8 + 7] * rsc);
                        const int c = half * (D / 16) + ch * 4 + q4;   // 8-element chunk of the row
                        st_global_v4(blk + partial_chunk(c, rtot, mg), h);
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
    if (!ep_ok) {
        if (tid == 0) atomicOr(p.status, kDevWaitTimeout);   // whichever role gave up, the call reports it
    } else if (final_out) {
        // ------------------------------------------------------------ copy-out (every thread)
        // The staged bf16 rows leave in coalesced 16-byte pieces, several
        // loads in flight per thread before their stores, to [row][head] with
        // the G heads of a window row adjacent.
        constexpr int kBatchPieces = 8;
        const int nt = blockDim.x;
        const uint32_t sbase = smem_addr(smem);
        constexpr int lg = (D == 64 ? 3 : D == 128 ? 4 : 5);   // 16-byte pieces per bf16 row
        constexpr int rs = D * 2 + 16;
        const int total = R << lg;
        for (int u0 = tid; u0 < total; u0 += nt * kBatchPieces) {
            uint4 v[kBatchPieces];
#pragma unroll
            for (int k = 0; k < kBatchPieces; ++k) {
                const int u = u0 + k * nt;
                if (u < total) v[k] = ld_shared_v4(sbase + (u >> lg) * rs + (u & ((1 << lg) - 1)) * 16);
            }
#pragma unroll
            for (int k = 0; k < kBatchPieces; ++k) {
                const int u = u0 + k * nt;
                if (u < total) {
                    const int mm = u >> lg, c = u & ((1 << lg) - 1);
                    unsigned char* dst = reinterpret_cast<unsigned char*>(p.o) +
                                         (((size_t)(ri.row0 + w_lo + mm / G) * p.num_q_heads + kvh * G + mm % G) * D) * 2 +
                                         c * 16;
                    st_global_v4(dst, v[k]);
                }
            }
        }
    }
}

using TcKernel = void (*)(const SplitParams, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const CUtensorMap, const CUtensorMap);

template <int D, int KV, bool RG>
TcKernel pick_trace(bool traced) {
    return traced ? &split_attn_tc_kernel<D, KV, true, RG> : &split_attn_tc_kernel<D, KV, false, RG>;
}

template <int D, int KV>
TcKernel pick_rg(bool traced, bool row_groups) {
    return row_groups ? pick_trace<D, KV, true>(traced) : pick_trace<D, KV, false>(traced);
}

template <int KV>
TcKernel pick_d(int d, bool traced, bool row_groups) {
    switch (d) {
        case 64: return pick_rg<64, KV>(traced, row_groups);
        case 128: return pick_rg<128, KV>(traced, row_groups);
        case 256: return pick_rg<256, KV>(traced, row_groups);
        default: return nullptr;
    }
}

// row_groups: the launch has more than one row group per (request, KV head, split)
TcKernel pick(int d, int kv, bool traced, bool row_groups) {
    return kv ? pick_d<1>(d, traced, row_groups) : pick_d<0>(d, traced, row_groups);
}

template <int KV>
int smem_d(int d) {
    switch (d) {
        case 64: return TcLayout<64, KV>::kSmem;
        case 128: return TcLayout<128, KV>::kSmem;
        case 256: return TcLayout<256, KV>::kSmem;
        default: return 0;
    }
}

int smem_for(int d, int kv) { return kv ? smem_d<1>(d) : smem_d<0>(d); }

// The driver's tensor-map encoder, looked up once (a function-local static:
// initialised by the first caller, safely when plans are made from several
// host threads).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        const bool ok = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                                         &q) == cudaSuccess &&
                        q == cudaDriverEntryPointSuccess;
        return ok ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr) : nullptr;
    }();
    return fn;
}

// Pool pages [Hkv, ps, d] bf16, page_stride bytes apart, viewed as a 4-D tensor
// (d, slot, kv head, page); box = 64 head_dim elements x 16 slots of one page
// and head (one 16-key unit), 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int num_pages, int hkv, int d, int ps,
                     long long page_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)ps, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * ps, (cuuint64_t)page_stride};
    cuuint32_t box[4] = {64, 16, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// The same pool as a 5-D tensor (64 elements, slot, 64-element chunk, kv head,
// page); box = one whole 16-key unit of a page-head, landing chunk-major:
// [chunk][16 slots][128 B].
bool encode_pool_map_units(CUtensorMap* map, const void* pool, int num_pages, int hkv, int d, int ps,
                           long long page_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {64, (cuuint64_t)ps, (cuuint64_t)d / 64, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {(cuuint64_t)d * 2, 128, (cuuint64_t)d * 2 * ps, (cuuint64_t)page_stride};
    cuuint32_t box[5] = {64, 16, (cuuint32_t)d / 64, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// NVFP4 code pool pages [Hkv, ps, d/2] bytes viewed as (d/2 bytes, slot, kv head,
// page); box = one 16-key unit of a page-head, swizzled 128/64/32 bytes for
// d = 256/128/64 (the row is d/2 bytes).
bool encode_code_map(CUtensorMap* map, const void* pool, int num_pages, int hkv, int d, int ps,
                     long long page_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d / 2, (cuuint64_t)ps, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d / 2, (cuuint64_t)d / 2 * ps, (cuuint64_t)page_stride};
    cuuint32_t box[4] = {(cuuint32_t)d / 2, 16, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = d == 256 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// NVFP4 scale pool pages [Hkv, ps, d/16] bytes viewed as (ps * d/16 bytes, kv
// head, page); box = the d bytes of scales of one 16-key unit.
bool encode_scale_map(CUtensorMap* map, const void* pool, int num_pages, int hkv, int d, int ps,
                      long long page_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)ps * d / 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[2] = {(cuuint64_t)ps * d / 16, (cuuint64_t)page_stride};
    cuuint32_t box[3] = {(cuuint32_t)d, 1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// Dense block operand [total_rows, Hkv, d] bf16 viewed as (d, row, kv head);
// box = 64 elements x 16 rows of one head (a 16-key unit of K), 128-byte
// swizzle; rows past total_rows are zero-filled.
bool encode_block_k_map(CUtensorMap* map, const void* t, int total_rows, int hkv, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)total_rows, (cuuint64_t)hkv};
    cuuint64_t strides[2] = {(cuuint64_t)hkv * d * 2, (cuuint64_t)d * 2};
    cuuint32_t box[3] = {64, 16, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(t), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// The same tensor as (64 elements, row, 64-element chunk, kv head); box = 16
// rows of one head with all their chunks, landing [chunk][16 rows][128 B] like
// a page unit of V.
bool encode_block_v_map(CUtensorMap* map, const void* t, int total_rows, int hkv, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)total_rows, (cuuint64_t)d / 64, (cuuint64_t)hkv};
    cuuint64_t strides[3] = {(cuuint64_t)hkv * d * 2, 128, (cuuint64_t)d * 2};
    cuuint32_t box[4] = {64, 16, (cuuint32_t)d / 64, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(t), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// Q [total_rows, Hq, d] bf16 viewed as (d, head, row); box = 64 elements x G heads
// x max_w rows, 128-byte swizzle, out-of-range rows zero-filled.
bool encode_q_map(CUtensorMap* map, const void* q, int total_rows, int hq, int d, int group, int max_w) {
    auto fn = encode_fn();
    if (!fn) return false;
    // Q [total_rows, Hq, d] bf16 as (64 elements, head, row, 64-element chunk):
    // one box takes every chunk of G heads x max_w rows, chunk-major
    cuuint64_t dims[4] = {64, (cuuint64_t)hq, (cuuint64_t)total_rows, (cuuint64_t)d / 64};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * hq, 128};
    cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)max_w, (cuuint32_t)d / 64};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

}  // namespace

// Any row count: windows of more than 128 query rows per KV head are split
// into row groups of whole window rows (G <= 16 rows each, so a group is never
// empty).
bool tc_supported(int head_dim, int kv_dtype, int max_rows) {
    return (kv_dtype == 0 || kv_dtype == 1) && max_rows >= 1 && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

int tc_window_rows_per_cta(int max_w, int group) { return max_w < kM / group ? max_w : kM / group; }

int tc_smem_bytes(int head_dim, int kv_dtype) { return smem_for(head_dim, kv_dtype); }
int tc_threads(int kv_dtype) { return kv_dtype ? kTcThreadsFp4 : kTcThreadsBf16; }

cudaError_t tc_prepare(int head_dim, int kv_dtype) {
    for (int v = 0; v < 4; ++v) {
        TcKernel k = pick(head_dim, kv_dtype, (v & 1) != 0, (v & 2) != 0);
        if (!k) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_for(head_dim, kv_dtype));
        if (e != cudaSuccess) return e;
    }
    return encode_fn() ? cudaSuccess : cudaErrorNotSupported;
}

bool tc_encode_maps(const SplitParams& p, int kv_dtype, TcMaps* maps) {
    static_assert(sizeof(CUtensorMap) == sizeof(maps->q), "tensor map size");
    if (!encode_q_map(reinterpret_cast<CUtensorMap*>(maps->q), p.q, p.total_rows, p.num_q_heads, p.head_dim,
                      p.group, p.window_rows_per_cta))
        return false;
    const int ps = 16 << p.page_shift;
    if (kv_dtype != 0)
        return encode_code_map(reinterpret_cast<CUtensorMap*>(maps->k), p.k_pool, p.num_pages, p.num_kv_heads,
                               p.head_dim, ps, p.kv_page_stride) &&
               encode_code_map(reinterpret_cast<CUtensorMap*>(maps->v), p.v_pool, p.num_pages, p.num_kv_heads,
                               p.head_dim, ps, p.kv_page_stride) &&
               encode_scale_map(reinterpret_cast<CUtensorMap*>(maps->ks), p.k_scales, p.num_pages,
                                p.num_kv_heads, p.head_dim, ps, p.scale_page_stride) &&
               encode_scale_map(reinterpret_cast<CUtensorMap*>(maps->vs), p.v_scales, p.num_pages,
                                p.num_kv_heads, p.head_dim, ps, p.scale_page_stride);
    memset(maps->ks, 0, sizeof(maps->ks));
    memset(maps->vs, 0, sizeof(maps->vs));
    if (p.dense_block &&
        !(encode_block_k_map(reinterpret_cast<CUtensorMap*>(maps->ks), p.block_k, p.total_rows, p.num_kv_heads,
                             p.head_dim) &&
          encode_block_v_map(reinterpret_cast<CUtensorMap*>(maps->vs), p.block_v, p.total_rows, p.num_kv_heads,
                             p.head_dim)))
        return false;
    return encode_pool_map(reinterpret_cast<CUtensorMap*>(maps->k), p.k_pool, p.num_pages, p.num_kv_heads,
                           p.head_dim, ps, p.kv_page_stride) &&
           encode_pool_map_units(reinterpret_cast<CUtensorMap*>(maps->v), p.v_pool, p.num_pages, p.num_kv_heads,
                                 p.head_dim, ps, p.kv_page_stride);
}

cudaError_t tc_launch(const SplitParams& p, int kv_dtype, const TcMaps& maps, bool traced, dim3 grid,
                      cudaStream_t stream, bool programmatic) {
    TcKernel k = pick(p.head_dim, kv_dtype, traced, p.row_groups > 1);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(tc_threads(kv_dtype), 1, 1);
    lc.dynamicSmemBytes = smem_for(p.head_dim, kv_dtype);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k, p, *reinterpret_cast<const CUtensorMap*>(maps.q),
                              *reinterpret_cast<const CUtensorMap*>(maps.k),
                              *reinterpret_cast<const CUtensorMap*>(maps.v),
                              *reinterpret_cast<const CUtensorMap*>(maps.ks),
                              *reinterpret_cast<const CUtensorMap*>(maps.vs));
}

}  // namespace spec_attn
