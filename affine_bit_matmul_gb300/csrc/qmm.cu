// Quantized GEMM on the sm_103a tensor cores: y = x . w^T with w dequantised
// on the fly (w^ = s*q + b per group of 32, 64 or 128 consecutive k), dense
// and sorted-MoE forms.
//
// Prior art: the qmm_naive and grouped-GEMM kernels profiled in mlxcel issue
// #1536 (Baseline profile table; Diagnosis items 1, 4 and 5) and PR #1562
// (Summary: the sorted-MoE prefill path over B = tokens * top_k rows).  Those
// ran FP32 FMA on CUDA cores; this kernel is built for tcgen05 instead:
//
//  * swap-AB: the MMA's M side is 128 rows of w (output columns n), its N side
//    is a tile of up to 256 activation rows, so a 36-row expert segment or a
//    single decode row still fills the 128-row tensor-core tile;
//  * a TMA copy brings the packed codes of the 128 w rows into a ring of
//    slots of 256 bytes per row (two 128-byte-swizzled boxes); per 64-wide
//    block the activation tile comes by TMA with 128-byte swizzle into its
//    own ring (in the grouped form from a copy of the activation rows in
//    sorted order);
//  * eight dequant warps (two groups of four take alternate 128-wide stages;
//    thread r owns w row r, its tensor-memory lane) turn codes into bf16
//    w^ = s*q + b (one rounding) and store them in tensor memory, where the
//    MMA reads its A operand;
//  * one elected lane issues eight 128xNx16 tcgen05.mma per stage into fp32
//    tensor memory; the epilogue reads the accumulators with tcgen05.ld and
//    stores bf16.
//
// Three launch forms:
//  * qmm_tc_kernel: one CTA per output tile.  With few tiles (small M), K is
//    split over the CTAs of a cluster and the fp32 partials are added through
//    distributed shared memory in rank order, so the result does not depend
//    on timing;
//  * qmm_persistent_kernel, dense: one CTA per SM walks the tiles with its
//    rings running across tile boundaries and four epilogue warps;
//  * qmm_persistent_kernel, compact (grouped, 4-bit): two CTAs per SM, tiles
//    handed out by a counter, the dequant warps run the epilogue.
//
// Every wait on an mbarrier is bounded; on expiry the kernel sets
// MXQ_DEV_TIMEOUT, stops issuing work, lets issued work finish and frees its
// tensor memory before returning.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_device.cuh"
#include "mxq_internal.h"
#include "tc_common.cuh"

namespace mxq {
namespace {

constexpr int kDequantWarps = 8;     // warps 0-7: dequant + epilogue
constexpr int kDequantThreads = kDequantWarps * 32;
constexpr int kCodeWarp = 8;         // codes TMA
constexpr int kMmaWarp = 9;          // TMEM owner, MMA issue
constexpr int kXWarp0 = 10;          // activation TMA
constexpr int kThreads = 11 * 32;
constexpr int kTileN = 128;          // rows of w per CTA (MMA M)
constexpr int kBK = 128;             // K per dequant/MMA stage: two 64-wide halves
constexpr int kHalfK = 64;           // K per activation slot (one 128-byte swizzle atom)
constexpr int kMaxCodeStages = 8;    // code slots
// A code slot holds 256 bytes of each of the 128 w rows (the TMA engine
// handles long row segments far faster than 64-byte ones), as two boxes of
// 128 bytes per row stored with the 128-byte swizzle: 16-byte chunk c of row
// r sits at chunk c ^ (r % 8) of its 128-byte line, so the eight threads of
// a quarter warp, reading the same chunk of eight consecutive rows, hit
// eight different bank groups.
constexpr int kCodeSlotRowBytes = 256;
constexpr int kCodeBoxRowBytes = 128;
// 3- and 6-bit stages are 48 and 96 bytes per row: their slots hold 384
// bytes (three boxes, 8 or 4 stages), so a stage may cross a box boundary.
// The compact form (two CTAs per SM, 108 KB each) uses one-box slots: a
// slot is held until its last stage is dequantised, so with 16 KB slots
// three of four can be loading where two 32 KB slots left one.
__host__ __device__ constexpr int slot_row_bytes(int bits, bool compact = false) {
    return compact ? kCodeBoxRowBytes : (bits == 3 || bits == 6) ? 384 : kCodeSlotRowBytes;
}
constexpr int kCodeBoxBytes = kTileN * kCodeBoxRowBytes;
constexpr int kMaxAStages = 6;       // dequantised stages held in tensor memory
constexpr int kMaxClusterSplits = 8; // K splits per tile: the portable cluster size
constexpr int kMaxXStages = 16;
constexpr int kSmemBudget = 224 * 1024;
constexpr int kTmemCols = 512;       // accumulator + dequantised A stages
// Compact layout (grouped form, tiles of at most 64 activation rows, 4-bit
// codes): half the shared and tensor memory, so two persistent CTAs share an
// SM and their two pipelines hide
// each other's latency.
constexpr int kCompactRows = 64;
constexpr int kCompactSmemBudget = 108 * 1024;
constexpr int kCompactTmemCols = 256;

// Scale/bias pairs of one 128-wide stage.  Groups of 64 or 128 give one
// pair per 64-wide half (two halves of one 128-group load the same pair);
// groups of 32 give one pair per 32-wide quarter.  Pair i of a stage whose
// first 64-wide block is kb (counted from k = 0) belongs to group
// group_of(kb, i); the dequantiser's half h, 32-wide chunk c uses pair
// pair_of(h, c).
template <int GROUP>
struct StageGroups {
    static_assert(GROUP == 32 || GROUP == 64 || GROUP == 128, "group of 32, 64 or 128");
    static constexpr int kPairs = GROUP == 32 ? 4 : 2;
    __device__ static constexpr int half_of(int i) { return GROUP == 32 ? i >> 1 : i; }
    __device__ static constexpr int pair_of(int h, int c) { return GROUP == 32 ? h * 2 + c : h; }
    __device__ static int group_of(int kb, int i) {
        return GROUP == 32 ? kb * 2 + i : (kb + i) / (GROUP / 64);
    }
};

__host__ __device__ constexpr bool compact_mode(int bits, int max_rows, bool gather) {
    return gather && (bits == 2 || bits == 4) && max_rows <= kCompactRows;
}
constexpr int kAStageCols = kBK / 2; // one bf16 pair per 32-bit column

struct SmemLayout {
    int c_bytes, c_stages;    // packed-code ring: slots of slot_row_bytes(bits) per w row
    int x_bytes, x_stages;    // activation ring (MMA B operand), one 64-wide atom per slot
    int c_offset;             // rings: x at 0, then codes
    int bar_offset, total;
};

// Ring depths in shared memory (the dequantised A operand lives in tensor
// memory).  The activation tile comes from L2 with about a microsecond of
// latency and the packed codes stream from HBM with up to two: two code
// slots, up to six activation slots, then more code slots (up to 8), then
// more activation slots (up to 16).  A code slot is 32 KB at every width
// (4 stages of 4-bit codes or 2 of 8-bit), 48 KB for 3- and 6-bit codes,
// and 16 KB in the compact form.
__host__ __device__ inline SmemLayout make_layout(int max_rows, bool compact, int slot_bytes) {
    SmemLayout L;
    const int budget = compact ? kCompactSmemBudget : kSmemBudget;
    const int rows16 = (max_rows + 15) & ~15;
    L.c_bytes = kTileN * slot_bytes;  // 32 KB: 8, 4 or 2 stages of 2-, 4-, 8-bit; 48 KB: 8 or 4 of 3-, 6-bit; compact 16 KB
    L.x_bytes = (rows16 / 8) * 1024;                  // 128 B per row, 8-row atoms
    // two code slots, up to six activation slots, then more code slots (up
    // to kMaxCodeStages), then more activation slots (up to kMaxXStages)
    L.c_stages = 2;
    int room = budget - L.c_stages * L.c_bytes;
    L.x_stages = room / L.x_bytes;
    if (L.x_stages > 6) L.x_stages = 6;
    if (L.x_stages < 2) L.x_stages = 2;
    room -= L.x_stages * L.x_bytes;
    while (L.c_stages < kMaxCodeStages && room >= L.c_bytes) {
        ++L.c_stages;
        room -= L.c_bytes;
    }
    while (L.x_stages < kMaxXStages && room >= L.x_bytes) {
        ++L.x_stages;
        room -= L.x_bytes;
    }
    L.c_offset = L.x_stages * L.x_bytes;
    L.bar_offset = L.c_offset + L.c_stages * L.c_bytes;
    // cfull, cempty (per code slot); afull, aempty; xfull, xempty; accf; tmem base
    L.total = L.bar_offset + (2 * kMaxCodeStages + 2 * kMaxAStages + 2 * kMaxXStages + 1) * 8 +
              16 + 1024;                              // + alignment slack
    return L;
}

// Word j of a stage's codes (uint4 chunks in order, four words each).
template <int BITS>
__device__ __forceinline__ uint32_t stage_word(const uint4 (&cw)[BITS], int j) {
    const uint4 v = cw[j >> 2];
    const int e = j & 3;
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Bits [p, p + BITS) of the little-endian bit stream in the stage's words,
// placed at bit `at` of the result (0 or 16), all other bits zero.
template <int BITS>
__device__ __forceinline__ uint32_t stream_field(const uint4 (&cw)[BITS], int p, int at) {
    const int j = p >> 5, off = p & 31;
    uint32_t t;
    if (off + BITS > 32)
        t = __funnelshift_r(stage_word<BITS>(cw, j), stage_word<BITS>(cw, j + 1), off - at);
    else if (off >= at)
        t = stage_word<BITS>(cw, j) >> (off - at);
    else
        t = stage_word<BITS>(cw, j) << (at - off);
    return t & (((1u << BITS) - 1u) << at);
}

// 32 codes of 3 or 6 bits starting at word w0 of the stage (32 * BITS bits,
// word aligned) -> sixteen bf16x2 words of s*q + b, one rounding each.
template <int BITS>
__device__ __forceinline__ void dequant_stream32(const uint4 (&cw)[BITS], int w0, uint32_t s2,
                                                 uint32_t b2, uint32_t (&out)[16]) {
    const uint32_t k128 = 0x43004300u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int p = w0 * 32 + 2 * i * BITS;
        // bf16 0x43qq = 128 + q exactly (q < 64); subtracting 128 is exact
        const uint32_t e = stream_field<BITS>(cw, p, 0) | stream_field<BITS>(cw, p + BITS, 16) |
                           0x43004300u;
        out[i] = hfma2_bf16(hsub2_bf16(e, k128), s2, b2);
    }
}

template <int BITS, bool GATHER, int GROUP>
__global__ void __launch_bounds__(kThreads, 1)
    qmm_tc_kernel(const QmmParams p, int max_rows, const __grid_constant__ CUtensorMap code_map0,
                  const __grid_constant__ CUtensorMap x_map,
                  const __grid_constant__ CUtensorMap code_map1) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const SmemLayout L = make_layout(max_rows, false, slot_row_bytes(BITS));
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + L.bar_offset);
    uint64_t* cempty = cfull + kMaxCodeStages;
    uint64_t* afull = cempty + kMaxCodeStages;
    uint64_t* aempty = afull + kMaxAStages;
    uint64_t* xfull = aempty + kMaxAStages;
    uint64_t* xempty = xfull + kMaxXStages;
    uint64_t* accf = xempty + kMaxXStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t x_base0 = smem_base;
    const uint32_t c_base0 = smem_base + L.c_offset;

    const int warp = threadIdx.x >> 5;
    const int lane = lane_id();

    // ---- which tile this CTA computes
    int e = 0, row_start, rows;
    if (GATHER) {
        if ((int)blockIdx.y >= *p.tile_count) return;  // whole CTA, before any sync
        const MTile t = p.tiles[blockIdx.y];
        e = t.e;
        row_start = t.row_start;
        rows = t.rows;
    } else {
        row_start = blockIdx.y * p.m_tile;
        rows = min(p.m_tile, p.M - row_start);
    }
    const int n_mma = (rows + 15) & ~15;
    const int n0 = blockIdx.x * kTileN;
    const int KB = p.K / kHalfK;                       // 64-wide blocks
    // grid z: the K split (dense form) or the weight set (grouped form: the
    // gate/up pair's second set in z = 1)
    const int set = GATHER ? (int)blockIdx.z : 0;
    const CUtensorMap& code_map = set ? code_map1 : code_map0;
    const uint16_t* const set_scales = set ? p.scales1 : p.scales;
    const uint16_t* const set_biases = set ? p.biases1 : p.biases;
    void* const set_y = set ? p.y1 : p.y;
    const int kb_begin = (GATHER ? 0 : (int)blockIdx.z) * p.kb_per_split;  // in 64-wide blocks
    const int nkb = min(KB, kb_begin + p.kb_per_split) - kb_begin;
    const int nst = (nkb + 1) / 2;                     // 128-wide stages
    const int groups = p.K / GROUP;
    using SG = StageGroups<GROUP>;
    constexpr int kP = SG::kPairs;
    const int SC = L.c_stages;
    constexpr int kStagesPerSlot = slot_row_bytes(BITS) / (kBK * BITS / 8);
    const int SX = L.x_stages;
    // tensor memory: accumulator in columns [0, n_mma), dequantised stages
    // of 64 columns from a0 on
    const int a0 = (n_mma + kAStageCols - 1) / kAStageCols * kAStageCols;
    constexpr int kCols = kTmemCols;
    const int SA = min(kMaxAStages, (kCols - a0) / kAStageCols);

    if (warp == kCodeWarp && lane == 0) {
        prefetch_tmap(&code_map);
        if (!GATHER) {
            // the dense form starts while the previous kernel finishes (see
            // the wait below): have L2 fetch this CTA's first code slot now
            constexpr int kWordsPerBox = kCodeBoxRowBytes / 4;
            const int c0 = kb_begin * (kHalfK * BITS / 32);
            const int words = p.K * BITS / 32;
            for (int b = 0; b < slot_row_bytes(BITS) / kCodeBoxRowBytes; ++b)
                if (c0 + b * kWordsPerBox < words)
                    tma_prefetch_l2_2d(&code_map, c0 + b * kWordsPerBox, n0);
        }
    }
    if (warp == kXWarp0 && lane == 0) prefetch_tmap(&x_map);
    if (threadIdx.x == 0) {
        for (int i = 0; i < SC; ++i) {
            mbar_init(&cfull[i], 1);
            mbar_init(&cempty[i], kDequantThreads / 2 * kStagesPerSlot);  // 128 per stage
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(&afull[i], kDequantThreads / 2);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < SX; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        mbar_init(accf, 1);
        mbar_init_fence();
        if (!GATHER) pdl_launch_dependents();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, (uint32_t)kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // the dense form is a programmatic dependent launch: everything above
    // touched only this CTA's own resources; from here on it reads x, w,
    // scales and biases and writes y, after the previous kernel completed
    if (!GATHER) pdl_wait();

    if (warp == kCodeWarp) {
        // ---------------------------------------------------------------- codes TMA
        // [128 rows x 128 k] packed codes per stage; a box that runs past K
        // is zero-filled, a second half that belongs to the next K split is
        // loaded but never dequantised
        constexpr int kWordsPerSlot = slot_row_bytes(BITS) / 4;
        constexpr int kWordsPerBox = kCodeBoxRowBytes / 4;
        constexpr int kBoxes = slot_row_bytes(BITS) / kCodeBoxRowBytes;
        const int words = p.K * BITS / 32;
        const int nslots = (nst + kStagesPerSlot - 1) / kStagesPerSlot;
        Ring ring(SC);
        int i = 0;
        for (; i < nslots; ++i, ring.next()) {
            if (i >= SC && !warp_wait(&cempty[ring.slot], ring.parity ^ 1, p.wait_budget)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                const int c0 = kb_begin * (kHalfK * BITS / 32) + i * kWordsPerSlot;
                // a box that starts past the end of the row is not loaded
                // (its stages are never dequantised)
                const int nbox = min(kBoxes, (words - c0 + kWordsPerBox - 1) / kWordsPerBox);
                mbar_expect_tx(&cfull[ring.slot], (uint32_t)(nbox * kCodeBoxBytes));
                const uint32_t dst = c_base0 + ring.slot * L.c_bytes;
                for (int b = 0; b < nbox; ++b) {
                    if (GATHER)
                        tma_load_3d(dst + b * kCodeBoxBytes, &code_map, c0 + b * kWordsPerBox, n0,
                                    e, &cfull[ring.slot]);
                    else
                        tma_load_2d(dst + b * kCodeBoxBytes, &code_map, c0 + b * kWordsPerBox, n0,
                                    &cfull[ring.slot]);
                }
            }
            __syncwarp();
        }
        // the slots issued last may still be loading if a consumer gave up
        if (lane == 0 && !drain_ring(cfull, SC, i, SC)) ok = false;
        __syncwarp();
    } else if (warp == kXWarp0) {
        // ---------------------------------------------------------------- activation TMA
        // per 64-wide block, boxes of [x_box_rows x 64] bf16 (128-byte
        // swizzle) stacked to cover the tile's n_mma rows; rows past the end
        // of x read as zero, rows past the tile are never stored
        const int boxes = (n_mma + p.x_box_rows - 1) / p.x_box_rows;
        const uint32_t x_bytes_in = (uint32_t)(boxes * p.x_box_rows * 128);
        Ring ring(SX);
        int q = 0;
        for (; q < nkb; ++q, ring.next()) {
            if (q >= SX && !warp_wait(&xempty[ring.slot], ring.parity ^ 1, p.wait_budget)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_expect_tx(&xfull[ring.slot], x_bytes_in);
                for (int b = 0; b < boxes; ++b)
                    tma_load_2d(x_base0 + ring.slot * L.x_bytes + b * p.x_box_rows * 128, &x_map,
                                (kb_begin + q) * kHalfK, row_start + b * p.x_box_rows,
                                &xfull[ring.slot]);
            }
            __syncwarp();
        }
        if (lane == 0 && !drain_ring(xfull, SX, q, SX)) ok = false;
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        // the whole warp waits (three barriers per stage in one round trip);
        // one elected lane issues the MMAs and the commits
        const uint32_t idesc = umma_idesc_bf16(kTileN, (uint32_t)n_mma);
        Ring ar(SA), xr(SX);
        for (int s = 0; s < nst; ++s, ar.next()) {
            const bool two = 2 * s + 1 < nkb;
            const int x0 = xr.slot;
            const uint32_t p0 = xr.parity;
            xr.next();
            const int x1 = two ? xr.slot : x0;
            const uint32_t p1 = two ? xr.parity : p0;
            if (two) xr.next();
            if (!warp_wait3(&afull[ar.slot], ar.parity, &xfull[x0], p0, &xfull[x1], p1,
                            p.wait_budget)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
                const uint32_t a_col = tmem + (uint32_t)(a0 + ar.slot * kAStageCols);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !two) break;
                    const uint64_t bd = umma_desc_sw128(x_base0 + (h ? x1 : x0) * L.x_bytes);
#pragma unroll
                    for (int j = 0; j < kHalfK / 16; ++j)
                        umma_bf16_tmem_a(tmem, a_col + h * (kAStageCols / 2) + j * 8, bd + 2 * j,
                                         idesc, (s > 0 || h > 0 || j > 0) ? 1u : 0u);
                }
                umma_commit(&aempty[ar.slot]);
                umma_commit(&xempty[x0]);
                if (two) umma_commit(&xempty[x1]);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(accf);  // also after an abort: fires once issued MMAs finish
        __syncwarp();
    } else if (warp < kDequantWarps) {
        // ---------------------------------------------------------------- dequant
        // two groups of four warps take alternate 128-wide stages, so two
        // stages are dequantised at once; thread r handles w row r (its TMEM
        // lane) over the whole stage
        const int r = threadIdx.x & (kTileN - 1);
        const int grp = warp >> 2;
        const int n = n0 + r;
        const bool row_ok = n < p.N;
        const uint16_t* srow = set_scales + (long long)e * p.sb_expert_stride + (long long)n * groups;
        const uint16_t* brow = set_biases + (long long)e * p.sb_expert_stride + (long long)n * groups;
        constexpr int kRowBytes = kBK * BITS / 8;  // codes of one row per stage
        // this warp's 32 TMEM lanes
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // slot and phase of stage s in the code and A rings, advanced by two
        // stages per step (this group's stages), without divisions
        Ring cr(SC), ar(SA);
        int csub = grp;  // stage within the code slot (kStagesPerSlot >= 2)
        if (grp) ar.next();
        auto stage = [&](int s, const uint32_t (&sb)[2 * kP]) -> bool {
            const int cs = cr.slot;
            if (!warp_wait(&cfull[cs], cr.parity, p.wait_budget)) return false;
            // this stage's kRowBytes of row r: box (off / 128), chunks from
            // (off % 128) / 16 on, each at its swizzled place in the line
            const int off = csub * kRowBytes;
            uint4 cw[BITS];
            if (BITS == 3 || BITS == 6) {
                // 48- or 96-byte stages may cross a box: place each 16-byte
                // chunk by its own box
                const uint32_t c_slot = c_base0 + cs * L.c_bytes + r * kCodeBoxRowBytes;
#pragma unroll
                for (int j = 0; j < BITS; ++j) {
                    const int byte = off + 16 * j;
                    cw[j] = ld_shared_v4(c_slot + (uint32_t)((byte >> 7) * kCodeBoxBytes) +
                                         (uint32_t)((((byte >> 4) & 7) ^ (r & 7)) << 4));
                }
            } else {
                const uint32_t c_line = c_base0 + cs * L.c_bytes +
                                        (off / kCodeBoxRowBytes) * kCodeBoxBytes +
                                        r * kCodeBoxRowBytes;
                const int chunk0 = (off % kCodeBoxRowBytes) / 16;
#pragma unroll
                for (int j = 0; j < BITS; ++j)
                    cw[j] = ld_shared_v4(c_line + (uint32_t)(((chunk0 + j) ^ (r & 7)) << 4));
            }
            const int as = ar.slot;
            if (s >= SA && !warp_wait(&aempty[as], ar.parity ^ 1, p.wait_budget)) return false;
            tc_fence_after();
            const uint32_t a_col = t_lane + (uint32_t)(a0 + as * kAStageCols);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (2 * s + h >= nkb) break;  // the second half past this split's K
#pragma unroll
                for (int c = 0; c < 2; ++c) {  // 32 k = 16 columns per store
                    const uint32_t sbits = sb[SG::pair_of(h, c)];
                    const uint32_t bbits = sb[kP + SG::pair_of(h, c)];
                    uint32_t o[16];
                    if (BITS == 3 || BITS == 6) {
                        const uint32_t s2 = sbits | (sbits << 16);
                        const uint32_t b2 = bbits | (bbits << 16);
                        dequant_stream32<BITS>(cw, (2 * h + c) * BITS, s2, b2, o);
                    } else if (BITS == 2) {
                        const uint32_t s2 = sbits | (sbits << 16);
                        const uint32_t b2 = bbits | (bbits << 16);
                        const uint4 cv = cw[h];  // 64 codes: words 0-1 are chunk 0
                        const uint32_t wd[2] = {c ? cv.z : cv.x, c ? cv.w : cv.y};
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            uint32_t q8[8];
                            dequant_word2(wd[j], s2, b2, q8);
#pragma unroll
                            for (int t = 0; t < 8; ++t) o[j * 8 + t] = q8[t];
                        }
                    } else if (BITS == 4) {
                        const uint32_t s2 = sbits | (sbits << 16);
                        const uint32_t b2 = bbits | (bbits << 16);
                        const uint4 cv = cw[h * 2 + c];
                        const uint32_t wd[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t q4[4];
                            dequant_word4(wd[j], s2, b2, q4);
#pragma unroll
                            for (int t = 0; t < 4; ++t) o[j * 4 + t] = q4[t];
                        }
                    } else {
                        const float sf = bf16_bits_to_float(sbits);
                        const float bf = bf16_bits_to_float(bbits);
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const uint4 cv = cw[h * 4 + c * 2 + q];
                            const uint32_t wd[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint32_t q2[2];
                                dequant_word8(wd[j], sf, bf, q2);
                                o[q * 8 + j * 2] = q2[0];
                                o[q * 8 + j * 2 + 1] = q2[1];
                            }
                        }
                    }
                    tmem_st16(a_col + h * (kAStageCols / 2) + c * 16, o);
                }
            }
            tmem_st_wait();
            // release the code slot only now that the loaded words have been
            // consumed: an arrive placed right after the shared loads let the
            // next TMA overwrite the slot before the loads had returned
            mbar_arrive(&cempty[cs]);
            tc_fence_before();
            mbar_arrive(&afull[as]);
            csub += 2;  // on to stage s + 2
            if (csub >= kStagesPerSlot) {
                csub -= kStagesPerSlot;
                cr.next();
            }
            ar.next();
            ar.next();
            return true;
        };
        // scales then biases of a stage's pairs: {s_0 .. s_kP-1, b_0 .. b_kP-1}
        auto sb_load = [&](int s, uint32_t (&sb)[2 * kP]) {
#pragma unroll
            for (int i = 0; i < kP; ++i) {
                const int b = 2 * s + SG::half_of(i);
                if (row_ok && s < nst && b < nkb) {
                    const int g = SG::group_of(kb_begin + 2 * s, i);
                    sb[i] = __ldg(srow + g);
                    sb[kP + i] = __ldg(brow + g);
                }
            }
        };
        // this group's stages grp, grp + 2, ...; scales loaded a stage ahead
        uint32_t sbA[2 * kP] = {}, sbB[2 * kP] = {};
        sb_load(grp, sbA);
        sb_load(grp + 2, sbB);
        for (int s = grp; s < nst && ok; s += 4) {
            ok = stage(s, sbA);
            sb_load(s + 4, sbA);
            if (!ok || s + 2 >= nst) break;
            ok = stage(s + 2, sbB);
            sb_load(s + 6, sbB);
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && !mbar_wait(accf, 0, p.wait_budget)) ok = false;
        tc_fence_after();
        const int quarter = warp & 3;     // tensor-memory lanes 32*quarter ...
        const int colhalf = warp >> 2;    // 16-column chunks of this parity
        const int lane_row = quarter * 32 + lane;
        const int ny = n0 + lane_row;
        const bool y_ok = ny < p.N;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(set_y);
        if (p.splits == 1) {
            for (int c0 = colhalf * 16; c0 < n_mma; c0 += 32) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
                if (ok && y_ok) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = c0 + j;
                        if (m < rows)
                            y[(long long)(row_start + m) * p.N + ny] =
                                __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
        } else {
            // K split over the CTAs of a cluster: each writes its fp32 partial
            // tile [m][128] into its own shared memory (the rings are idle now:
            // every stage has been consumed by the MMAs)
            const uint32_t part = smem_base;
            for (int c0 = colhalf * 16; c0 < n_mma; c0 += 32) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(part + ((c0 + j) * kTileN + lane_row) * 4),
                                 "r"(v[j])
                                 : "memory");
            }
        }
    }

    if (p.splits > 1) {
        // every thread of every CTA of the cluster takes part in both barriers
        cluster_sync();
        if (warp < kDequantWarps) {
            // rank z sums rows m = z, z + S, ... over all ranks in rank order;
            // a thread takes 4 consecutive columns of one row at a time and
            // issues the remote loads of all S ranks before adding, so each
            // row costs one distributed-shared-memory round trip
            const int rank = (int)cluster_rank();
            const int S = p.splits;  // at most kMaxClusterSplits
            const int c4 = (threadIdx.x & 31) * 4;
            const int ph = threadIdx.x >> 5;
            const int n_out = n0 + c4;
            __nv_bfloat16* y = static_cast<__nv_bfloat16*>(set_y);
            const bool vec_ok = (p.N % 4 == 0) && (n_out + 3 < p.N);
            for (int m = rank + S * ph; m < rows; m += S * kDequantWarps) {
                float4 v[kMaxClusterSplits];
#pragma unroll
                for (int z = 0; z < kMaxClusterSplits; ++z) {
                    v[z] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (z < S)
                        v[z] = ld_cluster_f32x4(map_cluster(smem_base + (m * kTileN + c4) * 4, (uint32_t)z));
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int z = 0; z < kMaxClusterSplits; ++z) {  // rank order
                    if (z < S) {
                        acc.x += v[z].x;
                        acc.y += v[z].y;
                        acc.z += v[z].z;
                        acc.w += v[z].w;
                    }
                }
                if (!ok) continue;
                __nv_bfloat16* yr = y + (long long)(row_start + m) * p.N;
                if (vec_ok) {
                    uint2 pk;
                    pk.x = cvt_bf16x2(acc.x, acc.y);
                    pk.y = cvt_bf16x2(acc.z, acc.w);
                    *reinterpret_cast<uint2*>(yr + n_out) = pk;
                } else {
                    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
                    for (int j = 0; j < 4; ++j)
                        if (n_out + j < p.N) yr[n_out + j] = __float2bfloat16_rn(a4[j]);
                }
            }
        }
        cluster_sync();  // partials stay readable until every rank is done
    }

    if (!ok) flag_status(p.status, MXQ_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        // no MMA may still be writing tensor memory when it is freed: accf
        // fires once every MMA issued has finished (the epilogue may have
        // given up on it under a short budget; this wait takes the default)
        if (lane == 0 && !mbar_wait(accf, 0)) flag_status(p.status, MXQ_DEV_TIMEOUT);
        __syncwarp();
        tmem_dealloc(tmem, (uint32_t)kCols);
    }
}

// ================================================================== persistent form
//
// One CTA per SM walks a fixed sequence of output tiles (tile t = blockIdx.x,
// blockIdx.x + gridDim.x, ...).  Every ring (packed codes, activations,
// dequantised A stages in tensor memory) runs on across tile boundaries, so
// the loads of the next tile start while the current one is still being
// multiplied, and the pipeline fills once per CTA instead of once per tile.
// Four epilogue warps drain the fp32 accumulator of a finished tile while
// the MMAs of the next tile run: with tiles of at most 128 activation rows
// the accumulator is double-buffered in tensor memory.
//
// Warps: 0-7 dequantise (two groups of four take alternate 128-wide stages
// of the global stage sequence), 8 issues the code copies, 9 owns tensor
// memory and issues the MMAs, 10 issues the activation copies, 11-14 are the
// epilogue (warp w reads tensor-memory lanes 32 * (w % 4) ...).
constexpr int kPEpiWarp0 = 11;
constexpr int kPThreads = 15 * 32;
constexpr int kPEpiThreads = 128;
constexpr int kTQ = 4;          // tile-id queue between the code-copy warp and the others
constexpr int kPBarBytes = 64 + kTQ * 20;  // accfull[2], accempty[2], done, tmem slot, abort flag,
                                           // tile queue (ids, full and empty barriers)

struct PTile {
    int e, row_start, rows, n0, n_mma, set;
};

// Tile t of the sequence.  Grouped form: tiles of set 0 (all row tiles x n
// tiles), then those of set 1 (the gate/up pair's second weight set);
// per_set = row tiles x n tiles.
template <bool GATHER>
__device__ __forceinline__ PTile ptile(const QmmParams& p, int t, int m_tiles, int n_tiles,
                                       int per_set = 0) {
    PTile r;
    int nt;
    r.set = 0;
    if (GATHER && per_set > 0 && t >= per_set) {
        r.set = 1;
        t -= per_set;
    }
    if (GATHER) {
        const int lt = t / n_tiles;  // tile of rows (one expert); its n tiles run side by side
        nt = t - lt * n_tiles;
        const MTile mt = p.tiles[lt];
        r.e = mt.e;
        r.row_start = mt.row_start;
        r.rows = mt.rows;
    } else {
        nt = t / m_tiles;  // the M tiles of one n tile run side by side: its codes come from
        const int mt = t - nt * m_tiles;  // HBM once and from L2 for the others
        r.e = 0;
        r.row_start = mt * p.m_tile;
        r.rows = min(p.m_tile, p.M - r.row_start);
    }
    r.n0 = nt * kTileN;
    r.n_mma = (r.rows + 15) & ~15;
    return r;
}

// Bounded wait that also gives up as soon as another role has given up.  The
// first poll does not suspend, and the abort flag and the budget are checked
// before every suspending one, so a budget shorter than one poll gives up at
// the first wait that is not already satisfied.
__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        long long budget) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    do {
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            *abort_flag = 1;
            return false;
        }
    } while (!mbar_try_wait_s(bar, parity, kSuspendNs));
    return true;
}

__device__ __forceinline__ bool warp_wait_ab(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             long long budget) {
    const bool ok = wait_ab(bar, parity, abort_flag, budget);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool warp_wait3_ab(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                              uint64_t* c, uint32_t pc, volatile int* abort_flag,
                                              long long budget) {
    const bool ok = wait_ab(a, pa, abort_flag, budget) && wait_ab(b, pb, abort_flag, budget) &&
                    wait_ab(c, pc, abort_flag, budget);
    return __all_sync(0xffffffffu, ok);
}


// Arrive with a count (the arrivals of stages a partly used code slot never
// holds are made by the threads of the tile's last stage).
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t count) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(count)
        : "memory");
}

template <int BITS, bool GATHER, bool COMPACT, int GROUP>
__global__ void __launch_bounds__(COMPACT ? kThreads : kPThreads, COMPACT ? 2 : 1)
    qmm_persistent_kernel(const QmmParams p, int max_rows, int m_tiles, int n_tiles,
                          const __grid_constant__ CUtensorMap code_map,
                          const __grid_constant__ CUtensorMap x_map,
                          const __grid_constant__ CUtensorMap code_map1) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const SmemLayout L = make_layout(max_rows, COMPACT, slot_row_bytes(BITS, COMPACT));
    constexpr int kCols = COMPACT ? kCompactTmemCols : kTmemCols;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + L.bar_offset);
    uint64_t* cempty = cfull + kMaxCodeStages;
    uint64_t* afull = cempty + kMaxCodeStages;
    uint64_t* aempty = afull + kMaxAStages;
    uint64_t* xfull = aempty + kMaxAStages;
    uint64_t* xempty = xfull + kMaxXStages;
    uint64_t* accfull = xempty + kMaxXStages;   // [2]
    uint64_t* accempty = accfull + 2;           // [2]
    uint64_t* done = accempty + 2;
    uint64_t* tqfull = done + 1;                // [kTQ]
    uint64_t* tqempty = tqfull + kTQ;           // [kTQ]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tqempty + kTQ);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* tq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [kTQ] tile ids
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t x_base0 = smem_base;
    const uint32_t c_base0 = smem_base + L.c_offset;

    const int warp = threadIdx.x >> 5;
    const int lane = lane_id();
    // grouped form: tiles of each weight set (the gate/up pair has two)
    const int per_set = GATHER ? (*p.tile_count) * n_tiles : 0;
    const int total = GATHER ? per_set * p.sets : m_tiles * n_tiles;
    const int KB = p.K / kHalfK;              // 64-wide blocks
    const int nst = (KB + 1) / 2;             // 128-wide stages per tile
    constexpr int kSPS = slot_row_bytes(BITS, COMPACT) / (kBK * BITS / 8);  // stages per code slot
    const int nslots = (nst + kSPS - 1) / kSPS;
    const int groups = p.K / GROUP;
    using SG = StageGroups<GROUP>;
    constexpr int kP = SG::kPairs;
    const int SC = L.c_stages;
    const int SX = L.x_stages;
    // tensor memory: one or two accumulators, then the dequantised A stages
    const int rows16 = (max_rows + 15) & ~15;
    const int acc_cols = (rows16 + kAStageCols - 1) / kAStageCols * kAStageCols;
    // the compact form (two CTAs per SM) has one accumulator: its epilogue is
    // done by the dequant warps, and the SM's other CTA keeps the tensor
    // cores busy meanwhile
    const int acc_bufs = (!COMPACT && acc_cols <= 128) ? 2 : 1;
    const int a0 = acc_bufs * acc_cols;
    const int SA = min(kMaxAStages, (kCols - a0) / kAStageCols);

    if (warp == kCodeWarp && lane == 0) prefetch_tmap(&code_map);
    if (warp == kXWarp0 && lane == 0) prefetch_tmap(&x_map);
    if (threadIdx.x == 0) {
        for (int i = 0; i < SC; ++i) {
            mbar_init(&cfull[i], 1);
            mbar_init(&cempty[i], kDequantThreads / 2 * kSPS);  // 128 per stage
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(&afull[i], kDequantThreads / 2);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < SX; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], 1);
            mbar_init(&accempty[i], COMPACT ? kDequantThreads : kPEpiThreads);
        }
        mbar_init(done, 1);
        // tile queue: filled by the code-copy warp, read by the activation
        // copy warp, the MMA warp, each dequant warp and each epilogue warp
        for (int i = 0; i < kTQ; ++i) {
            mbar_init(&tqfull[i], 1);
            mbar_init(&tqempty[i], 2 + kDequantWarps + (COMPACT ? 0 : 4));
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, (uint32_t)kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    // The tile sequence.  The code-copy warp takes tile i: blockIdx.x first,
    // then (with a tile counter, zeroed by the prepass) the next unclaimed
    // tile, so CTAs that finish early take more; without one, every
    // gridDim.x-th tile.  It passes the id through a kTQ-deep queue; a tile
    // id >= total tells every role to stop.
    auto tq_push = [&](int i, int t) -> bool {
        const int slot = i % kTQ;
        if (i >= kTQ && !warp_wait_ab(&tqempty[slot], (uint32_t)(((i / kTQ) - 1) & 1), abort_flag,
                                      p.wait_budget))
            return false;
        if (lane == 0) {
            tq[slot] = t;
            mbar_arrive(&tqfull[slot]);
        }
        __syncwarp();
        return true;
    };
    auto tq_pop = [&](int i, int* t) -> bool {
        const int slot = i % kTQ;
        if (!warp_wait_ab(&tqfull[slot], (uint32_t)((i / kTQ) & 1), abort_flag, p.wait_budget))
            return false;
        *t = tq[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&tqempty[slot]);
        return true;
    };

    if (warp == kCodeWarp) {
        // ---------------------------------------------------------------- codes TMA
        constexpr int kWordsPerSlot = slot_row_bytes(BITS, COMPACT) / 4;
        constexpr int kWordsPerBox = kCodeBoxRowBytes / 4;
        constexpr int kBoxes = slot_row_bytes(BITS, COMPACT) / kCodeBoxRowBytes;
        const int words = p.K * BITS / 32;
        // grouped form: each expert's codes are read once, so they may leave
        // L2 first (the activation rows, read once per n tile, stay)
        const uint64_t code_policy = l2_policy_evict_first();
        Ring ring(SC);
        int issued = 0;
        for (int i = 0; ok; ++i) {
            int t = blockIdx.x + i * gridDim.x;
            if (i > 0 && p.tile_counter) {
                int c = 0;
                if (lane == 0) c = atomicAdd(p.tile_counter, 1);
                t = gridDim.x + __shfl_sync(0xffffffffu, c, 0);
            }
            if (t > total) t = total;
            if (!tq_push(i, t)) {
                ok = false;
                break;
            }
            if (t >= total) break;
            const PTile ti = ptile<GATHER>(p, t, m_tiles, n_tiles, per_set);
            for (int j = 0; j < nslots; ++j, ring.next(), ++issued) {
                if (issued >= SC && !warp_wait_ab(&cempty[ring.slot], ring.parity ^ 1, abort_flag,
                                                  p.wait_budget)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const int c0 = j * kWordsPerSlot;
                    const int nbox = min(kBoxes, (words - c0 + kWordsPerBox - 1) / kWordsPerBox);
                    mbar_expect_tx(&cfull[ring.slot], (uint32_t)(nbox * kCodeBoxBytes));
                    const uint32_t dst = c_base0 + ring.slot * L.c_bytes;
                    for (int b = 0; b < nbox; ++b) {
                        if (GATHER)
                            tma_load_3d_hint(dst + b * kCodeBoxBytes, ti.set ? &code_map1 : &code_map,
                                             c0 + b * kWordsPerBox, ti.n0, ti.e, &cfull[ring.slot],
                                             code_policy);
                        else
                            tma_load_2d(dst + b * kCodeBoxBytes, &code_map, c0 + b * kWordsPerBox,
                                        ti.n0, &cfull[ring.slot]);
                    }
                }
                __syncwarp();
            }
        }
        // the slots issued last may still be loading if a consumer gave up
        if (lane == 0 && !drain_ring(cfull, SC, issued, SC)) ok = false;
        __syncwarp();
    } else if (warp == kXWarp0) {
        // ---------------------------------------------------------------- activation TMA
        const uint64_t x_policy = l2_policy_evict_last();
        Ring ring(SX);
        int issued = 0;
        for (int i = 0; ok; ++i) {
            int t;
            if (!tq_pop(i, &t)) {
                ok = false;
                break;
            }
            if (t >= total) break;
            const PTile ti = ptile<GATHER>(p, t, m_tiles, n_tiles, per_set);
            const int boxes = (ti.n_mma + p.x_box_rows - 1) / p.x_box_rows;
            const uint32_t x_bytes_in = (uint32_t)(boxes * p.x_box_rows * 128);
            for (int q = 0; q < KB; ++q, ring.next(), ++issued) {
                if (issued >= SX && !warp_wait_ab(&xempty[ring.slot], ring.parity ^ 1, abort_flag,
                                                  p.wait_budget)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_expect_tx(&xfull[ring.slot], x_bytes_in);
                    for (int b = 0; b < boxes; ++b) {
                        const uint32_t dst = x_base0 + ring.slot * L.x_bytes + b * p.x_box_rows * 128;
                        if (GATHER)
                            tma_load_2d_hint(dst, &x_map, q * kHalfK, ti.row_start + b * p.x_box_rows,
                                             &xfull[ring.slot], x_policy);
                        else
                            tma_load_2d(dst, &x_map, q * kHalfK, ti.row_start + b * p.x_box_rows,
                                        &xfull[ring.slot]);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0 && !drain_ring(xfull, SX, issued, SX)) ok = false;
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        Ring ar(SA), xr(SX);
        for (int i = 0; ok; ++i) {
            int t;
            if (!tq_pop(i, &t)) {
                ok = false;
                break;
            }
            if (t >= total) break;
            const PTile ti = ptile<GATHER>(p, t, m_tiles, n_tiles, per_set);
            const int buf = acc_bufs == 2 ? (i & 1) : 0;
            const int use = acc_bufs == 2 ? (i >> 1) : i;  // earlier tiles on this buffer
            if (use > 0 && !warp_wait_ab(&accempty[buf], (uint32_t)((use - 1) & 1), abort_flag,
                                         p.wait_budget)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t idesc = umma_idesc_bf16(kTileN, (uint32_t)ti.n_mma);
            const uint32_t d_tmem = tmem + (uint32_t)(buf * acc_cols);
            for (int s = 0; s < nst; ++s, ar.next()) {
                const bool two = 2 * s + 1 < KB;
                const int x0 = xr.slot;
                const uint32_t p0 = xr.parity;
                xr.next();
                const int x1 = two ? xr.slot : x0;
                const uint32_t p1 = two ? xr.parity : p0;
                if (two) xr.next();
                if (!warp_wait3_ab(&afull[ar.slot], ar.parity, &xfull[x0], p0, &xfull[x1], p1,
                                   abort_flag, p.wait_budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t a_col = tmem + (uint32_t)(a0 + ar.slot * kAStageCols);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !two) break;
                        const uint64_t bd = umma_desc_sw128(x_base0 + (h ? x1 : x0) * L.x_bytes);
#pragma unroll
                        for (int j = 0; j < kHalfK / 16; ++j)
                            umma_bf16_tmem_a(d_tmem, a_col + h * (kAStageCols / 2) + j * 8, bd + 2 * j,
                                             idesc, (s > 0 || h > 0 || j > 0) ? 1u : 0u);
                    }
                    umma_commit(&aempty[ar.slot]);
                    umma_commit(&xempty[x0]);
                    if (two) umma_commit(&xempty[x1]);
                    if (s == nst - 1) umma_commit(&accfull[buf]);
                }
                __syncwarp();
            }
        }
        // every MMA issued so far has finished before tensor memory is freed
        if (elect_one()) {
            umma_commit(done);
            if (!mbar_wait(done, 0)) ok = false;  // default budget: these MMAs were issued
        }
        __syncwarp();
    } else if (!COMPACT && warp >= kPEpiWarp0) {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;  // tensor-memory lanes 32 * quarter ...
        const int lane_row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
        for (int i = 0; ok; ++i) {
            int t;
            if (!tq_pop(i, &t)) {
                ok = false;
                break;
            }
            if (t >= total) break;
            const PTile ti = ptile<GATHER>(p, t, m_tiles, n_tiles, per_set);
            const int buf = acc_bufs == 2 ? (i & 1) : 0;
            const int use = acc_bufs == 2 ? (i >> 1) : i;
            if (!warp_wait_ab(&accfull[buf], (uint32_t)(use & 1), abort_flag, p.wait_budget)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int ny = ti.n0 + lane_row;
            const bool y_ok = ny < p.N;
            const uint32_t acc = t_lane + (uint32_t)(buf * acc_cols);
            for (int c0 = 0; c0 < ti.n_mma; c0 += 32) {
                uint32_t v[32];
                tmem_ld16(acc + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                if (c0 + 16 < ti.n_mma) tmem_ld16(acc + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tmem_ld_wait();
                if (y_ok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = c0 + j;
                        if (m < ti.rows)
                            y[(long long)(ti.row_start + m) * p.N + ny] =
                                __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&accempty[buf]);
        }
    } else if (warp < kDequantWarps) {
        // ---------------------------------------------------------------- dequant
        // group g takes the stages whose global index (over all tiles of this
        // CTA) is congruent to g mod 2; thread r handles w row r (its TMEM
        // lane) over the whole stage
        const int r = threadIdx.x & (kTileN - 1);
        const int grp = warp >> 2;
        constexpr int kRowBytes = kBK * BITS / 8;  // codes of one row per stage
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // last code slot of a tile: stages it never holds, whose arrivals the
        // threads of the tile's last stage make
        const int missing = nslots * kSPS - nst;
        Ring cr(SC), ar(SA);
        if (grp) ar.next();
        long long cpos = 0;   // global index of the code slot cr points at
        long long g0 = 0;     // global index of the tile's first stage
        long long tile_i = 0;
        for (int qi = 0; ok; ++qi, ++tile_i, g0 += nst) {
            int t;
            if (!tq_pop(qi, &t)) {
                ok = false;
                break;
            }
            if (t >= total) break;
            const PTile ti = ptile<GATHER>(p, t, m_tiles, n_tiles, per_set);
            const int n = ti.n0 + r;
            const bool row_ok = n < p.N;
            const uint16_t* srow = (ti.set ? p.scales1 : p.scales) + (long long)ti.e * p.sb_expert_stride +
                                   (long long)n * groups;
            const uint16_t* brow = (ti.set ? p.biases1 : p.biases) + (long long)ti.e * p.sb_expert_stride +
                                   (long long)n * groups;
            const int s0 = (int)((grp + g0) & 1);
            int csub = s0;  // stage within the code slot (kSPS >= 2, so s0 < kSPS)
            // scales then biases of a stage's pairs: {s_0 .. s_kP-1, b_0 .. b_kP-1}
            auto sb_load = [&](int s, uint32_t (&sb)[2 * kP]) {
#pragma unroll
                for (int i = 0; i < kP; ++i) {
                    const int b = 2 * s + SG::half_of(i);
                    sb[i] = 0;
                    sb[kP + i] = 0;
                    if (row_ok && s < nst && b < KB) {
                        const int g = SG::group_of(2 * s, i);
                        sb[i] = __ldg(srow + g);
                        sb[kP + i] = __ldg(brow + g);
                    }
                }
            };
            auto stage = [&](int s, const uint32_t (&sb)[2 * kP]) -> bool {
                const int cs = cr.slot;
                if (!warp_wait_ab(&cfull[cs], cr.parity, abort_flag, p.wait_budget)) return false;
                const int off = csub * kRowBytes;
                uint4 cw[BITS];
                if (BITS == 3 || BITS == 6) {
                    // 48- or 96-byte stages may cross a box
                    const uint32_t c_slot = c_base0 + cs * L.c_bytes + r * kCodeBoxRowBytes;
#pragma unroll
                    for (int j = 0; j < BITS; ++j) {
                        const int byte = off + 16 * j;
                        cw[j] = ld_shared_v4(c_slot + (uint32_t)((byte >> 7) * kCodeBoxBytes) +
                                             (uint32_t)((((byte >> 4) & 7) ^ (r & 7)) << 4));
                    }
                } else {
                    const uint32_t c_line = c_base0 + cs * L.c_bytes +
                                            (off / kCodeBoxRowBytes) * kCodeBoxBytes +
                                            r * kCodeBoxRowBytes;
                    const int chunk0 = (off % kCodeBoxRowBytes) / 16;
#pragma unroll
                    for (int j = 0; j < BITS; ++j)
                        cw[j] = ld_shared_v4(c_line + (uint32_t)(((chunk0 + j) ^ (r & 7)) << 4));
                }
                const int as = ar.slot;
                if (g0 + s >= SA &&
                    !warp_wait_ab(&aempty[as], ar.parity ^ 1, abort_flag, p.wait_budget))
                    return false;
                tc_fence_after();
                const uint32_t a_col = t_lane + (uint32_t)(a0 + as * kAStageCols);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (2 * s + h >= KB) break;  // a last half-stage when K / 64 is odd
#pragma unroll
                    for (int c = 0; c < 2; ++c) {  // 32 k = 16 columns per store
                        const uint32_t sbits = sb[SG::pair_of(h, c)];
                        const uint32_t bbits = sb[kP + SG::pair_of(h, c)];
                        uint32_t o[16];
                        if (BITS == 3 || BITS == 6) {
                            const uint32_t s2 = sbits | (sbits << 16);
                            const uint32_t b2 = bbits | (bbits << 16);
                            dequant_stream32<BITS>(cw, (2 * h + c) * BITS, s2, b2, o);
                        } else if (BITS == 2) {
                            const uint32_t s2 = sbits | (sbits << 16);
                            const uint32_t b2 = bbits | (bbits << 16);
                            const uint4 cv = cw[h];  // 64 codes: words 0-1 are chunk 0
                            const uint32_t wd[2] = {c ? cv.z : cv.x, c ? cv.w : cv.y};
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                uint32_t q8[8];
                                dequant_word2(wd[j], s2, b2, q8);
#pragma unroll
                                for (int u = 0; u < 8; ++u) o[j * 8 + u] = q8[u];
                            }
                        } else if (BITS == 4) {
                            const uint32_t s2 = sbits | (sbits << 16);
                            const uint32_t b2 = bbits | (bbits << 16);
                            const uint4 cv = cw[h * 2 + c];
                            const uint32_t wd[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint32_t q4[4];
                                dequant_word4(wd[j], s2, b2, q4);
#pragma unroll
                                for (int u = 0; u < 4; ++u) o[j * 4 + u] = q4[u];
                            }
                        } else {
                            const float sf = bf16_bits_to_float(sbits);
                            const float bf = bf16_bits_to_float(bbits);
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const uint4 cv = cw[h * 4 + c * 2 + q];
                                const uint32_t wd[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    uint32_t q2[2];
                                    dequant_word8(wd[j], sf, bf, q2);
                                    o[q * 8 + j * 2] = q2[0];
                                    o[q * 8 + j * 2 + 1] = q2[1];
                                }
                            }
                        }
                        tmem_st16(a_col + h * (kAStageCols / 2) + c * 16, o);
                    }
                }
                tmem_st_wait();
                // release the code slot once its words are consumed; the last
                // stage of the tile also makes the arrivals of the stages its
                // slot never holds
                mbar_arrive_n(&cempty[cs], s == nst - 1 ? 1u + (uint32_t)missing : 1u);
                tc_fence_before();
                mbar_arrive(&afull[as]);
                csub += 2;
                if (csub >= kSPS) {
                    csub -= kSPS;
                    cr.next();
                    ++cpos;
                }
                ar.next();
                ar.next();
                return true;
            };
            // this group's stages s0, s0 + 2, ...: two scale/bias buffers,
            // each reloaded (two of this group's stages ahead) right after
            // its use, so no register copy ever waits on a pending load
            uint32_t sbA[2 * kP], sbB[2 * kP];
            sb_load(s0, sbA);
            sb_load(s0 + 2, sbB);
            for (int s = s0; s < nst && ok; s += 4) {
                ok = stage(s, sbA);
                sb_load(s + 4, sbA);
                if (!ok || s + 2 >= nst) break;
                ok = stage(s + 2, sbB);
                sb_load(s + 6, sbB);
            }
            // on to the next tile's first code slot
            while (ok && cpos < (tile_i + 1) * nslots) {
                cr.next();
                ++cpos;
            }
            if (COMPACT && ok) {
                // epilogue of this tile: warp w reads tensor-memory lanes
                // 32 * (w % 4) ... and every other 16-column chunk
                if (!warp_wait_ab(&accfull[0], (uint32_t)(tile_i & 1), abort_flag, p.wait_budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int quarter = warp & 3;
                const int colhalf = warp >> 2;
                const int ny = ti.n0 + quarter * 32 + lane;
                const bool y_ok = ny < p.N;
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
                __nv_bfloat16* y = static_cast<__nv_bfloat16*>(ti.set ? p.y1 : p.y);
                for (int c0 = colhalf * 16; c0 < ti.n_mma; c0 += 32) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_ld_wait();
                    if (y_ok) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = c0 + j;
                            if (m < ti.rows)
                                y[(long long)(ti.row_start + m) * p.N + ny] =
                                    __float2bfloat16_rn(__uint_as_float(v[j]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&accempty[0]);
            }
        }
    }

    // a role that gave up, or a drain that ran out of its budget
    if (!ok || (threadIdx.x == 0 && *abort_flag)) flag_status(p.status, MXQ_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)kCols);
    }
}

template <int BITS, bool GATHER, bool COMPACT, int GROUP>
cudaError_t launch_persistent(const QmmParams& p, int max_rows, int m_tiles, int n_tiles,
                              int grid, const CUtensorMap& cm, const CUtensorMap& xm,
                              const CUtensorMap& cm1, cudaStream_t stream) {
    const SmemLayout L = make_layout(max_rows, COMPACT, slot_row_bytes(BITS, COMPACT));
    const int smem = L.total + kPBarBytes;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(qmm_persistent_kernel<BITS, GATHER, COMPACT, GROUP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               232448);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    if (smem > 232448) return cudaErrorInvalidConfiguration;
    qmm_persistent_kernel<BITS, GATHER, COMPACT, GROUP>
        <<<grid, COMPACT ? kThreads : kPThreads, smem, stream>>>(p, max_rows, m_tiles, n_tiles, cm,
                                                                 xm, cm1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ host side

EncodeTiledFn encode_fn() { return tensor_map_encoder(); }

template <int BITS, bool GATHER, int GROUP>
cudaError_t launch_variant(const QmmParams& p, int grid_m, int max_rows, const CUtensorMap& cm,
                           const CUtensorMap& xm, const CUtensorMap& cm1, cudaStream_t stream) {
    const SmemLayout L = make_layout(max_rows, false, slot_row_bytes(BITS));
    // the shared-memory opt-in is per device; do it once each
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(qmm_tc_kernel<BITS, GATHER, GROUP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               232448);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    if (L.total > 232448) return cudaErrorInvalidConfiguration;  // cannot happen for rows <= 256
    // z: the K splits (dense form, a cluster) or the weight sets (grouped form)
    const dim3 grid((p.N + kTileN - 1) / kTileN, grid_m, GATHER ? (p.sets > 1 ? p.sets : 1) : p.splits);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = p.splits;  // the K splits of one tile form a cluster
    // the dense form may start while the previous kernel finishes (it waits
    // before touching global memory); the grouped form reads the tile table
    // the previous kernel writes, so it starts after it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = GATHER ? 1 : 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, qmm_tc_kernel<BITS, GATHER, GROUP>, p, max_rows, cm, xm,
                                         cm1);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// Launch form for one group size: persistent (dense, every width; grouped 2-
// and 4-bit compact), else one CTA per tile (dense with a K split; grouped 3-,
// 6- and 8-bit).
template <int GROUP>
cudaError_t launch_group(const QmmParams& p, int bits, bool gather, int grid_m,
                         int max_rows_per_tile, const CUtensorMap& cm, const CUtensorMap& xm,
                         const CUtensorMap& cm1, cudaStream_t stream) {
    if (p.persistent) {
        const int n_tiles = (p.N + kTileN - 1) / kTileN;
        if (gather) {
            // grouped, 2- or 4-bit, short tiles: two persistent CTAs per SM
            if (!compact_mode(bits, max_rows_per_tile, true)) return cudaErrorNotSupported;
            return bits == 2 ? launch_persistent<2, true, true, GROUP>(p, max_rows_per_tile, 0,
                                                                       n_tiles, p.grid_ctas, cm, xm, cm1,
                                                                       stream)
                             : launch_persistent<4, true, true, GROUP>(p, max_rows_per_tile, 0,
                                                                       n_tiles, p.grid_ctas, cm, xm, cm1,
                                                                       stream);
        }
        if (bits == 2)
            return launch_persistent<2, false, false, GROUP>(p, max_rows_per_tile, p.m_tiles,
                                                             n_tiles, p.grid_ctas, cm, xm, cm1, stream);
        if (bits == 3)
            return launch_persistent<3, false, false, GROUP>(p, max_rows_per_tile, p.m_tiles,
                                                             n_tiles, p.grid_ctas, cm, xm, cm1, stream);
        if (bits == 6)
            return launch_persistent<6, false, false, GROUP>(p, max_rows_per_tile, p.m_tiles,
                                                             n_tiles, p.grid_ctas, cm, xm, cm1, stream);
        return bits == 4 ? launch_persistent<4, false, false, GROUP>(
                               p, max_rows_per_tile, p.m_tiles, n_tiles, p.grid_ctas, cm, xm, cm1, stream)
                         : launch_persistent<8, false, false, GROUP>(
                               p, max_rows_per_tile, p.m_tiles, n_tiles, p.grid_ctas, cm, xm, cm1, stream);
    }
    if (bits == 2) {
        if (gather) return cudaErrorNotSupported;  // 2-bit grouped calls are persistent (above)
        return launch_variant<2, false, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
    }
    if (bits == 3)
        return gather ? launch_variant<3, true, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream)
                      : launch_variant<3, false, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
    if (bits == 6)
        return gather ? launch_variant<6, true, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream)
                      : launch_variant<6, false, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
    if (bits == 4) {
        if (gather) return cudaErrorNotSupported;  // 4-bit grouped calls are persistent (above)
        return launch_variant<4, false, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
    }
    return gather ? launch_variant<8, true, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream)
                  : launch_variant<8, false, GROUP>(p, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

cudaError_t launch_qmm_tc(const QmmParams& p, int bits, int grid_m, int max_rows_per_tile,
                          cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const bool gather = p.tiles != nullptr;
    // packed codes: words along K, rows n, experts
    CUtensorMap cm, xm, cm1;
    const cuuint64_t words = (cuuint64_t)p.K * bits / 32;
    const cuuint32_t box_words = kCodeBoxRowBytes / 4;    // 128 bytes of each row
    const cuuint32_t estr[3] = {1, 1, 1};
    if (gather) {
        const cuuint64_t dims[3] = {words, (cuuint64_t)p.N, (cuuint64_t)p.E};
        const cuuint64_t strides[2] = {words * 4, words * 4 * (cuuint64_t)p.N};
        const cuuint32_t box[3] = {box_words, (cuuint32_t)kTileN, 1};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(p.w), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // the gate/up pair's second weight set: same shape, its own map
        if (p.sets > 1 &&
            enc(&cm1, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(p.w1), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t dims[2] = {words, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {words * 4};
        const cuuint32_t box[2] = {box_words, (cuuint32_t)kTileN};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(p.w), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // activation rows: [x_rows, K] bf16 (the sorted copy in the grouped form)
    const cuuint64_t xdims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.x_rows};
    const cuuint64_t xstrides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t xbox[2] = {(cuuint32_t)kHalfK, (cuuint32_t)p.x_box_rows};
    if (enc(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), xdims, xstrides, xbox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (!(gather && p.sets > 1)) cm1 = cm;  // one weight set: the second map is never read
    QmmParams q = p;
    q.wait_budget = wait_budget_cycles();
    switch (q.group) {
        case 32: return launch_group<32>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
        case 64: return launch_group<64>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
        case 128: return launch_group<128>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, cm1, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mxq
