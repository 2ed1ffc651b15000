// Quantized GEMM on the sm_103a tensor cores for weights stored [K, N]: row k
// of w holds the codes of every output column n as one little-endian bit
// stream, and each group is G consecutive n of one row, so
//
//     y[m, n] = sum_k x[m, k] * (s[k, n/G] * q[k, n] + b[k, n/G]),
//
// the second operand layout the grouped GEMM is checked in (mlxcel PR #1562,
// What changed).  Dense and sorted-MoE forms.
//
// In this layout one code word holds consecutive n of one k, so a word
// dequantises into 16 bytes (8 bf16) that are contiguous along n: the natural
// tensor-core operand is MN-major.  Per 64-wide block of k:
//  * a TMA copy brings the block's codes of the CTA's 128 columns ([64 rows
//    of k] x [128 * bits / 8 bytes]) into a ring of code slots, and another
//    the activation tile (128-byte swizzle, the MMA's B operand, K-major);
//  * a group of eight dequant warps (two groups, on alternate blocks) turns
//    the codes into bf16 w^ = s*q + b (one rounding, as in the [N, K]
//    kernels) and stores them into a shared-memory A stage
//    in the MN-major 128-byte-swizzled layout: 64-column atoms of 8 k rows x
//    128 bytes, 16-byte chunk c of row r at chunk c ^ r; the two atoms along
//    n are 1024 bytes apart (the descriptor's leading byte offset) and the
//    8-row atoms along k 2048 bytes apart (its stride byte offset);
//  * one elected lane issues four 128 x N x 16 tcgen05.mma with A read from
//    shared memory ("transpose A" set in the instruction descriptor) and the
//    fp32 accumulator in tensor memory; the epilogue reads it back with
//    tcgen05.ld and stores bf16.
// With few tiles (small M), K is split over the CTAs of a cluster and the
// fp32 partials are added through distributed shared memory in rank order.
//
// Every pipeline wait is bounded by the kernel's wait budget; the copy warps
// wait for their issued copies and the MMA warp for its MMAs before the CTA
// exits or frees tensor memory (default budget), whatever happened.
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

constexpr int kDequantWarps = 16;    // warps 0-15: dequant, then epilogue
constexpr int kDequantThreads = kDequantWarps * 32;
constexpr int kGroups = 2;                       // dequant groups taking stages in turn
constexpr int kGroupWarps = kDequantWarps / kGroups;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kCodeWarp = 16;        // codes TMA
constexpr int kMmaWarp = 17;         // TMEM owner, MMA issue
constexpr int kXWarp = 18;           // activation TMA
constexpr int kThreads = 19 * 32;
constexpr int kTileN = 128;          // output columns per CTA (MMA M)
constexpr int kBK = 64;              // k per stage (one activation swizzle atom)
constexpr int kAStageBytes = kTileN * kBK * 2;  // 16 KB of bf16, MN-major
constexpr int kAtomMN = 1024;        // bytes between the two 64-column atoms
constexpr int kAtomK = 2048;         // bytes between 8-row atoms along k
constexpr int kAStages = 4;
constexpr int kMaxCodeStages = 8;
constexpr int kMaxXStages = 8;
constexpr int kSmemBudget = 224 * 1024;
constexpr int kMaxClusterSplits = 8; // K splits per tile: the portable cluster size

struct KnLayout {
    int x_bytes, x_stages;   // activation ring at 0 (one 64-wide atom column per slot)
    int a_offset;            // A stages after it
    int c_bytes, c_stages;   // code ring after the A stages
    int c_offset;
    int bar_offset, total;
};

__host__ __device__ inline KnLayout make_kn_layout(int max_rows, int bits) {
    KnLayout L;
    const int rows16 = (max_rows + 15) & ~15;
    L.x_bytes = (rows16 / 8) * 1024;          // 128 B per row, 8-row atoms
    L.c_bytes = kBK * kTileN * bits / 8;      // 2, 4 or 8 KB
    int room = kSmemBudget - kAStages * kAStageBytes;
    L.c_stages = 4;
    room -= L.c_stages * L.c_bytes;
    L.x_stages = room / L.x_bytes;
    if (L.x_stages > kMaxXStages) L.x_stages = kMaxXStages;
    if (L.x_stages < 2) L.x_stages = 2;
    room -= L.x_stages * L.x_bytes;
    while (L.c_stages < kMaxCodeStages && room >= L.c_bytes) {
        ++L.c_stages;
        room -= L.c_bytes;
    }
    L.a_offset = L.x_stages * L.x_bytes;
    L.c_offset = L.a_offset + kAStages * kAStageBytes;
    L.bar_offset = L.c_offset + L.c_stages * L.c_bytes;
    // cfull, cempty, afull, aempty, xfull, xempty, accf; tmem base
    L.total = L.bar_offset + (2 * kMaxCodeStages + 2 * kAStages + 2 * kMaxXStages + 1) * 8 + 16;
    // a K split adds fp32 partial tiles [rows16][128] through the rings
    if (L.total < rows16 * kTileN * 4) L.total = rows16 * kTileN * 4;
    L.total += 1024;  // alignment slack
    return L;
}

// Shared-memory descriptor of an MN-major operand in the 128-byte-swizzled
// layout: leading byte offset = bytes between 64-column atoms along M,
// stride byte offset = bytes between 8-row atoms along K; version 1,
// swizzle mode "128B" = 2.
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(kAtomMN >> 4) << 16;
    d |= (uint64_t)(kAtomK >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Byte offset of the 16-byte chunk holding columns [8c, 8c + 8) of row k in
// an A stage.
__device__ __forceinline__ uint32_t a_chunk(int k, int c) {
    return (uint32_t)((c >> 3) * kAtomMN + (k >> 3) * kAtomK + (k & 7) * 128 +
                      (((c & 7) ^ (k & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <int BITS, bool GATHER, int GROUP>
__global__ void __launch_bounds__(kThreads, 1)
    qmm_kn_kernel(const QmmParams p, int max_rows, const __grid_constant__ CUtensorMap code_map,
                  const __grid_constant__ CUtensorMap x_map) {
    static_assert(BITS == 2 || BITS == 4 || BITS == 8, "2-, 4- or 8-bit codes");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const KnLayout L = make_kn_layout(max_rows, BITS);
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + L.bar_offset);
    uint64_t* cempty = cfull + kMaxCodeStages;
    uint64_t* afull = cempty + kMaxCodeStages;
    uint64_t* aempty = afull + kAStages;
    uint64_t* xfull = aempty + kAStages;
    uint64_t* xempty = xfull + kMaxXStages;
    uint64_t* accf = xempty + kMaxXStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t x_base0 = smem_base;
    const uint32_t a_base0 = smem_base + L.a_offset;
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
    const int KB = (p.K + kBK - 1) / kBK;  // a last partial block reads zeros past K
    const int kb_begin = (GATHER ? 0 : (int)blockIdx.z) * p.kb_per_split;
    const int nkb = min(KB, kb_begin + p.kb_per_split) - kb_begin;
    const int SC = L.c_stages;
    const int SX = L.x_stages;
    const int kCols = p.tmem_cols;

    if (warp == kCodeWarp && lane == 0) prefetch_tmap(&code_map);
    if (warp == kXWarp && lane == 0) prefetch_tmap(&x_map);
    if (threadIdx.x == 0) {
        for (int i = 0; i < SC; ++i) {
            mbar_init(&cfull[i], 1);
            mbar_init(&cempty[i], kGroupWarps);
        }
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(&afull[i], kGroupWarps);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < SX; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        mbar_init(accf, 1);
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

    if (warp == kCodeWarp) {
        // ---------------------------------------------------------------- codes TMA
        // one box per stage: 64 rows of k x the tile's 128 columns of codes;
        // columns past N read as zero
        const int x0 = n0 * BITS / 8;  // bytes; a multiple of 32
        Ring ring(SC);
        int q = 0;
        for (; q < nkb; ++q, ring.next()) {
            if (q >= SC &&
                !warp_wait_sleep(&cempty[ring.slot], ring.parity ^ 1, p.wait_budget)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_expect_tx(&cfull[ring.slot], (uint32_t)L.c_bytes);
                const uint32_t dst = c_base0 + ring.slot * L.c_bytes;
                const int k0 = (kb_begin + q) * kBK;
                if (GATHER)
                    tma_load_3d(dst, &code_map, x0, k0, e, &cfull[ring.slot]);
                else
                    tma_load_2d(dst, &code_map, x0, k0, &cfull[ring.slot]);
            }
            __syncwarp();
        }
        // the slots issued last may still be loading if a consumer gave up
        if (lane == 0 && !drain_ring(cfull, SC, q, SC)) ok = false;
        __syncwarp();
    } else if (warp == kXWarp) {
        // ---------------------------------------------------------------- activation TMA
        const int boxes = (n_mma + p.x_box_rows - 1) / p.x_box_rows;
        const uint32_t x_bytes_in = (uint32_t)(boxes * p.x_box_rows * 128);
        Ring ring(SX);
        int q = 0;
        for (; q < nkb; ++q, ring.next()) {
            if (q >= SX &&
                !warp_wait_sleep(&xempty[ring.slot], ring.parity ^ 1, p.wait_budget)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_expect_tx(&xfull[ring.slot], x_bytes_in);
                for (int b = 0; b < boxes; ++b)
                    tma_load_2d(x_base0 + ring.slot * L.x_bytes + b * p.x_box_rows * 128, &x_map,
                                (kb_begin + q) * kBK, row_start + b * p.x_box_rows,
                                &xfull[ring.slot]);
            }
            __syncwarp();
        }
        if (lane == 0 && !drain_ring(xfull, SX, q, SX)) ok = false;
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        const uint32_t idesc = umma_idesc_bf16(kTileN, (uint32_t)n_mma) | (1u << 15);  // A MN-major
        // two stages per round: the MMAs of one round keep the tensor pipe
        // busy while the warp waits for the next round's operands
        Ring ar(kAStages), xr(SX);
        for (int q = 0; q < nkb; q += 2) {
            const bool two = q + 1 < nkb;
            const int a0 = ar.slot, x0 = xr.slot;
            const uint32_t pa0 = ar.parity, px0 = xr.parity;
            ar.next();
            xr.next();
            const int a1 = ar.slot, x1 = xr.slot;
            const uint32_t pa1 = ar.parity, px1 = xr.parity;
            if (two) {
                ar.next();
                xr.next();
            }
            if (!warp_wait_sleep(&afull[a0], pa0, p.wait_budget) ||
                !warp_wait_sleep(&xfull[x0], px0, p.wait_budget) ||
                (two && (!warp_wait_sleep(&afull[a1], pa1, p.wait_budget) ||
                         !warp_wait_sleep(&xfull[x1], px1, p.wait_budget)))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !two) break;
                    const uint32_t a_stage = a_base0 + (h ? a1 : a0) * kAStageBytes;
                    const uint64_t bd = umma_desc_sw128(x_base0 + (h ? x1 : x0) * L.x_bytes);
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j)  // 16 k = two 8-row atoms of A, 32 B of B
                        umma_bf16(tmem, umma_desc_mn_sw128(a_stage + j * 2 * kAtomK), bd + 2 * j,
                                  idesc, (q > 0 || h > 0 || j > 0) ? 1u : 0u);
                }
                umma_commit(&aempty[a0]);
                umma_commit(&xempty[x0]);
                if (two) {
                    umma_commit(&aempty[a1]);
                    umma_commit(&xempty[x1]);
                }
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(accf);  // also after an abort: fires once issued MMAs finish
        __syncwarp();
    } else if (warp < kDequantWarps) {
        // ---------------------------------------------------------------- dequant
        // kGroups groups of warps take the stages in turn (group g: stages g,
        // g + kGroups, ...), so several stages are dequantised at once and
        // each warp has kGroups stage times for one stage.  Each thread takes
        // one row r of the stage's 64 rows of k and 32 columns [32 cb, + 32)
        // of the tile: BITS consecutive code words (one 8-, 16- or two
        // 16-byte loads), one scale and one bias (32 columns aligned to 32 lie
        // in one group, G being 32, 64 or 128), and four 16-byte chunks of A.
        // Warp w of a group covers the 8-row atom 8w .. 8w + 7, all four
        // column blocks; within it, quarter warp q (lanes 8q .. 8q + 7) takes
        // rows {0,1} (or {4,5} for q >= 2) with one pair of column blocks and
        // rows {2,3} (or {6,7}) with the other pair, so that its eight
        // threads' code loads fall on eight different 16-byte bank quads and
        // so do each of their four stores (chunk c of row k sits at quad
        // (c & 7) ^ (k & 7)): no shared-memory bank conflicts.
        constexpr int W = kTileN * BITS / 32;                // words per code row
        constexpr int kColBlocks = kTileN / 32;              // threads per row of k
        static_assert(kBK * kColBlocks == kGroupThreads, "one row block per thread");
        const int grp = warp / kGroupWarps;
        const int t = threadIdx.x % kGroupThreads;
        const int ql = (t >> 3) & 3, l8 = t & 7;       // quarter warp, lane within it
        const int rowpair = l8 >> 2;
        const int r = 8 * (t >> 5) + (ql >> 1) * 4 + rowpair * 2 + ((l8 >> 1) & 1);
        const int cb = (l8 & 1) + 2 * (rowpair ^ (ql & 1));
        const bool col_ok = n0 + cb * 32 < p.N; // columns past N: zero codes, no scale read
        const int groups = p.N / GROUP;         // scale/bias entries per row of k
        // scale and bias of row r of the CTA's first block; a stage moves
        // them kBK rows on
        const long long sb0 = (long long)e * p.sb_expert_stride +
                              ((long long)kb_begin * kBK + r) * groups + (n0 + cb * 32) / GROUP;
        const uint16_t* sp = p.scales + sb0;
        const uint16_t* bp = p.biases + sb0;
        const long long stage_step = (long long)kBK * groups;
        const int k_left0 = p.K - kb_begin * kBK - r;  // rows of k left from row r of block 0
        // 8-bit: the thread's 32 code bytes are two 16-byte halves, read
        // half hx first (hx = r & 1), so that odd and even rows of a quarter
        // warp fall on different bank quads; its store order follows
        const int hx = BITS == 8 ? (r & 1) : 0;
        const uint32_t c_off = (uint32_t)(r * W * 4 + cb * BITS * 4);
        uint32_t a_off[4];  // the A chunk that the thread's i-th store fills
#pragma unroll
        for (int i = 0; i < 4; ++i) a_off[i] = a_chunk(r, cb * 4 + (i ^ (2 * hx)));
        // scale/bias pair of stage q, loaded two of the group's stages
        // (2 * kGroups stage times) before its use
        auto sb_load = [&](int q, uint32_t& sl, uint32_t& bl) {
            sl = 0u;
            bl = 0u;
            if (col_ok && q < nkb && q * kBK < k_left0) {
                sl = __ldg(sp + (long long)q * stage_step);
                bl = __ldg(bp + (long long)q * stage_step);
            }
        };
        Ring cr(SC), ar(kAStages);
        for (int i = 0; i < grp; ++i) {
            cr.next();
            ar.next();
        }
        // stage q with its scale/bias pair (sc, bc); loads the pair of stage
        // q + 2 * kGroups into (sn, bn)
        auto stage = [&](int q, uint32_t sc, uint32_t bc, uint32_t& sn, uint32_t& bn) -> bool {
            sb_load(q + 2 * kGroups, sn, bn);
            if (!warp_wait_sleep(&cfull[cr.slot], cr.parity, p.wait_budget)) return false;
            const uint32_t c_at = c_base0 + cr.slot * L.c_bytes + c_off;
            uint32_t wd[BITS];
            if (BITS == 2) {
                asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                             : "=r"(wd[0]), "=r"(wd[1])
                             : "r"(c_at)
                             : "memory");
            } else {
#pragma unroll
                for (int h = 0; h < BITS / 4; ++h) {
                    const uint4 v = ld_shared_v4(c_at + (uint32_t)((h ^ hx) * 16));
                    wd[4 * h] = v.x;
                    wd[4 * h + 1] = v.y;
                    wd[4 * h + 2] = v.z;
                    wd[4 * h + 3] = v.w;
                }
            }
            if (q >= kAStages &&
                !warp_wait_sleep(&aempty[ar.slot], ar.parity ^ 1, p.wait_budget))
                return false;
            const uint32_t a_stage = a_base0 + ar.slot * kAStageBytes;
            if (BITS == 8) {
                const float s = bf16_bits_to_float(sc), b = bf16_bits_to_float(bc);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t o0[2], o1[2];
                    dequant_word8(wd[2 * i], s, b, o0);
                    dequant_word8(wd[2 * i + 1], s, b, o1);
                    st_shared_v4(a_stage + a_off[i], o0[0], o0[1], o1[0], o1[1]);
                }
            } else {
                // both halves of a bf16x2 take the scale and bias
                const uint32_t sw = prmt(sc, 0u, 0x1010u), bw = prmt(bc, 0u, 0x1010u);
                if (BITS == 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t o[4];
                        dequant_word4(wd[i], sw, bw, o);
                        st_shared_v4(a_stage + a_off[i], o[0], o[1], o[2], o[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint32_t o[8];
                        dequant_word2(wd[j], sw, bw, o);
                        st_shared_v4(a_stage + a_off[2 * j], o[0], o[1], o[2], o[3]);
                        st_shared_v4(a_stage + a_off[2 * j + 1], o[4], o[5], o[6], o[7]);
                    }
                }
            }
            // the tensor cores read the stage through the async proxy; the
            // code slot is released only now that its words have been used
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&cempty[cr.slot]);
                mbar_arrive(&afull[ar.slot]);
            }
#pragma unroll
            for (int i = 0; i < kGroups; ++i) {
                cr.next();
                ar.next();
            }
            return true;
        };
        // three register pairs in turn (the loop is unrolled by three), so
        // no pair is ever copied
        uint32_t sA, bA, sB, bB, sC, bC;
        sb_load(grp, sA, bA);
        sb_load(grp + kGroups, sB, bB);
        for (int q = grp; q < nkb && ok; q += 3 * kGroups) {
            ok = stage(q, sA, bA, sC, bC);
            if (!ok || q + kGroups >= nkb) break;
            ok = stage(q + kGroups, sB, bB, sA, bA);
            if (!ok || q + 2 * kGroups >= nkb) break;
            ok = stage(q + 2 * kGroups, sC, bC, sB, bB);
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && !mbar_wait_sleep(accf, 0, p.wait_budget)) ok = false;
        tc_fence_after();
        const int quarter = warp & 3;     // tensor-memory lanes 32*quarter ...
        const int colq = warp >> 2;       // every fourth 16-column chunk from colq
        const int lane_row = quarter * 32 + lane;
        const int ny = n0 + lane_row;
        const bool y_ok = ny < p.N;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
        if (p.splits == 1) {
            for (int c0 = colq * 16; c0 < n_mma; c0 += 16 * (kDequantWarps / 4)) {
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
            // K split: each CTA writes its fp32 partial tile [m][128] into its
            // own shared memory (every stage has been consumed by the MMAs)
            const uint32_t part = smem_base;
            for (int c0 = colq * 16; c0 < n_mma; c0 += 16 * (kDequantWarps / 4)) {
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
            // a thread loads all S ranks' partials of its 4 columns before
            // adding them, one remote round trip per row
            const int rank = (int)cluster_rank();
            const int S = p.splits;  // at most kMaxClusterSplits
            const int c4 = (threadIdx.x & 31) * 4;
            const int ph = threadIdx.x >> 5;
            const int n_out = n0 + c4;
            __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
            const bool vec_ok = n_out + 3 < p.N;  // N % 64 == 0: four columns stay together
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
                if (ok && vec_ok) {
                    uint2 pk;
                    pk.x = cvt_bf16x2(acc.x, acc.y);
                    pk.y = cvt_bf16x2(acc.z, acc.w);
                    *reinterpret_cast<uint2*>(y + (long long)(row_start + m) * p.N + n_out) = pk;
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
        // accf fires once every MMA issued has finished; tensor memory is
        // freed only after that (default budget)
        if (lane == 0 && !mbar_wait(accf, 0)) flag_status(p.status, MXQ_DEV_TIMEOUT);
        __syncwarp();
        tmem_dealloc(tmem, (uint32_t)kCols);
    }
}

template <int BITS, bool GATHER, int GROUP>
cudaError_t launch_kn(const QmmParams& p, int grid_m, int max_rows, const CUtensorMap& cm,
                      const CUtensorMap& xm, cudaStream_t stream) {
    const KnLayout L = make_kn_layout(max_rows, BITS);
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(qmm_kn_kernel<BITS, GATHER, GROUP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    if (L.total > 232448) return cudaErrorInvalidConfiguration;
    // the partial tiles of a K split must stay below the barriers
    if (((max_rows + 15) & ~15) * kTileN * 4 > L.bar_offset) return cudaErrorInvalidConfiguration;
    const dim3 grid((p.N + kTileN - 1) / kTileN, grid_m, GATHER ? 1 : p.splits);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = GATHER ? 1 : p.splits;  // the K splits of one tile form a cluster
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, qmm_kn_kernel<BITS, GATHER, GROUP>, p, max_rows, cm, xm);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

template <int GROUP>
cudaError_t launch_kn_group(const QmmParams& p, int bits, bool gather, int grid_m, int max_rows,
                            const CUtensorMap& cm, const CUtensorMap& xm, cudaStream_t stream) {
    if (gather) {
        if (bits == 2) return launch_kn<2, true, GROUP>(p, grid_m, max_rows, cm, xm, stream);
        if (bits == 4) return launch_kn<4, true, GROUP>(p, grid_m, max_rows, cm, xm, stream);
        return launch_kn<8, true, GROUP>(p, grid_m, max_rows, cm, xm, stream);
    }
    if (bits == 2) return launch_kn<2, false, GROUP>(p, grid_m, max_rows, cm, xm, stream);
    if (bits == 4) return launch_kn<4, false, GROUP>(p, grid_m, max_rows, cm, xm, stream);
    return launch_kn<8, false, GROUP>(p, grid_m, max_rows, cm, xm, stream);
}

}  // namespace

cudaError_t launch_qmm_kn(const QmmParams& p, int bits, int grid_m, int max_rows_per_tile,
                          cudaStream_t stream) {
    if (bits != 2 && bits != 4 && bits != 8) return cudaErrorInvalidValue;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const bool gather = p.tiles != nullptr;
    // packed codes as bytes: [E][K][N * bits / 8]; box = the tile's 128
    // columns x 64 rows of k
    CUtensorMap cm, xm;
    const cuuint64_t row_bytes = (cuuint64_t)p.N * bits / 8;
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint32_t box[3] = {(cuuint32_t)(kTileN * bits / 8), (cuuint32_t)kBK, 1};
    if (gather) {
        const cuuint64_t dims[3] = {row_bytes, (cuuint64_t)p.K, (cuuint64_t)p.E};
        const cuuint64_t strides[2] = {row_bytes, row_bytes * (cuuint64_t)p.K};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint32_t*>(p.w), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)p.K};
        const cuuint64_t strides[1] = {row_bytes};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(p.w), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // activation rows: [x_rows, K] bf16, 64-wide boxes with 128-byte swizzle
    const cuuint64_t xdims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.x_rows};
    const cuuint64_t xstrides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t xbox[2] = {(cuuint32_t)kBK, (cuuint32_t)p.x_box_rows};
    if (enc(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), xdims, xstrides, xbox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    QmmParams q = p;
    q.wait_budget = wait_budget_cycles();
    switch (q.group) {
        case 32: return launch_kn_group<32>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, stream);
        case 64: return launch_kn_group<64>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, stream);
        case 128: return launch_kn_group<128>(q, bits, gather, grid_m, max_rows_per_tile, cm, xm, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mxq
