// Quantized GEMM on the sm_103a tensor cores: y = x . w^T with w dequantised
// on the fly (w^ = s*q + b per 64-wide group), dense and sorted-MoE forms.
//
// Prior art: the qmm_naive and grouped-GEMM kernels profiled in mlxcel issue
// #1536 (Baseline profile table; Diagnosis items 1, 4 and 5) and PR #1562
// (Summary: the sorted-MoE prefill path over B = tokens * top_k rows).  Those
// ran FP32 FMA on CUDA cores; this kernel is built for tcgen05 instead:
//
//  * swap-AB: the MMA's M side is 128 rows of w (output columns n), its N side
//    is a tile of up to 256 activation rows, so a 36-row expert segment or a
//    single decode row still fills the 128-row tensor-core tile;
//  * per 64-wide K block (one quantisation group), producer warps copy the
//    packed codes and the activation rows (gathered through row_src in the
//    grouped form) into a shared-memory ring with cp.async; four dequant warps
//    turn codes into bf16 w^ = s*q + b (one bf16 rounding) written directly in
//    the 128-byte-swizzled K-major layout the tensor core reads; one thread
//    issues four 128xNx16 tcgen05.mma per block into fp32 tensor memory;
//  * the dequant warps then read the accumulators back with tcgen05.ld and
//    store bf16 (or, with K split across CTAs, fp32 partials that the last
//    CTA of the tile sums in a fixed order: results do not depend on timing).
//
// Every wait on an mbarrier is bounded; on expiry the kernel sets
// MXQ_DEV_TIMEOUT, stops issuing work, drains what it issued and frees its
// tensor memory before returning.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;       // 8 warps
constexpr int kDequantWarps = 4;    // warps 0-3: dequant + epilogue (thread t <-> w row t)
constexpr int kProducerFirst = 4;   // warps 4-6: cp.async producers
constexpr int kProducerThreads = 96;
constexpr int kMmaWarp = 7;         // warp 7: TMEM owner, lane 0 issues MMAs
constexpr int kTileN = 128;         // rows of w per CTA (MMA M)
constexpr int kBK = 64;             // K per pipeline stage (= one group)
constexpr int kMaxStages = 8;
constexpr int kLag = 2;             // stages a producer keeps in flight before signalling
constexpr int kMaxRows = 256;       // activation rows per tile (MMA N <= 256)
constexpr int kSmemBudget = 200 * 1024;

__host__ __device__ constexpr int code_bytes_per_stage(int bits) { return kTileN * kBK * bits / 8; }

struct SmemLayout {
    int stages;
    int a_bytes, x_bytes, c_bytes, stage_bytes;
    int bar_offset;  // after all stages
    int src_offset;  // activation row of each tile row (-1 = zero row)
    int total;
};

__host__ __device__ inline SmemLayout make_layout(int bits, int max_rows) {
    SmemLayout L;
    const int rows16 = (max_rows + 15) & ~15;          // n_mma never exceeds this
    L.a_bytes = kTileN * kBK * 2;                      // 16 KB bf16
    L.x_bytes = (rows16 / 8) * 1024;                   // rows x 128 B, 8-row atoms
    L.c_bytes = code_bytes_per_stage(bits);            // 4 KB or 8 KB
    L.stage_bytes = L.a_bytes + L.x_bytes + L.c_bytes; // multiple of 1024
    int s = kSmemBudget / L.stage_bytes;
    // the producers signal a stage kLag stages late, so the ring needs more
    L.stages = s > kMaxStages ? kMaxStages : (s < kLag + 1 ? kLag + 1 : s);
    L.bar_offset = L.stages * L.stage_bytes;
    // full, afull, empty per stage, accf, tmem base, flag, then source rows
    L.src_offset = L.bar_offset + (3 * kMaxStages + 1) * 8 + 16;
    L.total = L.src_offset + kMaxRows * 4 + 1024 /* alignment slack */;
    return L;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_bf16(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Eight 4-bit codes (one word, lowest k in the lowest nibble) -> four bf16x2
// words (k pairs 0-1, 2-3, 4-5, 6-7) of s*q + b, one rounding each.
__device__ __forceinline__ void dequant_word4(uint32_t wd, uint32_t s2, uint32_t b2,
                                              uint32_t (&out)[4]) {
    const uint32_t lo = wd & 0x0F0F0F0Fu;          // q0 q2 q4 q6
    const uint32_t hi = (wd >> 4) & 0x0F0F0F0Fu;   // q1 q3 q5 q7
    const uint32_t e0 = prmt(lo, hi, 0x5140u);     // q0 q1 q2 q3
    const uint32_t e1 = prmt(lo, hi, 0x7362u);     // q4 q5 q6 q7
    // bf16 0x43qq = 128 + q exactly (q < 128); subtracting 128 is exact
    const uint32_t k128 = 0x43004300u;
    out[0] = hfma2_bf16(hsub2_bf16(prmt(e0, 0x43u, 0x4140u), k128), s2, b2);
    out[1] = hfma2_bf16(hsub2_bf16(prmt(e0, 0x43u, 0x4342u), k128), s2, b2);
    out[2] = hfma2_bf16(hsub2_bf16(prmt(e1, 0x43u, 0x4140u), k128), s2, b2);
    out[3] = hfma2_bf16(hsub2_bf16(prmt(e1, 0x43u, 0x4342u), k128), s2, b2);
}

// Four 8-bit codes (lowest k in the lowest byte) -> two bf16x2 words.  The
// code is exact in fp32 (2^23 + q, minus 2^23), s*q + b is formed by one fp32
// FMA (s*q is exact) and rounded to bf16.
__device__ __forceinline__ void dequant_word8(uint32_t wd, float s, float b, uint32_t (&out)[2]) {
    const float m = 8388608.f;
    const float q0 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7440u)) - m;
    const float q1 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7441u)) - m;
    const float q2 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7442u)) - m;
    const float q3 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7443u)) - m;
    out[0] = cvt_bf16x2(fmaf(s, q0, b), fmaf(s, q1, b));
    out[1] = cvt_bf16x2(fmaf(s, q2, b), fmaf(s, q3, b));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) qmm_tc_kernel(const QmmParams p, int max_rows) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const SmemLayout L = make_layout(BITS, max_rows);
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_offset);
    uint64_t* afull = full + kMaxStages;
    uint64_t* empty = afull + kMaxStages;
    uint64_t* accf = empty + kMaxStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);
    int* src_rows = reinterpret_cast<int*>(smem + L.src_offset);
    const uint32_t smem_base = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = lane_id();

    // ---- which tile this CTA computes
    int e = 0, row_start, rows;
    if (p.tiles) {
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
    const int KB = p.K / kBK;
    const int kb_begin = blockIdx.z * p.kb_per_split;
    const int kb_end = min(KB, kb_begin + p.kb_per_split);
    const int nkb = kb_end - kb_begin;
    const int groups = p.K / 64;
    const long long wpr = (long long)p.K * BITS / 32;  // words per w row
    const uint32_t* wexp = p.w + (long long)e * p.w_expert_stride;
    const uint16_t* sexp = p.scales + (long long)e * p.sb_expert_stride;
    const uint16_t* bexp = p.biases + (long long)e * p.sb_expert_stride;
    const int S = L.stages;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], kProducerThreads);
            mbar_init(&afull[i], kDequantWarps * 32);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accf, 1);
        *last_flag = 0;
        mbar_init_fence();
    }
    for (int r = threadIdx.x; r < n_mma; r += kThreads) {
        int src = -1;
        if (r < rows) {
            const int sr = row_start + r;
            src = p.row_src ? p.row_src[sr] : sr;
            const int limit = p.tiles ? p.T : p.M;
            if (src < 0 || src >= limit) src = -1;  // reported by the prepass; row reads as zero
        }
        src_rows[r] = src;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp >= kProducerFirst && warp < kProducerFirst + 3) {
        // ---------------------------------------------------------------- producers
        const int pt = threadIdx.x - kProducerFirst * 32;
        constexpr int kCodeChunksPerRow = kBK * BITS / 8 / 16;  // 2 or 4
        const int code_chunks = kTileN * kCodeChunksPerRow;
        const int x_chunks = n_mma * 8;
        const int total = code_chunks + x_chunks;
        for (int i = 0; i < nkb; ++i) {
            const int slot = i % S;
            if (i >= S && !mbar_wait(&empty[slot], ((i / S) + 1) & 1)) { ok = false; break; }
            const int kb = kb_begin + i;
            const uint32_t a_base = smem_base + slot * L.stage_bytes;
            const uint32_t x_base = a_base + L.a_bytes;
            const uint32_t c_base = x_base + L.x_bytes;
            for (int c = pt; c < total; c += kProducerThreads) {
                if (c < code_chunks) {
                    const int r = c / kCodeChunksPerRow;
                    const int ch = c % kCodeChunksPerRow;
                    const int n = n0 + r;
                    const bool valid = n < p.N;
                    const uint32_t* src =
                        wexp + (valid ? (long long)n * wpr + (long long)kb * (kBK * BITS / 32) + ch * 4
                                      : 0);
                    cp_async_16(c_base + r * (kCodeChunksPerRow * 16) + ch * 16, src, valid ? 16u : 0u);
                } else {
                    const int xc = c - code_chunks;
                    const int r = xc >> 3;
                    const int ch = xc & 7;
                    const int src_row = src_rows[r];
                    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(p.x);
                    const void* src = xb + (src_row >= 0 ? (long long)src_row * p.K + kb * kBK + ch * 8 : 0);
                    cp_async_16(x_base + sw128_offset(r, ch), src, src_row >= 0 ? 16u : 0u);
                }
            }
            cp_async_commit();
            if (i >= kLag) {
                cp_async_wait<kLag>();
                fence_proxy_async_smem();
                mbar_arrive(&full[(i - kLag) % S]);
            }
        }
        cp_async_wait<0>();
        if (ok) {
            fence_proxy_async_smem();
            for (int i = (nkb > kLag ? nkb - kLag : 0); i < nkb; ++i) mbar_arrive(&full[i % S]);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(kTileN, (uint32_t)n_mma);
            for (int i = 0; i < nkb; ++i) {
                const int slot = i % S;
                const uint32_t par = (i / S) & 1;
                if (!mbar_wait(&full[slot], par) || !mbar_wait(&afull[slot], par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_base + slot * L.stage_bytes;
                const uint32_t x_base = a_base + L.a_bytes;
                const uint64_t ad = umma_desc_sw128(a_base);
                const uint64_t bd = umma_desc_sw128(x_base);
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j)
                    umma_bf16(tmem, ad + 2 * j, bd + 2 * j, idesc, (i > 0 || j > 0) ? 1u : 0u);
                umma_commit(&empty[slot]);
            }
            umma_commit(accf);  // also after an abort: fires once issued MMAs finish
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- dequant
        const int t = threadIdx.x;  // row of the w tile, lane of tensor memory
        const int n = n0 + t;
        const bool row_ok = n < p.N;
        const uint16_t* srow = sexp + (long long)n * groups;
        const uint16_t* brow = bexp + (long long)n * groups;
        // scale/bias of the block two ahead are loaded while this one is used
        uint32_t sA = 0, bA = 0, sB = 0, bB = 0;
        if (row_ok && nkb > 0) { sA = __ldg(srow + kb_begin); bA = __ldg(brow + kb_begin); }
        if (row_ok && nkb > 1) { sB = __ldg(srow + kb_begin + 1); bB = __ldg(brow + kb_begin + 1); }
        auto stage = [&](int i, uint32_t sbits, uint32_t bbits) -> bool {
            const int slot = i % S;
            if (!mbar_wait(&full[slot], (i / S) & 1)) return false;
            const uint32_t a_base = smem_base + slot * L.stage_bytes;
            const uint32_t c_base = a_base + L.a_bytes + L.x_bytes;
            const uint32_t a_row = a_base + (t >> 3) * 1024 + (t & 7) * 128;
            if (BITS == 4) {
                const uint32_t s2 = sbits | (sbits << 16);
                const uint32_t b2 = bbits | (bbits << 16);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 cw = ld_shared_v4(c_base + t * 32 + h * 16);
                    const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t o[4];
                        dequant_word4(wd[j], s2, b2, o);
                        const int chunk = h * 4 + j;  // 8 k per word = one 16-byte chunk
                        st_shared_v4(a_row + ((chunk ^ (t & 7)) << 4), o[0], o[1], o[2], o[3]);
                    }
                }
            } else {
                const float s = bf16_bits_to_float(sbits);
                const float b = bf16_bits_to_float(bbits);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint4 cw = ld_shared_v4(c_base + t * 64 + h * 16);
                    const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint32_t o0[2], o1[2];
                        dequant_word8(wd[2 * j], s, b, o0);
                        dequant_word8(wd[2 * j + 1], s, b, o1);
                        const int chunk = h * 2 + j;
                        st_shared_v4(a_row + ((chunk ^ (t & 7)) << 4), o0[0], o0[1], o1[0], o1[1]);
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&afull[slot]);
            return true;
        };
        for (int i = 0; i < nkb && ok; i += 2) {
            ok = stage(i, sA, bA);
            if (row_ok && i + 2 < nkb) { sA = __ldg(srow + kb_begin + i + 2); bA = __ldg(brow + kb_begin + i + 2); }
            if (!ok || i + 1 >= nkb) break;
            ok = stage(i + 1, sB, bB);
            if (row_ok && i + 3 < nkb) { sB = __ldg(srow + kb_begin + i + 3); bB = __ldg(brow + kb_begin + i + 3); }
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && !mbar_wait(accf, 0)) ok = false;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
        if (p.splits == 1) {
            for (int c0 = 0; c0 < n_mma; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + c0, r);
                tmem_ld_wait();
                if (ok && row_ok) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = c0 + j;
                        if (m < rows)
                            y[(long long)(row_start + m) * p.N + n] =
                                __float2bfloat16_rn(__uint_as_float(r[j]));
                    }
                }
            }
        } else {
            // fp32 partial [m][128] of this split, then the last split to
            // arrive sums all of them in split order
            const long long tile_id = blockIdx.x + (long long)gridDim.x * blockIdx.y;
            const long long tile_elems = (long long)p.m_tile * kTileN;
            float* mine = p.partial + (tile_id * p.splits + blockIdx.z) * tile_elems;
            for (int c0 = 0; c0 < n_mma; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = c0 + j;
                    if (m < rows) mine[(long long)m * kTileN + t] = __uint_as_float(r[j]);
                }
            }
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"n"(kDequantWarps * 32) : "memory");
            if (t == 0) {
                const int prev = atomicAdd(p.counters + tile_id, 1);
                *last_flag = (prev == p.splits - 1) ? 1 : 0;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kDequantWarps * 32) : "memory");
            if (*last_flag) {
                __threadfence();
                const float* base = p.partial + tile_id * p.splits * tile_elems;
                for (int m = 0; m < rows; ++m) {
                    float acc = 0.f;
                    for (int z = 0; z < p.splits; ++z)
                        acc += __ldcg(base + z * tile_elems + (long long)m * kTileN + t);
                    if (ok && row_ok)
                        y[(long long)(row_start + m) * p.N + n] = __float2bfloat16_rn(acc);
                }
                if (t == 0) p.counters[tile_id] = 0;  // ready for the next call
            }
        }
    }

    if (!ok) flag_status(p.status, MXQ_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        // make sure no MMA is still writing tensor memory (bounded wait)
        if (!ok) (void)mbar_wait(accf, 0);
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
    }
}

}  // namespace

cudaError_t launch_qmm_tc(const QmmParams& p, int bits, int grid_m, int max_rows_per_tile,
                          cudaStream_t stream) {
    const SmemLayout L = make_layout(bits, max_rows_per_tile);
    const dim3 grid((p.N + kTileN - 1) / kTileN, grid_m, p.splits);
    const dim3 block(kThreads);
    cudaError_t err;
    if (bits == 4) {
        err = cudaFuncSetAttribute(qmm_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   L.total);
        if (err != cudaSuccess) return err;
        qmm_tc_kernel<4><<<grid, block, L.total, stream>>>(p, max_rows_per_tile);
    } else {
        err = cudaFuncSetAttribute(qmm_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   L.total);
        if (err != cudaSuccess) return err;
        qmm_tc_kernel<8><<<grid, block, L.total, stream>>>(p, max_rows_per_tile);
    }
    return cudaGetLastError();
}

}  // namespace mxq
