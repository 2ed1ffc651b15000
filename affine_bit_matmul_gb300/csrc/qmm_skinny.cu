// Quantized GEMM for a few activation rows at a time ("skinny" GEMM):
// the small-M prefill shapes (M <= 8) and the decode-sized sorted-MoE
// calls, where each expert sees one to eight routed rows (mlxcel issue #1538,
// comment "Correction: MoE decode does not route to qmm_naive": decode runs
// fused per-expert gate/up and down kernels instead of the grouped GEMM).
// These shapes are HBM-bound: every code byte is used by at most eight
// activation rows, so the kernel is built to stream the codes once at full
// bandwidth and to spend as few instructions per code as possible.
//
// Arithmetic.  For a W row n, a group g of G consecutive k and an activation
// row m,
//     sum_{k in g} x[m,k] * (s q[n,k] + b) = s * A_g + (b - 128 s) * X_g,
//     A_g = sum_{k in g} x[m,k] * (128 + q[n,k]),   X_g = sum_{k in g} x[m,k].
// 128 + q is an exact bf16 (exponent of 128, the code in the low mantissa
// bits), made from a packed word with one AND/OR per pair of codes, and A_g
// is a tensor-core product (mma.sync m16n8k16, bf16 operands, fp32
// accumulation): 16 W rows x 16 k times 16 k x 8 activation rows.  The
// affine terms are applied per group in fp32 registers.  No bf16 rounding of
// dequantised weights takes place at all.
//
// Order of k inside an MMA.  The contraction index of an MMA may be any
// permutation of the physical k, as long as both operands use the same one.
// A thread of the MMA owns contraction slots {2t, 2t+1, 2t+8, 2t+9} (t =
// lane % 4); for a 32-wide block of k the thread takes the 8 codes of one
// packed word (k = 8t .. 8t+7) of its two W rows and pairs them as (0,4),
// (1,5) in the first MMA and (2,6), (3,7) in the second, which is what an
// AND with 0x000F000F after a shift of 0, 4, 8 or 12 bits yields.  The
// activations are stored in shared memory with every 8 values reordered as
// 0,4,1,5,2,6,3,7, so the matching operand is one 16-byte load.
//
// Work.  A task is (activation item, 16-row slab of W): an item is up to
// eight activation rows that share one weight matrix (the dense call's M
// rows, or one expert's routed rows).  K is split over the CTAs of a
// thread-block cluster when there are too few slabs for the SMs; each CTA's
// eight compute warps split its part of K by groups, add their partials in
// a fixed order through shared memory, and the cluster adds its CTAs'
// partials in rank order through distributed shared memory: deterministic.
// A producer warp streams the codes of each task's slab by TMA (128-byte
// swizzled boxes: the fragment loads are conflict-free) into a ring of
// stages, and the activation rows of each new item into one of two slots.
// For the gate/up pair ("sets" = 2) a task streams both matrices' slabs
// against the one copy of its activation rows.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kSkWarps = 8;                   // compute warps
constexpr int kSkThreads = (kSkWarps + 1) * 32;  // + the producer warp
constexpr int kSkRows = 16;                   // W rows per task (the MMA's M)
constexpr int kSkMaxRows = 8;                 // activation rows per item (the MMA's N)
constexpr int kSkMaxStages = 12;
constexpr int kSkBoxK = 256;                  // k per 128-byte box row of 4-bit codes
constexpr int kSkBoxBytes = kSkRows * 128;    // one TMA box: 16 rows x 128 bytes
constexpr int kSkMaxGpw = 12;                 // groups per warp at most
constexpr int kSkSmemMax = 227 * 1024;

__device__ __forceinline__ uint32_t sk_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void sk_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void sk_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void sk_tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void sk_tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                          int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void sk_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t sk_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float sk_ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Named barrier of the compute warps only (the producer warp never joins).
__device__ __forceinline__ void sk_compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSkWarps * 32) : "memory");
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool sk_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitBudgetCycles) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// D += A . B for one m16n8k16 tile: A = 16 W rows x 16 k (bf16), B = 16 k x
// 8 activation rows (bf16), D fp32.
__device__ __forceinline__ void sk_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Codes i and i+4 of a packed 4-bit word as the bf16 pair (128 + q_i,
// 128 + q_{i+4}) (low half first).
__device__ __forceinline__ uint32_t sk_pair(uint32_t w, int shift) {
    return ((w >> shift) & 0x000F000Fu) | 0x43004300u;
}

// The 8 activations of a 16-byte chunk reordered 0,4,1,5,2,6,3,7 (as bf16
// pairs), and their fp32 sum added to *sum in k order.
__device__ __forceinline__ uint4 sk_permute8(uint4 v, float* sum) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    float s = *sum;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s += __uint_as_float(u[j] << 16);
        s += __uint_as_float(u[j] & 0xFFFF0000u);
    }
    *sum = s;
    uint4 o;
    o.x = sk_prmt(v.x, v.z, 0x5410u);  // x0 x4
    o.y = sk_prmt(v.x, v.z, 0x7632u);  // x1 x5
    o.z = sk_prmt(v.y, v.w, 0x5410u);  // x2 x6
    o.w = sk_prmt(v.y, v.w, 0x7632u);  // x3 x7
    return o;
}

template <bool GATHER>
__global__ void __launch_bounds__(kSkThreads, 1)
    qmm_skinny_kernel(const SkinnyParams p, const __grid_constant__ CUtensorMap cm0,
                      const __grid_constant__ CUtensorMap cm1) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // [kSkMaxStages]
    uint64_t* empty = full + kSkMaxStages;                           // [kSkMaxStages]
    uint64_t* xfull = empty + kSkMaxStages;                          // [2]
    uint64_t* xempty = xfull + 2;                                    // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xempty + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int z = p.S > 1 ? (int)sk_cluster_rank() : 0;  // this CTA's part of K
    const int cid = blockIdx.x / p.S;                    // cluster
    const int C = gridDim.x / p.S;                       // clusters
    const int n_items = GATHER ? *p.item_count : 1;
    const int total = n_items * p.slabs;                 // tasks
    const int kz0 = z * p.kc;                            // first k of this CTA's part
    const int groups_c = p.kc / p.group;                 // groups in the part
    const int xslot_bytes = p.slot_rows * p.xstride;
    const int xsslot_bytes = p.slot_rows * p.xs_row * 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kSkWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], kSkWarps);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kSkWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const char* xb = static_cast<const char*>(p.x);
            int st = 0;
            uint32_t ph = 0;
            long long issued = 0;
            int prev_item = -1, xloads = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                const int t = cid + j * C;
                if (t >= total) break;
                const int it = t / p.slabs;
                const int n0 = (t - it * p.slabs) * kSkRows;
                MTile item;
                if (GATHER) {
                    item = p.items[it];
                } else {
                    item.e = 0;
                    item.row_start = 0;
                    item.rows = p.M;
                }
                if (it != prev_item) {
                    // the activation rows (and, grouped, their group sums) of a new item
                    const int xs = xloads & 1;
                    const int use = xloads >> 1;
                    if (use > 0 && !sk_wait(&xempty[xs], (uint32_t)((use - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t row_bytes = (uint32_t)(p.kc * 2);
                    const uint32_t xs_bytes = (uint32_t)(p.xs_row * 4);
                    sk_expect_tx(&xfull[xs], (uint32_t)item.rows * (row_bytes + (GATHER ? xs_bytes : 0u)));
                    const uint32_t xdst = base + p.x_off + xs * xslot_bytes;
                    const uint32_t sdst = base + p.xs_off + xs * xsslot_bytes;
                    for (int r = 0; r < item.rows; ++r) {
                        const long long row = item.row_start + r;
                        sk_bulk_g2s(xdst + r * p.xstride, xb + (row * p.K + kz0) * 2, row_bytes,
                                    &xfull[xs]);
                        if (GATHER)
                            sk_bulk_g2s(sdst + r * p.xs_row * 4, p.xsum + row * p.xs_ld, xs_bytes,
                                        &xfull[xs]);
                    }
                    prev_item = it;
                    ++xloads;
                }
                for (int set = 0; set < p.sets; ++set) {
                    if (issued >= p.stages && !sk_wait(&empty[st], ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    sk_expect_tx(&full[st], (uint32_t)(p.nbox * kSkBoxBytes));
                    const uint32_t dst = base + st * p.stage_bytes;
                    const CUtensorMap* map = set ? &cm1 : &cm0;
                    for (int bx = 0; bx < p.nbox; ++bx) {
                        const int c0 = kz0 / 8 + bx * 32;  // 32 words = 256 codes per box row
                        if (GATHER)
                            sk_tma_3d(dst + bx * kSkBoxBytes, map, c0, n0, item.e, &full[st]);
                        else
                            sk_tma_2d(dst + bx * kSkBoxBytes, map, c0, n0, &full[st]);
                    }
                    ++issued;
                    if (++st == p.stages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // every copy issued into the ring lands before the CTA exits:
                // wait for the last `stages` stages (bounded by the full budget
                // each; copies complete unless the device itself has failed)
                for (long long g = issued - 1; g >= 0 && g >= issued - p.stages; --g) {
                    const int slot = (int)(g % p.stages);
                    const uint32_t par = (uint32_t)((g / p.stages) & 1);
                    (void)mbar_wait(&full[slot], par);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute
        const int gq = lane >> 2;  // W rows gq, gq + 8 of the slab; activation row gq (B operand)
        const int tq = lane & 3;   // contraction slots 2t, 2t+1, 2t+8, 2t+9
        const int gpw = p.gpw;
        const int g0 = warp * gpw;                          // this warp's groups of the part
        const int g1 = min(groups_c, g0 + gpw);
        const int upg = p.group / 32;                       // 32-wide k blocks per group
        // this warp's scale/bias stage in shared memory: [buf][set][row 16][gpw] (s | b << 16)
        const uint32_t sb_warp = base + p.sb_off + warp * (2 * 2 * kSkRows * kSkMaxGpw * 4);
        float* red = reinterpret_cast<float*>(smem + p.red_off);  // [2][kSkWarps][16][8]
        float* part = reinterpret_cast<float*>(smem + p.part_off);
        bool ok = true;
        int st = 0;
        uint32_t ph = 0;
        int prev_item = -1, xloads = 0, xs = 0;

        // scale/bias pairs of task t for this warp's groups: lane l loads row
        // l % 16, groups of parity l / 16; kept in registers until the task
        // before it has finished, then stored to shared memory
        uint32_t sbreg[2][kSkMaxGpw / 2];
        auto sb_issue = [&](int t) {
            const int it = t / p.slabs;
            const int n = (t - it * p.slabs) * kSkRows + (lane & 15);
            const int e = GATHER ? p.items[it].e : 0;
#pragma unroll
            for (int set = 0; set < 2; ++set)
#pragma unroll
                for (int i = 0; i < kSkMaxGpw / 2; ++i) {
                    const int gl = 2 * i + (lane >> 4);
                    uint32_t v = 0;
                    if (set < p.sets && g0 + gl < g1 && n < p.N) {
                        const long long at = (long long)e * p.sb_estride +
                                             (long long)n * (p.K / p.group) + (kz0 / p.group) + g0 + gl;
                        v = (uint32_t)__ldg(p.s[set] + at) | ((uint32_t)__ldg(p.b[set] + at) << 16);
                    }
                    sbreg[set][i] = v;
                }
        };
        auto sb_store = [&](int buf) {
#pragma unroll
            for (int set = 0; set < 2; ++set)
#pragma unroll
                for (int i = 0; i < kSkMaxGpw / 2; ++i) {
                    const int gl = 2 * i + (lane >> 4);
                    if (gl < kSkMaxGpw)
                        asm volatile("st.shared.u32 [%0], %1;" ::"r"(
                                         sb_warp + (uint32_t)((((buf * 2 + set) * kSkRows + (lane & 15)) *
                                                               kSkMaxGpw + gl) * 4)),
                                     "r"(sbreg[set][i])
                                     : "memory");
                }
        };

        int j = 0;
        int t = cid;
        if (t < total) {
            sb_issue(t);
            sb_store(0);
            __syncwarp();
        }
        for (; t < total; ++j, t += C) {
            const int it = t / p.slabs;
            const int n0 = (t - it * p.slabs) * kSkRows;
            MTile item;
            if (GATHER) {
                item = p.items[it];
            } else {
                item.e = 0;
                item.row_start = 0;
                item.rows = p.M;
            }
            const int tn = t + C;
            if (tn < total) sb_issue(tn);  // the next task's scale/bias pairs, in flight
            if (it != prev_item) {
                if (prev_item >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&xempty[xs]);  // done with the old item's rows
                }
                xs = xloads & 1;
                if (ok && !sk_wait(&xfull[xs], (uint32_t)((xloads >> 1) & 1), abort_flag)) ok = false;
                if (!GATHER) {
                    // the dense call's rows arrive as plain bf16: reorder each 8
                    // values in place and form the group sums, once per launch
                    const uint32_t xa = base + p.x_off + xs * xslot_bytes;
                    float* xsum = reinterpret_cast<float*>(smem + p.xs_off + xs * xsslot_bytes);
                    for (int idx = threadIdx.x; ok && idx < item.rows * groups_c; idx += kSkWarps * 32) {
                        const int m = idx / groups_c, g = idx - m * groups_c;
                        float sum = 0.f;
                        for (int c = 0; c < p.group / 8; ++c) {
                            const uint32_t a = xa + m * p.xstride + (g * p.group + 8 * c) * 2;
                            uint4 v;
                            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                         : "r"(a));
                            v = sk_permute8(v, &sum);
                            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x),
                                         "r"(v.y), "r"(v.z), "r"(v.w)
                                         : "memory");
                        }
                        xsum[m * p.xs_row + g] = sum;
                    }
                    sk_compute_sync();
                }
                prev_item = it;
                ++xloads;
            }
            const uint32_t xa = base + p.x_off + xs * xslot_bytes + gq * p.xstride;
            const float* xsum = reinterpret_cast<const float*>(smem + p.xs_off + xs * xsslot_bytes);
            const int buf = j & 1;
            for (int set = 0; set < p.sets; ++set) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (ok && !sk_wait(&full[st], ph, abort_flag)) ok = false;
                if (ok) {
                    const uint32_t cbase = base + st * p.stage_bytes;
                    const uint32_t sbb = sb_warp + (uint32_t)((buf * 2 + set) * kSkRows * kSkMaxGpw * 4);
                    for (int g = g0; g < g1; ++g) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int u = 0; u < upg; ++u) {
                            const int kk = g * p.group + 32 * u;  // k within the part
                            const int box = kk / kSkBoxK;
                            const int chunk = (kk % kSkBoxK) / 32;
                            const uint32_t c_lo = cbase + box * kSkBoxBytes + gq * 128 +
                                                  ((chunk ^ (gq & 7)) << 4) + 4 * tq;
                            uint32_t w0, w1;  // W rows gq and gq + 8 (same swizzle: rows differ by 8)
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(c_lo));
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w1) : "r"(c_lo + 8 * 128));
                            uint4 xv;
                            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                                         : "r"(xa + (kk + 8 * tq) * 2));
                            sk_mma(d, sk_pair(w0, 0), sk_pair(w1, 0), sk_pair(w0, 4), sk_pair(w1, 4),
                                   xv.x, xv.y);
                            sk_mma(d, sk_pair(w0, 8), sk_pair(w1, 8), sk_pair(w0, 12), sk_pair(w1, 12),
                                   xv.z, xv.w);
                        }
                        // affine terms of group g: rows gq, gq + 8; activation rows 2t, 2t + 1
                        uint32_t sb0, sb1;
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(sb0)
                                     : "r"(sbb + (uint32_t)((gq * kSkMaxGpw + (g - g0)) * 4)));
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(sb1)
                                     : "r"(sbb + (uint32_t)(((gq + 8) * kSkMaxGpw + (g - g0)) * 4)));
                        const float s0 = __uint_as_float(sb0 << 16), b0 = __uint_as_float(sb0 & 0xFFFF0000u);
                        const float s1 = __uint_as_float(sb1 << 16), b1 = __uint_as_float(sb1 & 0xFFFF0000u);
                        const float c0 = fmaf(-128.f, s0, b0), c1 = fmaf(-128.f, s1, b1);
                        const float X0 = xsum[(2 * tq) * p.xs_row + g];
                        const float X1 = xsum[(2 * tq + 1) * p.xs_row + g];
                        acc[0] = fmaf(s0, d[0], fmaf(c0, X0, acc[0]));
                        acc[1] = fmaf(s0, d[1], fmaf(c0, X1, acc[1]));
                        acc[2] = fmaf(s1, d[2], fmaf(c1, X0, acc[2]));
                        acc[3] = fmaf(s1, d[3], fmaf(c1, X1, acc[3]));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
                if (++st == p.stages) {
                    st = 0;
                    ph ^= 1u;
                }
                // the warps' partials, added in warp order
                float* rb = red + (size_t)(buf * kSkWarps + warp) * kSkRows * 8;
                rb[gq * 8 + 2 * tq] = acc[0];
                rb[gq * 8 + 2 * tq + 1] = acc[1];
                rb[(gq + 8) * 8 + 2 * tq] = acc[2];
                rb[(gq + 8) * 8 + 2 * tq + 1] = acc[3];
                sk_compute_sync();
                if (threadIdx.x < kSkRows * 8) {
                    const int n = threadIdx.x >> 3, m = threadIdx.x & 7;
                    float v = 0.f;
                    for (int w = 0; w < kSkWarps; ++w)
                        v += red[(size_t)(buf * kSkWarps + w) * kSkRows * 8 + threadIdx.x];
                    if (p.S == 1) {
                        if (ok && m < item.rows && n0 + n < p.N)
                            p.y[set][(long long)(item.row_start + m) * p.N + n0 + n] =
                                __float2bfloat16_rn(v);
                    } else {
                        part[((j * p.sets + set) * kSkRows + n) * 8 + m] = v;
                    }
                }
                // the next set (or task) writes the other buffer half
                if (p.sets == 2 && set == 0) sk_compute_sync();
            }
            // this task's successor's scale/bias pairs into the other buffer
            __syncwarp();
            if (tn < total) sb_store(buf ^ 1);
            __syncwarp();
        }
    }

    if (p.S > 1) {
        // the cluster's CTAs hold partials of the same tasks for their parts
        // of K: rank z adds those of tasks j with j % S == z, in rank order
        sk_cluster_sync();
        if (warp < kSkWarps) {
            const uint32_t part_a = base + p.part_off;
            for (int jj = z, tt = cid + z * C; tt < total; jj += p.S, tt += p.S * C) {
                const int it = tt / p.slabs;
                const int n0 = (tt - it * p.slabs) * kSkRows;
                for (int idx = threadIdx.x; idx < p.sets * kSkRows * 8; idx += kSkWarps * 32) {
                    const int set = idx / (kSkRows * 8);
                    const int n = (idx >> 3) % kSkRows, m = idx & 7;
                    float v = 0.f;
                    for (int r = 0; r < p.S; ++r)
                        v += sk_ld_cluster_f32(part_a + (uint32_t)(((jj * p.sets + set) * kSkRows + n) * 8 + m) * 4,
                                               (uint32_t)r);
                    if (!*abort_flag && m < p.M && n0 + n < p.N)
                        p.y[set][(long long)m * p.N + n0 + n] = __float2bfloat16_rn(v);
                }
            }
        }
        sk_cluster_sync();
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, MXQ_DEV_TIMEOUT);
}

// Grouped form, step 2: the routed activation rows in sorted order, each 8
// values reordered 0,4,1,5,2,6,3,7 for the kernel above, and their per-group
// sums (zero rows for an invalid source row).  One warp per sorted row.
__global__ void __launch_bounds__(256) skinny_xprep_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const int32_t* __restrict__ row_src,
                                                           int T, int B, int K, int group,
                                                           int xs_ld, uint4* __restrict__ xp,
                                                           float* __restrict__ xsum) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r < B) {
        const int src = row_src ? row_src[r] : r;
        const bool valid = src >= 0 && src < T;
        const int groups = K / group;
        const uint4* xs = reinterpret_cast<const uint4*>(x + (long long)(valid ? src : 0) * K);
        uint4* dst = xp + (long long)r * (K / 8);
        for (int g = lane; g < groups; g += 32) {
            float sum = 0.f;
            for (int c = 0; c < group / 8; ++c) {
                const int ci = g * (group / 8) + c;
                uint4 v = valid ? __ldg(xs + ci) : make_uint4(0u, 0u, 0u, 0u);
                dst[ci] = sk_permute8(v, &sum);
            }
            xsum[(long long)r * xs_ld + g] = sum;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

size_t skinny_smem_bytes(const SkinnyParams& p) { return (size_t)p.bar_off + 256 + 1024; }

// Plan of the skinny kernel's shared memory: code stages first (1024-byte
// aligned boxes), then the activation slots, group sums, scale/bias stages,
// partial-sum buffers and barriers.  Returns false if the shape does not fit.
bool plan_skinny(SkinnyParams& p, int part_tasks) {
    p.nbox = (p.kc + kSkBoxK - 1) / kSkBoxK;
    p.stage_bytes = p.nbox * kSkBoxBytes;
    p.xstride = p.kc * 2 + 16;  // rows 16 bytes apart modulo 128: conflict-free fragment loads
    const int groups_c = p.kc / p.group;
    p.gpw = (groups_c + kSkWarps - 1) / kSkWarps;
    if (p.gpw > kSkMaxGpw) return false;
    p.xs_row = (groups_c + 3) & ~3;
    p.part_tasks = p.S > 1 ? part_tasks : 0;
    if (p.slot_rows < 1 || p.slot_rows > kSkMaxRows) return false;
    const int fixed = p.xslots * p.slot_rows * (p.xstride + p.xs_row * 4) +
                      kSkWarps * 2 * 2 * kSkRows * kSkMaxGpw * 4 + 2 * kSkWarps * kSkRows * 8 * 4 +
                      p.part_tasks * p.sets * kSkRows * 8 * 4 + 256 + 1024;
    int stages = (kSkSmemMax - fixed) / p.stage_bytes;
    if (stages > kSkMaxStages) stages = kSkMaxStages;
    if (stages < 2) return false;
    p.stages = stages;
    p.x_off = stages * p.stage_bytes;
    p.xs_off = p.x_off + p.xslots * p.slot_rows * p.xstride;
    p.sb_off = p.xs_off + p.xslots * p.slot_rows * p.xs_row * 4;
    p.red_off = p.sb_off + kSkWarps * 2 * 2 * kSkRows * kSkMaxGpw * 4;
    p.part_off = p.red_off + 2 * kSkWarps * kSkRows * 8 * 4;
    p.bar_off = p.part_off + p.part_tasks * p.sets * kSkRows * 8 * 4;
    return (int)skinny_smem_bytes(p) <= kSkSmemMax;
}

cudaError_t launch_skinny(const SkinnyParams& p, const uint32_t* w0, const uint32_t* w1, int E,
                          int grid, cudaStream_t stream) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const bool gather = p.items != nullptr;
    CUtensorMap cm[2];
    const cuuint64_t words = (cuuint64_t)p.K / 8;
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int set = 0; set < p.sets; ++set) {
        const uint32_t* w = set ? w1 : w0;
        CUresult r;
        if (gather) {
            const cuuint64_t dims[3] = {words, (cuuint64_t)p.N, (cuuint64_t)E};
            const cuuint64_t strides[2] = {words * 4, words * 4 * (cuuint64_t)p.N};
            const cuuint32_t box[3] = {32, (cuuint32_t)kSkRows, 1};
            r = enc(&cm[set], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(w), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[2] = {words, (cuuint64_t)p.N};
            const cuuint64_t strides[1] = {words * 4};
            const cuuint32_t box[2] = {32, (cuuint32_t)kSkRows};
            r = enc(&cm[set], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(w), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    if (p.sets == 1) cm[1] = cm[0];
    const int smem = (int)skinny_smem_bytes(p);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (gather) {
        e = cudaFuncSetAttribute(qmm_skinny_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, qmm_skinny_kernel<true>, p, cm[0], cm[1]);
    } else {
        e = cudaFuncSetAttribute(qmm_skinny_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, qmm_skinny_kernel<false>, p, cm[0], cm[1]);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_skinny_xprep(const void* x, const int32_t* row_src, int T, int B, int K,
                                int group, int xs_ld, void* xp, float* xsum, cudaStream_t stream) {
    // a programmatic dependent launch after the tile-table prepass: it reads
    // only x and row_src, which the prepass does not write
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((B + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_xprep_kernel,
                                       static_cast<const __nv_bfloat16*>(x), row_src, T, B, K,
                                       group, xs_ld, static_cast<uint4*>(xp), xsum);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mxq
