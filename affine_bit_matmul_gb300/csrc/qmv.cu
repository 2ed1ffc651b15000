// Decode GEMV for affine group-wise quantized weights (M = 1).
//
// mlxcel issue #1536, Diagnosis item 3: the qmv kernel must accumulate in
// float at every bit width; it is the HBM-bound half of decoding (Baseline
// section: the qmv share of a decode step moves ~15 GB of codes).
//
// Two kernels share the arithmetic below.
//
// qmv_stream_kernel (K a multiple of 512, K <= 20480, 16-byte aligned
// scales/biases, a multiple of 8 groups per row): persistent CTAs, one per SM.  A producer thread streams
// chunks of R consecutive rows (their codes, scales and biases are each one
// contiguous block) into a ring of shared-memory stages with bulk async
// copies (cp.async.bulk + mbarrier transaction counts), so ~100 KB per SM
// stay in flight without any thread waiting on HBM.  Compute warps own one
// 1024-wide K segment each (several warps per segment take alternate rows);
// every lane keeps its 32 activations in registers for the whole kernel.
//
// The chunks are equal in size (within one row) and as many as a multiple
// of the grid, so every CTA streams the same share.  The kernel is a
// programmatic dependent launch: its CTAs start as the previous kernel's
// finish and wait for that kernel to complete before reading anything into
// shared memory; meanwhile each asks L2 to prefetch its first chunk.
//
// qmv_generic_kernel (any other shape): direct 16-byte loads, one CTA per 16
// rows.
//
// Layout of the work in both:
//  * a lane owns 16 bytes of codes per row (32 four-bit or 16 eight-bit
//    codes), or 8, 12 or 24 bytes (32 two-, three- or six-bit codes; the
//    last two only in the direct-load kernel), always inside one group: groups
//    are 32, 64 or 128 wide and a lane's first k is a multiple of its code
//    count; a warp covers a K segment of 1024 (2- and 4-bit) or 512 (8-bit)
//    values with one coalesced load per row;
//  * a CTA has one warp per K segment and owns a block of ROWS output rows;
//    each lane keeps its 32/16 activations in registers for all the rows;
//  * the affine terms are applied once per lane and row:
//        sum_k x_k (s q_k + b) = s * (sum_k x_k q_k) + b * X,
//    with X = sum_k x_k over the lane's values (fp32);
//  * the streaming kernel forms sum_k x_k q_k exactly with integer 4-way
//    dot products over byte planes of the activations (see lane_dot_int);
//    the direct-load kernel turns the codes into floats 1 + q*2^-7 (2- and
//    4-bit) or 1 + q*2^-15 (8-bit) by placing them in the mantissa of a constant
//    with one byte permute each, sums x_k v_k in fp32 and uses
//    sum_k x_k q_k = 2^p * (sum_k x_k v_k - X), p = 7 or 15;
//  * per-row partials are reduced across lanes with a reduce-scatter
//    butterfly, then across warps through shared memory in a fixed order,
//    so results are identical from run to run.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kRows = 16;    // output rows per CTA
constexpr int kUnroll = 4;   // rows whose codes are in flight together
constexpr int kMaxWarps = 20;  // one warp per K segment up to K = 20480 (4-bit)

// Warps per CTA of the direct-load kernels: 3- and 6-bit codes are cut out
// of the bit stream one by one and need more registers, so fewer warps.
__host__ __device__ constexpr int direct_max_warps(int bits) {
    return (bits == 3 || bits == 6) ? 16 : kMaxWarps;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
    unsigned long long A = *reinterpret_cast<unsigned long long*>(&a);
    unsigned long long B = *reinterpret_cast<unsigned long long*>(&b);
    unsigned long long C = *reinterpret_cast<unsigned long long*>(&acc);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(C) : "l"(A), "l"(B));
    acc = *reinterpret_cast<float2*>(&C);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ldg_stream2(const uint2* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// Sum over the lane's codes of x_k * v_k, v_k = 1 + q_k * 2^-7, for 32
// two-bit codes in c.x, c.y (lowest k in the lowest two bits of each word).
// Byte i of plane j = (word >> 2j) & 0x03030303 is code 4i + j of the word,
// so planes 2t and 2t + 1 give the pairs (x_{4i+2t}, x_{4i+2t+1}).
__device__ __forceinline__ float dot_chunk2(const uint4 c, const float2 (&x2)[16]) {
    const uint32_t words[2] = {c.x, c.y};
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t pe = ((words[w] >> (4 * t)) & 0x03030303u) | 0x80808080u;
            const uint32_t po = ((words[w] >> (4 * t + 2)) & 0x03030303u) | 0x80808080u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t sel = 0x7044u | (uint32_t(i) << 8);
                float2 v;
                v.x = __uint_as_float(prmt(pe, 0x3F000000u, sel));
                v.y = __uint_as_float(prmt(po, 0x3F000000u, sel));
                ffma2(acc, v, x2[w * 8 + i * 2 + t]);
            }
        }
    }
    return acc.x + acc.y;
}

// Sum over the lane's codes of x_k * v_k, v_k = 1 + q_k * 2^-7, for one
// 16-byte chunk of 4-bit codes (32 values).  x2[j] = (x_{2j}, x_{2j+1}).
__device__ __forceinline__ float dot_chunk4(const uint4 c, const float2 (&x2)[16]) {
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bytes of lo: 0x80 | nibble 0, 2, 4, 6; of hi: 0x80 | nibble 1, 3, 5, 7
        const uint32_t lo = (words[i] & 0x0F0F0F0Fu) | 0x80808080u;
        const uint32_t hi = ((words[i] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            // float bits 0x3F, (0x80 | q), 0x00, 0x00 -> 1 + q/128
            const uint32_t sel = 0x7044u | (uint32_t(b) << 8);
            float2 v;
            v.x = __uint_as_float(prmt(lo, 0x3F000000u, sel));
            v.y = __uint_as_float(prmt(hi, 0x3F000000u, sel));
            ffma2(acc, v, x2[i * 4 + b]);
        }
    }
    return acc.x + acc.y;
}

// 3- and 6-bit codes: the lane's 32 codes are BITS words of the row's
// little-endian bit stream (code m holds bits [m*BITS, m*BITS + BITS) of
// them, possibly across two words).  code_as_float places code m in the
// mantissa at bit 16: v = 1 + q * 2^-7.
template <int BITS>
__device__ __forceinline__ float code_as_float(const uint32_t (&w)[6], int m) {
    const int p = m * BITS;
    const int j = p >> 5, off = p & 31;
    uint32_t t;
    if (off + BITS > 32)
        t = __funnelshift_r(w[j], w[j + 1], off - 16);  // off > 26 here
    else if (off >= 16)
        t = w[j] >> (off - 16);
    else
        t = w[j] << (16 - off);
    return __uint_as_float((t & (((1u << BITS) - 1u) << 16)) | 0x3F800000u);
}

template <int BITS>
__device__ __forceinline__ float dot_chunk_stream(const uint32_t (&w)[6], const float2 (&x2)[16]) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 v;
        v.x = code_as_float<BITS>(w, 2 * i);
        v.y = code_as_float<BITS>(w, 2 * i + 1);
        ffma2(acc, v, x2[i]);
    }
    return acc.x + acc.y;
}

// Same for 16 eight-bit codes: v_k = 1 + q_k * 2^-15.  x2 holds 8 pairs.
__device__ __forceinline__ float dot_chunk8(const uint4 c, const float2 (&x2)[16]) {
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            // float bits 0x3F, 0x80, q, 0x00 -> 1 + q/32768
            float2 v;
            v.x = __uint_as_float(prmt(words[i], 0x3F800000u, 0x7604u | (uint32_t(2 * b) << 4)));
            v.y = __uint_as_float(prmt(words[i], 0x3F800000u, 0x7604u | (uint32_t(2 * b + 1) << 4)));
            ffma2(acc, v, x2[i * 2 + b]);
        }
    }
    return acc.x + acc.y;
}

// The direct-load GEMV for output rows [row0, row0 + kRows) of one matrix:
// y[n] = sum_k x[k] * w^[n, k].  Warps split K into segments; a CTA's warps
// then add their partials in a fixed order.
template <int BITS>
__device__ __forceinline__ void qmv_rows_direct(const __nv_bfloat16* __restrict__ x,
                                                const uint32_t* __restrict__ w,
                                                const uint16_t* __restrict__ scales,
                                                const uint16_t* __restrict__ biases,
                                                __nv_bfloat16* __restrict__ y, int K, int N,
                                                int group, int row0) {
    constexpr int kCodesPerLane = BITS == 8 ? 16 : 32;
    constexpr int kSegK = 32 * kCodesPerLane;          // 1024 or 512
    // rows whose codes are in flight together (two for 3- and 6-bit rows,
    // whose codes are cut out of the bit stream one by one)
    constexpr int kU = (BITS == 3 || BITS == 6) ? 2 : kUnroll;
    constexpr float kUnscale = BITS == 8 ? 32768.f : 128.f;
    __shared__ float red[kMaxWarps][kRows];

    const int lane = lane_id();
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nseg = (K + kSegK - 1) / kSegK;
    const long long words_per_row = (long long)K * BITS / 32;
    const int groups = K / group;

    float part[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) part[r] = 0.f;

    for (int seg = warp; seg < nseg; seg += nwarps) {
        const int k0 = seg * kSegK + lane * kCodesPerLane;
        if (k0 >= K) continue;  // lanes past the end of K (K % 64 == 0)
        // activations of this lane, as float pairs
        float2 x2[16];
        float X = 0.f;
        {
            const uint4* xp = reinterpret_cast<const uint4*>(x + k0);
#pragma unroll
            for (int c = 0; c < kCodesPerLane / 8; ++c) {
                const uint4 v = __ldg(xp + c);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x2[c * 4 + j].x = __uint_as_float(u[j] << 16);
                    x2[c * 4 + j].y = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int j = 0; j < kCodesPerLane / 2; ++j) X += x2[j].x + x2[j].y;
        }
        const int g = k0 / group;
        const long long wofs = (long long)k0 * BITS / 32;  // word offset in a row

#pragma unroll
        for (int r0 = 0; r0 < kRows; r0 += kU) {
            uint4 c[kU];
            uint32_t cs[kU][6];  // 3- and 6-bit codes: BITS words per lane
            float s[kU], b[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int n = row0 + r0 + u;
#pragma unroll
                for (int j = 0; j < 6; ++j) cs[u][j] = 0u;
                if (n < N) {
                    if (BITS == 3) {
                        const uint32_t* src = w + n * words_per_row + wofs;
#pragma unroll
                        for (int j = 0; j < 3; ++j) cs[u][j] = __ldg(src + j);
                        c[u] = make_uint4(0u, 0u, 0u, 0u);
                    } else if (BITS == 6) {
                        // 24 bytes from an 8-byte aligned offset (6 * k0 / 32 words)
                        const uint2* src = reinterpret_cast<const uint2*>(w + n * words_per_row + wofs);
#pragma unroll
                        for (int j = 0; j < 3; ++j) {
                            const uint2 v = __ldg(src + j);
                            cs[u][2 * j] = v.x;
                            cs[u][2 * j + 1] = v.y;
                        }
                        c[u] = make_uint4(0u, 0u, 0u, 0u);
                    } else if (BITS == 2) {
                        const uint2 v =
                            ldg_stream2(reinterpret_cast<const uint2*>(w + n * words_per_row + wofs));
                        c[u] = make_uint4(v.x, v.y, 0u, 0u);
                    } else {
                        c[u] = ldg_stream(reinterpret_cast<const uint4*>(w + n * words_per_row + wofs));
                    }
                    s[u] = bf16_bits_to_float(__ldg(scales + (long long)n * groups + g));
                    b[u] = bf16_bits_to_float(__ldg(biases + (long long)n * groups + g));
                } else {
                    c[u] = make_uint4(0, 0, 0, 0);
                    s[u] = 0.f;
                    b[u] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const float A = (BITS == 3 || BITS == 6) ? dot_chunk_stream<BITS>(cs[u], x2)
                                : BITS == 2                ? dot_chunk2(c[u], x2)
                                : BITS == 4                ? dot_chunk4(c[u], x2)
                                                           : dot_chunk8(c[u], x2);
                part[r0 + u] += fmaf(s[u] * kUnscale, A - X, b[u] * X);
            }
        }
    }

    // reduce-scatter over the warp: afterwards lane 2r holds row r's sum
#pragma unroll
    for (int half = kRows / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? part[i] : part[i + half];
            const float keep = upper ? part[i + half] : part[i];
            part[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
    }
    part[0] += __shfl_xor_sync(0xFFFFFFFFu, part[0], 1);
    if ((lane & 1) == 0) red[warp][lane >> 1] = part[0];
    __syncthreads();
    if (threadIdx.x < kRows) {
        const int n = row0 + threadIdx.x;
        float acc = 0.f;
        for (int wi = 0; wi < nwarps; ++wi) acc += red[wi][threadIdx.x];
        if (n < N) y[n] = __float2bfloat16_rn(acc);
    }
}

template <int BITS>
__global__ void __launch_bounds__(direct_max_warps(BITS) * 32) qmv_generic_kernel(const __nv_bfloat16* __restrict__ x,
                                                   const uint32_t* __restrict__ w,
                                                   const uint16_t* __restrict__ scales,
                                                   const uint16_t* __restrict__ biases,
                                                   __nv_bfloat16* __restrict__ y, int K, int N,
                                                   int group) {
    qmv_rows_direct<BITS>(x, w, scales, biases, y, K, N, group, blockIdx.x * kRows);
}

// Grouped form with few rows (decode): sorted row r = blockIdx.y is the GEMV
// of expert ids[r]'s matrix with activation row row_src[r].  Every CTA checks
// all the (few) ids itself, so no separate pass is needed: an id outside
// [0, E) or a source row outside [0, T) makes the row zero; ids that
// decrease anywhere make every row zero; the first CTA reports the bits.
// blockIdx.z selects the weight set of the gate/up pair (set 1: w1,
// scales1, biases1 -> y1).
template <int BITS>
__global__ void __launch_bounds__(direct_max_warps(BITS) * 32) gather_qmv_kernel(
    const __nv_bfloat16* __restrict__ x, const uint32_t* __restrict__ w0,
    const uint16_t* __restrict__ scales0, const uint16_t* __restrict__ biases0,
    const uint32_t* __restrict__ w1, const uint16_t* __restrict__ scales1,
    const uint16_t* __restrict__ biases1, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ row_src, __nv_bfloat16* __restrict__ y0,
    __nv_bfloat16* __restrict__ y1, int T, int B, int E, int K, int N, int group,
    long long w_expert_stride, long long sb_expert_stride, int32_t* status) {
    const bool second = blockIdx.z != 0;
    const uint32_t* __restrict__ w = second ? w1 : w0;
    const uint16_t* __restrict__ scales = second ? scales1 : scales0;
    const uint16_t* __restrict__ biases = second ? biases1 : biases0;
    __nv_bfloat16* __restrict__ y = second ? y1 : y0;
    __shared__ int flags;
    if (threadIdx.x == 0) flags = 0;
    __syncthreads();
    int f = 0;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int e = ids[i];
        if (e < 0 || e >= E) f |= 0x1;               // MXQ_DEV_BAD_EXPERT_ID
        if (i > 0 && ids[i - 1] > e) f |= 0x2;       // MXQ_DEV_UNSORTED_IDS
        if (row_src) {
            const int sr = row_src[i];
            if (sr < 0 || sr >= T) f |= 0x4;         // MXQ_DEV_BAD_ROW_SRC
        }
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    const int all = flags;
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && all && status)
        atomicOr(status, all);
    const int r = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int e = ids[r];
    const int src = row_src ? row_src[r] : r;
    if ((all & 0x2) || e < 0 || e >= E || src < 0 || src >= T) {
        if (threadIdx.x < kRows && row0 + (int)threadIdx.x < N)
            y[(long long)r * N + row0 + threadIdx.x] = __float2bfloat16_rn(0.f);
        return;  // the whole CTA: no barrier follows
    }
    qmv_rows_direct<BITS>(x + (long long)src * K, w + (long long)e * w_expert_stride,
                          scales + (long long)e * sb_expert_stride,
                          biases + (long long)e * sb_expert_stride, y + (long long)r * N, K, N,
                          group, row0);
}


// ---------------------------------------------------------------- streaming form

constexpr int kStreamStages = 4;
constexpr int kRedBufs = 4;        // partial-sum buffers between compute warps and reducer
constexpr int kStreamSmemMax = 227 * 1024 - 2048;  // dynamic shared memory (static part aside)
constexpr int kChunkBytes = 48 * 1024;   // codes per stage, about
constexpr int kTargetWarps = 20;
constexpr int kMaxStreamWarps = 20;  // K <= 20480; the activation planes need ~80 registers

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Ask L2 to fetch `bytes` (a multiple of 16) from global memory at `src`
// (16-byte aligned).  Only a hint: it returns nothing and orders nothing, so
// it may be issued before the previous kernel on the stream has finished --
// L2 is where every write lands, so a line fetched early cannot be stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: the kernel launched after this one on the
// stream may start its CTAs as ours finish; it waits in grid_dep_wait()
// until this grid has completed and its writes are visible.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits unless another role already gave up; on its own timeout it raises
// the shared abort flag so that every role winds down without waiting.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              long long budget) {
    if (mbar_poll(bar, parity, budget)) return true;
    const long long t0 = clock64();
    while (!mbar_poll(bar, parity, budget)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

struct StreamShape {
    int nseg;        // 1024-wide K segments
    int phases;      // warps per segment (they take alternate rows)
    int warps;       // compute warps = nseg * phases
    int rows;        // rows per chunk = phases * RPW
    int row_bytes;   // codes bytes per row
    int sb_bytes;    // scale (or bias) bytes per row
    int stage_bytes; // codes + scales + biases, 16-byte aligned pieces
    int x_offset;    // shared-memory offset of the activation copy (after the ring)
    int nchunks;     // chunks over all of N: at most `rows` rows each, a multiple of the grid
    int quantum;     // chunk boundaries fall on multiples of this many rows, so every
                     // chunk's scales and biases are whole 16-byte units
    long long wait_budget;  // pipeline-wait budget in SM cycles
};

// The grouped (segment) form: grid row y is sorted row r = blockIdx.y, the
// GEMV of expert ids[r]'s matrix with activation row row_src[r]; grid z
// selects the weight set of the gate/up pair (set 1: w1, s1, b1 -> y1).
struct StreamSeg {
    const int32_t* ids;      // null: every row multiplies matrix 0 (a dense call with
                             // a few activation rows, one row per grid row)
    const int32_t* row_src;  // null: row r
    const uint32_t* w1;
    const uint16_t* s1;
    const uint16_t* b1;
    __nv_bfloat16* y1;
    int T, B, E;
    long long w_expert_stride;   // words between experts
    long long sb_expert_stride;  // scale/bias entries between experts
};

// Rows go in units of `qu` rows (the shape's quantum); the first `rem` chunks
// of the launch have q + 1 units, the others q units (q = units / nchunks):
// nchunks is a multiple of the grid, so every CTA streams the same number of
// chunks of (within one unit) the same size.  CTA b takes
// chunks b, b + grid, ...:
// at any time the CTAs stream one contiguous window of the weights, which
// keeps all DRAM channels evenly loaded (a contiguous share per CTA instead
// spreads 152 streams at a fixed stride and runs markedly slower).
// QUANT = false: a quantum of one row (the arithmetic is then in rows).
template <bool QUANT>
struct ChunkRows {
    int q, rem, qu;
    __device__ ChunkRows(int N, const StreamShape& sh)
        : q(QUANT ? N / sh.quantum / sh.nchunks : N / sh.nchunks),
          rem(QUANT ? N / sh.quantum % sh.nchunks : N % sh.nchunks),
          qu(QUANT ? sh.quantum : 1) {}
    __device__ int begin(int chunk) const {
        return QUANT ? (chunk * q + min(chunk, rem)) * qu : chunk * q + min(chunk, rem);
    }
};

// ---- exact integer dot products (streaming form)
//
// A lane's 32 activations are written as integers on a common scale:
// x_k = X_k * 2^(emax - 149), emax the largest biased exponent among them,
// so X_k = (bf16 significand) * 2^(e_k - emax + 15) is an integer below
// 2^23 in magnitude (exact unless x_k lies more than 2^15 below the lane's
// largest value; then it is rounded to the nearest integer, an error under
// 2^-23 of the largest).  X_k is split into byte planes
// X_k = a_k 2^16 + b_k 2^8 + c_k (a_k signed, b_k and c_k unsigned), and the
// code sums sum_k q_k a_k, sum_k q_k b_k, sum_k q_k c_k are exact 4-way
// integer dot products (dp4a).  The lane's sum_k x_k q_k is then
// ((A * 256 + B) * 256 + C) * 2^(emax - 149) with one fp32 rounding, so the
// fp32 accumulation of the method is kept and the codes need no conversion
// to floating point at all.

__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Byte planes of a lane's 32 activations, arranged like its codes: for
// 4-bit codes register 2w holds k = 8w, 8w+2, 8w+4, 8w+6 (the even nibbles
// of word w) and register 2w+1 the odd ones; for 8-bit codes register w
// holds k = 4w .. 4w+3; for 2-bit codes register 4w+j holds
// k = 16w+j, 16w+4+j, 16w+8+j, 16w+12+j (code j of each byte of word w).
struct XPlanes {
    uint32_t a[8], b[8], c[8];
};

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Planes of the lane's activations xf (fp32 copies of the bf16 values) on
// the scale 2^(emax - 149).  X_k = rint(x_k * 2^(149 - emax)): the scaling
// is by a power of two, done as two exact multiplications (each factor a
// normal float), and the one rounding only touches values more than 2^15
// below the largest.  Returns emax.
template <int BITS>
__device__ __forceinline__ int make_planes(const float (&xf)[32], XPlanes& P) {
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) m = fmaxf(m, fabsf(xf[k]));
    const int emax = max(1, (int)(__float_as_uint(m) >> 23));  // biased exponent of the largest
    const int p = 149 - emax;                                    // -105 .. 148
    const int p1 = min(p, 127);
    const float s1 = __int_as_float((p1 + 127) << 23);
    const float s2 = __int_as_float((p - p1 + 127) << 23);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int X[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = BITS == 2   ? (r >> 2) * 16 + 4 * i + (r & 3)
                          : BITS == 4 ? (r >> 1) * 8 + 2 * i + (r & 1)
                                      : r * 4 + i;
            X[i] = __float2int_rn((xf[k] * s1) * s2);
        }
        // bytes 0 and 1 of X0..X3, then byte 2 (signed: |X| < 2^23)
        const uint32_t t01 = prmt_b32((uint32_t)X[0], (uint32_t)X[1], 0x5140u);
        const uint32_t t23 = prmt_b32((uint32_t)X[2], (uint32_t)X[3], 0x5140u);
        const uint32_t v01 = prmt_b32((uint32_t)X[0], (uint32_t)X[1], 0x7362u);
        const uint32_t v23 = prmt_b32((uint32_t)X[2], (uint32_t)X[3], 0x7362u);
        P.c[r] = prmt_b32(t01, t23, 0x5410u);
        P.b[r] = prmt_b32(t01, t23, 0x7632u);
        P.a[r] = prmt_b32(v01, v23, 0x5410u);
    }
    return emax;
}

// sum_k X_k q_k over the lane's 32 codes (exact up to the final rounding).
template <int BITS>
__device__ __forceinline__ float lane_dot_int(uint32_t codes_addr, const XPlanes& P) {
    uint32_t wd[8];
    if (BITS == 2) {
        asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(wd[0]), "=r"(wd[1]) : "r"(codes_addr));
    } else {
        uint4 c0;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(c0.x), "=r"(c0.y), "=r"(c0.z), "=r"(c0.w)
                     : "r"(codes_addr));
        wd[0] = c0.x; wd[1] = c0.y; wd[2] = c0.z; wd[3] = c0.w;
        if (BITS == 8) {
            uint4 c1;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(c1.x), "=r"(c1.y), "=r"(c1.z), "=r"(c1.w)
                         : "r"(codes_addr + 16));
            wd[4] = c1.x; wd[5] = c1.y; wd[6] = c1.z; wd[7] = c1.w;
        }
    }
    int A = 0;
    uint32_t B = 0, C = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        uint32_t q;
        if (BITS == 2)
            q = (wd[r >> 2] >> (2 * (r & 3))) & 0x03030303u;
        else if (BITS == 4)
            q = (r & 1) ? (wd[r >> 1] >> 4) & 0x0F0F0F0Fu : wd[r >> 1] & 0x0F0F0F0Fu;
        else
            q = wd[r];
        A = dp4a_su(P.a[r], q, A);
        B = dp4a_uu(P.b[r], q, B);
        C = dp4a_uu(P.c[r], q, C);
    }
    // |A| <= 32*15*128 and B < 32*15*256 (4-bit; less for 2-bit), or
    // 32*255*128 and 32*255*256 (8-bit): A*256 + B stays below 2^31 and
    // converts exactly when below 2^24 (always for 2- and 4-bit)
    const int AB = A * 256 + (int)B;
    return fmaf((float)AB, 256.f, (float)C);
}

template <int BITS, int RPW, bool SEG, bool QUANT>
__global__ void __launch_bounds__((kMaxStreamWarps + 2) * 32, 1)
    qmv_stream_kernel(const __nv_bfloat16* __restrict__ x, const uint32_t* __restrict__ w,
                      const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases,
                      __nv_bfloat16* __restrict__ y, int K, int N, int group,
                      const StreamShape sh, const StreamSeg sg, int32_t* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kStreamStages], empty[kStreamStages], xfull;
    if (SEG) {
        // the ids and source rows may come from the previous kernel
        grid_dep_wait();
        // every CTA checks all ids (there are few): an id outside [0, E) or
        // a source row outside [0, T) makes its row zero, ids that decrease
        // anywhere make every row zero; the first CTA reports the bits
        __shared__ int seg_flags;
        if (threadIdx.x == 0) seg_flags = 0;
        __syncthreads();
        int f = 0;
        for (int i = threadIdx.x; sg.ids && i < sg.B; i += blockDim.x) {
            const int ei = sg.ids[i];
            if (ei < 0 || ei >= sg.E) f |= MXQ_DEV_BAD_EXPERT_ID;
            if (i > 0 && sg.ids[i - 1] > ei) f |= MXQ_DEV_UNSORTED_IDS;
            if (sg.row_src) {
                const int sr = sg.row_src[i];
                if (sr < 0 || sr >= sg.T) f |= MXQ_DEV_BAD_ROW_SRC;
            }
        }
        if (f) atomicOr(&seg_flags, f);
        __syncthreads();
        const int all = seg_flags;
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && all &&
            status)
            atomicOr(status, all);
        const int r = blockIdx.y;
        const bool second = blockIdx.z != 0;
        const int e = sg.ids ? sg.ids[r] : 0;
        const int src = sg.row_src ? sg.row_src[r] : r;
        __nv_bfloat16* const yr = (second ? sg.y1 : y) + (long long)r * N;
        if ((all & MXQ_DEV_UNSORTED_IDS) || e < 0 || e >= sg.E || src < 0 || src >= sg.T) {
            if (blockIdx.x == 0)
                for (int n = threadIdx.x; n < N; n += blockDim.x) yr[n] = __float2bfloat16_rn(0.f);
            return;  // the whole CTA, before any barrier is initialised
        }
        x += (long long)src * K;
        w = (second ? sg.w1 : w) + (long long)e * sg.w_expert_stride;
        scales = (second ? sg.s1 : scales) + (long long)e * sg.sb_expert_stride;
        biases = (second ? sg.b1 : biases) + (long long)e * sg.sb_expert_stride;
        y = yr;
    }
    // per-chunk partial sums of each (row, K segment), handed to the reducer
    // warp through a ring of kRedBufs buffers
    __shared__ float red[kRedBufs][kMaxStreamWarps * 8];
    __shared__ uint64_t redfull[kRedBufs], redempty[kRedBufs];
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = lane_id();
    const uint32_t base = smem_u32(smem);
    const int groups = K / group;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStreamStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], sh.warps);
        }
        mbar_init(&xfull, 1);
        for (int i = 0; i < kRedBufs; ++i) {
            mbar_init(&redfull[i], sh.warps);
            mbar_init(&redempty[i], 1);
        }
        abort_flag = 0;
        mbar_init_fence();
        grid_dep_launch_dependents();
    }
    __syncthreads();

    if (warp == sh.warps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const char* wb = reinterpret_cast<const char*>(w);
            const char* sbp = reinterpret_cast<const char*>(scales);
            const char* bbp = reinterpret_cast<const char*>(biases);
            const ChunkRows<QUANT> cr(N, sh);
            // while the previous kernel finishes, have L2 fetch this CTA's
            // first chunk, so that the first copy after the wait does not
            // start from DRAM latency
            if ((int)blockIdx.x < sh.nchunks) {
                const int r0 = cr.begin(blockIdx.x);
                const int rows = cr.begin(blockIdx.x + 1) - r0;
                bulk_prefetch_l2(wb + (long long)r0 * sh.row_bytes, (uint32_t)(rows * sh.row_bytes));
                bulk_prefetch_l2(sbp + (long long)r0 * sh.sb_bytes, (uint32_t)(rows * sh.sb_bytes));
                bulk_prefetch_l2(bbp + (long long)r0 * sh.sb_bytes, (uint32_t)(rows * sh.sb_bytes));
            }
            // every read into shared memory, and every read of x or write
            // of y, comes after the previous kernel on the stream completed
            grid_dep_wait();
            // the activations first: copies issued by one SM are served in
            // order, so x arrives ahead of the weight stream instead of
            // queueing behind tens of megabytes of it
            expect_tx(&xfull, (uint32_t)(K * 2));
            bulk_g2s(base + sh.x_offset, x, (uint32_t)(K * 2), &xfull);
            int j = 0;  // chunks issued
            for (;; ++j) {
                const int chunk = blockIdx.x + j * gridDim.x;
                if (chunk >= sh.nchunks) break;
                const int st = j % kStreamStages;
                // a compute warp that gave up still hands its stage back:
                // after an abort the stage's last copy may not have landed,
                // so nothing more is issued into the ring
                if (j >= kStreamStages &&
                    (!wait_or_abort(&empty[st], ((j / kStreamStages) + 1) & 1, &abort_flag,
                                    sh.wait_budget) ||
                     *static_cast<volatile int*>(&abort_flag)))
                    break;
                const int r0 = cr.begin(chunk);
                const int rows = cr.begin(chunk + 1) - r0;
                const uint32_t cb = (uint32_t)(rows * sh.row_bytes);
                const uint32_t sbb = (uint32_t)(rows * sh.sb_bytes);
                const uint32_t dst = base + st * sh.stage_bytes;
                expect_tx(&full[st], cb + 2 * sbb);
                bulk_g2s(dst, wb + (long long)r0 * sh.row_bytes, cb, &full[st]);
                bulk_g2s(dst + sh.rows * sh.row_bytes, sbp + (long long)r0 * sh.sb_bytes, sbb,
                         &full[st]);
                bulk_g2s(dst + sh.rows * (sh.row_bytes + sh.sb_bytes),
                         bbp + (long long)r0 * sh.sb_bytes, sbb, &full[st]);
            }
            // every copy issued has landed before this CTA can exit (the
            // compute warps wait for them too, unless they gave up)
            const bool landed =
                mbar_wait(&xfull, 0) && drain_ring(full, kStreamStages, j, kStreamStages);
            if (!landed && status) atomicOr(status, 0x8 /* MXQ_DEV_TIMEOUT */);
        }
        return;
    }
    if (warp == sh.warps + 1) {
        // ---------------------------------------------------------------- reducer
        // sums each row's K-segment partials in a fixed order and stores y,
        // so the compute warps go on to the next chunk without waiting for
        // one another
        const ChunkRows<QUANT> cr(N, sh);
        for (int j = 0;; ++j) {
            const int chunk = blockIdx.x + j * gridDim.x;
            if (chunk >= sh.nchunks) break;
            const int buf = j % kRedBufs;
            if (!wait_or_abort(&redfull[buf], (j / kRedBufs) & 1, &abort_flag, sh.wait_budget)) break;
            const int r0 = cr.begin(chunk);
            const int rows = cr.begin(chunk + 1) - r0;
            for (int r = lane; r < rows; r += 32) {
                float acc = 0.f;
                for (int sgi = 0; sgi < sh.nseg; ++sgi) acc += red[buf][r * sh.nseg + sgi];
                y[r0 + r] = __float2bfloat16_rn(acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&redempty[buf]);
        }
        return;
    }

    // -------------------------------------------------------------------- compute
    grid_dep_wait();  // x may come from the previous kernel, y may be read by it
    const int seg = warp % sh.nseg;
    const int phase = warp / sh.nseg;
    const int k0 = seg * 1024 + lane * 32;   // this lane's 32 values
    const bool active = k0 < K;
    // 3- and 6-bit codes are cut out of the row's bit stream into floats
    // 1 + q * 2^-7 (the direct-load kernel's arithmetic), so those widths keep
    // the activations as fp32 pairs; the others use exact integer planes
    constexpr bool kFloatCodes = BITS == 3 || BITS == 6;
    XPlanes P;
    float2 x2[16];
    float X = 0.f;          // sum of the lane's activations (bias term)
    float xscale = 0.f;     // 2^(emax - 149)
    {
        uint32_t u[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] = 0;
        if (wait_or_abort(&xfull, 0, &abort_flag, sh.wait_budget) && active) {
            const uint32_t xs = base + sh.x_offset + (uint32_t)k0 * 2;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(u[4 * c]), "=r"(u[4 * c + 1]), "=r"(u[4 * c + 2]),
                               "=r"(u[4 * c + 3])
                             : "r"(xs + c * 16));
        }
        float xf[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            xf[2 * j] = __uint_as_float(u[j] << 16);
            xf[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
            X += xf[2 * j] + xf[2 * j + 1];
        }
        if (kFloatCodes) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x2[j] = make_float2(xf[2 * j], xf[2 * j + 1]);
        } else {
            const int emax = make_planes<BITS>(xf, P);
            // 2^(emax - 149): a normal float from emax = 23 on, else subnormal
            xscale = __int_as_float(emax >= 23 ? (emax - 22) << 23 : 1 << emax);
        }
    }
    const int g = k0 / group;
    const uint32_t lane_code_off = (uint32_t)(seg * 1024 + lane * 32) * BITS / 8;

    const ChunkRows<QUANT> cr(N, sh);
    for (int j = 0;; ++j) {
        const int chunk = blockIdx.x + j * gridDim.x;
        if (chunk >= sh.nchunks) break;
        const int st = j % kStreamStages;
        const bool have =
            wait_or_abort(&full[st], (j / kStreamStages) & 1, &abort_flag, sh.wait_budget);
        const uint32_t sbase = base + st * sh.stage_bytes;
        const uint32_t s_off = sbase + sh.rows * sh.row_bytes;
        const uint32_t b_off = s_off + sh.rows * sh.sb_bytes;
        const int r0 = cr.begin(chunk);
        const int rows = cr.begin(chunk + 1) - r0;
        float part[RPW];
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
            const int r = phase + q * sh.phases;   // row within the chunk
            part[q] = 0.f;
            if (have && active && r < rows) {
                const uint32_t caddr = sbase + r * sh.row_bytes + lane_code_off;
                float xq;  // sum over the lane's codes of x_k * q_k
                if (kFloatCodes) {
                    uint32_t wd[6] = {0u, 0u, 0u, 0u, 0u, 0u};
                    if (BITS == 3) {
                        // 12 bytes at a 4-byte aligned offset
#pragma unroll
                        for (int i = 0; i < 3; ++i)
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wd[i]) : "r"(caddr + 4 * i));
                    } else {
                        // 24 bytes at an 8-byte aligned offset
#pragma unroll
                        for (int i = 0; i < 3; ++i)
                            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                                         : "=r"(wd[2 * i]), "=r"(wd[2 * i + 1])
                                         : "r"(caddr + 8 * i));
                    }
                    xq = (dot_chunk_stream<BITS>(wd, x2) - X) * 128.f;
                } else {
                    xq = lane_dot_int<BITS>(caddr, P) * xscale;
                }
                uint16_t sv, bv;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(sv) : "r"(s_off + (r * groups + g) * 2));
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(bv) : "r"(b_off + (r * groups + g) * 2));
                const float s = bf16_bits_to_float(sv), b = bf16_bits_to_float(bv);
                part[q] = fmaf(s, xq, b * X);
            }
        }
        // all shared reads of this stage are consumed: hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        // reduce-scatter over lanes: row q ends on lanes q * (32 / RPW) ...
#pragma unroll
        for (int half = RPW / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = upper ? part[i] : part[i + half];
                const float keep = upper ? part[i + half] : part[i];
                part[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
            }
        }
#pragma unroll
        for (int off = 16 / RPW; off >= 1; off >>= 1)
            part[0] += __shfl_xor_sync(0xFFFFFFFFu, part[0], off);
        const int span = 32 / RPW;
        const int buf = j % kRedBufs;
        // the reducer must be done with this buffer's previous chunk
        const bool free_buf =
            j < kRedBufs ||
            wait_or_abort(&redempty[buf], ((j / kRedBufs) + 1) & 1, &abort_flag, sh.wait_budget);
        if (free_buf && (lane & (span - 1)) == 0) {
            const int q = lane / span;
            const int r = phase + q * sh.phases;
            red[buf][r * sh.nseg + seg] = part[0];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&redfull[buf]);
    }
    if (threadIdx.x == 0 && abort_flag && status) atomicOr(status, 0x8 /* MXQ_DEV_TIMEOUT */);
}

template <int BITS, bool SEG>
cudaError_t launch_stream(const __nv_bfloat16* x, const uint32_t* w, const uint16_t* s,
                          const uint16_t* b, __nv_bfloat16* y, int K, int N, int group, int rpw,
                          const StreamShape& sh, const StreamSeg& seg, dim3 grid,
                          int32_t* status, cudaStream_t stream) {
    const int smem = sh.x_offset + K * 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((sh.warps + 2) * 32);  // compute warps, producer, reducer
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the segment form always takes the general chunk arithmetic
    constexpr bool kAnyQuant = SEG;
#define MXQ_STREAM_CASE(R)                                                                      \
    case R: {                                                                                   \
        const auto kern = (kAnyQuant || sh.quantum > 1) ? qmv_stream_kernel<BITS, R, SEG, true>  \
                                                        : qmv_stream_kernel<BITS, R, SEG, SEG>;  \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                             smem);                                             \
        if (e != cudaSuccess) return e;                                                         \
        e = cudaLaunchKernelEx(&cfg, kern, x, w, s, b, y, K, N, group, sh, seg, status);        \
        if (e != cudaSuccess) return e;                                                         \
        break;                                                                                  \
    }
    switch (rpw) {
        MXQ_STREAM_CASE(1)
        MXQ_STREAM_CASE(2)
        MXQ_STREAM_CASE(4)
        MXQ_STREAM_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef MXQ_STREAM_CASE
    return cudaGetLastError();
}

// The streaming GEMV's shape for a [N, K] matrix, or false when the shape
// does not fit it (the direct-load kernel then runs): K % 64 == 0 (whole
// 16-byte code rows; the callers check K % 128 at 3 bits), K <= 20480,
// scales/biases 16-byte aligned, and N a multiple of the row quantum that
// makes a chunk's scales (and biases) whole 16-byte units.  `ctas` is the
// number of CTAs that will stream this matrix (the chunk count is made a
// multiple of it); a negative value -c means min(c, the chunks needed), and
// the number used is returned in it.
bool stream_shape(int K, int N, int bits, int group, const void* scales, const void* biases,
                  int& ctas, StreamShape& sh, int& rpw) {
    const bool sb_aligned = (reinterpret_cast<uintptr_t>(scales) % 16 == 0) &&
                            (reinterpret_cast<uintptr_t>(biases) % 16 == 0);
    const int nseg = (K + 1023) / 1024;
    if (K % 64 != 0 || nseg > kMaxStreamWarps || !sb_aligned) return false;
    sh.nseg = nseg;
    sh.phases = kTargetWarps / nseg > 1 ? kTargetWarps / nseg : 1;
    if (sh.phases * nseg > kMaxStreamWarps) sh.phases = kMaxStreamWarps / nseg;
    sh.warps = sh.phases * nseg;
    sh.row_bytes = K * bits / 8;
    sh.sb_bytes = (K / group) * 2;
    // rows per unit: 16 / gcd(sb_bytes, 16)
    int g = sh.sb_bytes & 15;
    sh.quantum = g == 0 ? 1 : (g % 8 == 0 ? 2 : (g % 4 == 0 ? 4 : 8));
    if (N % sh.quantum != 0) return false;
    rpw = kChunkBytes / (sh.row_bytes * sh.phases);
    rpw = rpw >= 8 ? 8 : rpw >= 4 ? 4 : rpw >= 2 ? 2 : 1;
    // the ring and the activation copy share the 227 KB of shared memory
    while (rpw > 1 && kStreamStages * sh.phases * rpw * (sh.row_bytes + 2 * sh.sb_bytes) + K * 2 >
                          kStreamSmemMax)
        rpw /= 2;
    // a stage holds at most sh.rows rows, a multiple of the quantum
    sh.rows = sh.phases * rpw / sh.quantum * sh.quantum;
    if (sh.rows < sh.quantum) return false;
    sh.stage_bytes = sh.rows * (sh.row_bytes + 2 * sh.sb_bytes);  // pieces are 16-byte multiples
    sh.x_offset = kStreamStages * sh.stage_bytes;
    sh.wait_budget = wait_budget_cycles();
    // chunks of at most sh.rows rows, as many as a multiple of the CTAs
    const int units = N / sh.quantum;
    const int per_chunk = sh.rows / sh.quantum;
    sh.nchunks = (units + per_chunk - 1) / per_chunk;
    if (ctas < 0) ctas = sh.nchunks < -ctas ? sh.nchunks : -ctas;
    sh.nchunks = (sh.nchunks + ctas - 1) / ctas * ctas;
    if (sh.nchunks > units) sh.nchunks = units;
    return true;
}

template <bool SEG>
cudaError_t launch_stream_bits(int bits, const __nv_bfloat16* x, const uint32_t* w,
                               const uint16_t* s, const uint16_t* b, __nv_bfloat16* y, int K,
                               int N, int group, int rpw, const StreamShape& sh,
                               const StreamSeg& seg, dim3 grid, int32_t* status,
                               cudaStream_t stream) {
    switch (bits) {
        case 2: return launch_stream<2, SEG>(x, w, s, b, y, K, N, group, rpw, sh, seg, grid, status, stream);
        case 3: return launch_stream<3, SEG>(x, w, s, b, y, K, N, group, rpw, sh, seg, grid, status, stream);
        case 4: return launch_stream<4, SEG>(x, w, s, b, y, K, N, group, rpw, sh, seg, grid, status, stream);
        case 6: return launch_stream<6, SEG>(x, w, s, b, y, K, N, group, rpw, sh, seg, grid, status, stream);
        case 8: return launch_stream<8, SEG>(x, w, s, b, y, K, N, group, rpw, sh, seg, grid, status, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gather_qmv(const void* x, const uint32_t* w, const void* scales,
                              const void* biases, const uint32_t* w1, const void* scales1,
                              const void* biases1, const int32_t* expert_ids,
                              const int32_t* row_src, void* y, void* y1, int sets, int T, int B,
                              int E, int K, int N, int bits, int group, int sms,
                              bool stream_form, int32_t* status, cudaStream_t stream) {
    const long long wst = (long long)N * K * bits / 32;
    const long long sbst = (long long)N * (K / group);
    if (stream_form) {
        // the streaming GEMV, one grid row per sorted row (and weight set):
        // each sorted row's expert matrix streams through `ctas` CTAs
        StreamShape sh;
        int rpw = 1;
        int ctas = sms / (B * sets) > 1 ? sms / (B * sets) : 1;
        const bool set1_aligned = sets < 2 || (reinterpret_cast<uintptr_t>(scales1) % 16 == 0 &&
                                               reinterpret_cast<uintptr_t>(biases1) % 16 == 0);
        if (set1_aligned && stream_shape(K, N, bits, group, scales, biases, ctas, sh, rpw)) {
            StreamSeg seg;
            seg.ids = expert_ids;
            seg.row_src = row_src;
            seg.w1 = w1;
            seg.s1 = static_cast<const uint16_t*>(scales1);
            seg.b1 = static_cast<const uint16_t*>(biases1);
            seg.y1 = static_cast<__nv_bfloat16*>(y1);
            seg.T = T;
            seg.B = B;
            seg.E = E;
            seg.w_expert_stride = wst;
            seg.sb_expert_stride = sbst;
            return launch_stream_bits<true>(
                bits, static_cast<const __nv_bfloat16*>(x), w, static_cast<const uint16_t*>(scales),
                static_cast<const uint16_t*>(biases), static_cast<__nv_bfloat16*>(y), K, N, group,
                rpw, sh, seg, dim3(ctas, B, sets), status, stream);
        }
        return cudaErrorNotSupported;  // the shape does not fit the streaming form
    }
    // the direct-load GEMV: grid (N / 16, sorted rows, weight sets)
    const int seg_k = bits == 8 ? 512 : 1024;
    const int nseg_g = (K + seg_k - 1) / seg_k;
    const int max_warps = direct_max_warps(bits);
    const int passes = (nseg_g + max_warps - 1) / max_warps;
    const int warps = (nseg_g + passes - 1) / passes;
    const dim3 grid((N + kRows - 1) / kRows, B, sets);
    const dim3 block(32 * warps);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* sb = static_cast<const uint16_t*>(scales);
    const auto* bb = static_cast<const uint16_t*>(biases);
    const auto* sb1 = static_cast<const uint16_t*>(scales1);
    const auto* bb1 = static_cast<const uint16_t*>(biases1);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    auto* yb1 = static_cast<__nv_bfloat16*>(y1);
#define MXQ_GATHER_QMV(BB)                                                                        \
    gather_qmv_kernel<BB><<<grid, block, 0, stream>>>(xb, w, sb, bb, w1, sb1, bb1, expert_ids,     \
                                                      row_src, yb, yb1, T, B, E, K, N, group, wst, \
                                                      sbst, status)
    if (bits == 2)
        MXQ_GATHER_QMV(2);
    else if (bits == 3)
        MXQ_GATHER_QMV(3);
    else if (bits == 6)
        MXQ_GATHER_QMV(6);
    else if (bits == 4)
        MXQ_GATHER_QMV(4);
    else
        MXQ_GATHER_QMV(8);
#undef MXQ_GATHER_QMV
    return cudaGetLastError();
}

cudaError_t launch_qmv_rows(const void* x, const uint32_t* w, const void* scales,
                            const void* biases, void* y, int M, int K, int N, int bits, int group,
                            int sms, int32_t* status, cudaStream_t stream) {
    StreamShape sh;
    int rpw = 1;
    int ctas = sms / M > 1 ? sms / M : 1;
    if (!stream_shape(K, N, bits, group, scales, biases, ctas, sh, rpw))
        return cudaErrorNotSupported;
    StreamSeg seg = {};
    seg.T = M;
    seg.B = M;
    seg.E = 1;
    return launch_stream_bits<true>(bits, static_cast<const __nv_bfloat16*>(x), w,
                                    static_cast<const uint16_t*>(scales),
                                    static_cast<const uint16_t*>(biases),
                                    static_cast<__nv_bfloat16*>(y), K, N, group, rpw, sh, seg,
                                    dim3(ctas, M, 1), status, stream);
}

cudaError_t launch_qmv(const void* x, const uint32_t* w, const void* scales, const void* biases,
                       void* y, int K, int N, int bits, int group, int sms, int32_t* status,
                       cudaStream_t stream) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* sb = static_cast<const uint16_t*>(scales);
    const auto* bb = static_cast<const uint16_t*>(biases);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    StreamShape sh;
    int rpw = 1, ctas = -sms;
    if (stream_shape(K, N, bits, group, scales, biases, ctas, sh, rpw)) {
        const StreamSeg none = {};
        return launch_stream_bits<false>(bits, xb, w, sb, bb, yb, K, N, group, rpw, sh, none,
                                         dim3(ctas), status, stream);
    }
    const int seg_k = bits == 8 ? 512 : 1024;
    const int nseg_g = (K + seg_k - 1) / seg_k;
    // as few passes over the segments as the warp limit allows, spread evenly
    const int max_warps = direct_max_warps(bits);
    const int passes = (nseg_g + max_warps - 1) / max_warps;
    const int warps = (nseg_g + passes - 1) / passes;
    const dim3 grid((N + kRows - 1) / kRows);
    const dim3 block(32 * warps);
    if (bits == 2)
        qmv_generic_kernel<2><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N, group);
    else if (bits == 3)
        qmv_generic_kernel<3><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N, group);
    else if (bits == 6)
        qmv_generic_kernel<6><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N, group);
    else if (bits == 4)
        qmv_generic_kernel<4><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N, group);
    else
        qmv_generic_kernel<8><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N, group);
    return cudaGetLastError();
}

}  // namespace mxq
