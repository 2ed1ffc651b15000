// Decode GEMV for affine group-wise quantized weights (M = 1).
//
// mlxcel issue #1536, Diagnosis item 3: the qmv kernel must accumulate in
// float at every bit width; it is the HBM-bound half of decoding (Baseline
// section: the qmv share of a decode step moves ~15 GB of codes).
//
// Layout of the work:
//  * a lane owns 16 bytes of codes per row (32 four-bit or 16 eight-bit
//    codes, always inside one group of 64), so a warp covers a K segment of
//    1024 (4-bit) or 512 (8-bit) values with one coalesced 512-byte load per
//    row;
//  * a CTA has one warp per K segment and owns a block of ROWS output rows;
//    each lane keeps its 32/16 activations in registers for all the rows;
//  * the codes are turned into floats 1 + q*2^-7 (4-bit) or 1 + q*2^-15
//    (8-bit) by placing them in the mantissa of a constant with one byte
//    permute each; the lane's products are summed in fp32 and the affine
//    terms are applied once per lane and row:
//        sum_k x_k (s q_k + b) = s * 2^p * (sum_k x_k v_k - X) + b * X,
//    with X = sum_k x_k over the lane's values, p = 7 or 15;
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

template <int BITS>
__global__ void __launch_bounds__(kMaxWarps * 32) qmv_kernel(const __nv_bfloat16* __restrict__ x,
                                                   const uint32_t* __restrict__ w,
                                                   const uint16_t* __restrict__ scales,
                                                   const uint16_t* __restrict__ biases,
                                                   __nv_bfloat16* __restrict__ y, int K, int N) {
    constexpr int kCodesPerLane = 128 / BITS;          // 32 or 16
    constexpr int kSegK = 32 * kCodesPerLane;          // 1024 or 512
    constexpr float kUnscale = BITS == 4 ? 128.f : 32768.f;
    __shared__ float red[kMaxWarps][kRows];

    const int lane = lane_id();
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row0 = blockIdx.x * kRows;
    const int nseg = (K + kSegK - 1) / kSegK;
    const long long words_per_row = (long long)K * BITS / 32;
    const int groups = K / 64;

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
        const int g = k0 / 64;
        const long long wofs = (long long)k0 * BITS / 32;  // word offset in a row

#pragma unroll
        for (int r0 = 0; r0 < kRows; r0 += kUnroll) {
            uint4 c[kUnroll];
            float s[kUnroll], b[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int n = row0 + r0 + u;
                if (n < N) {
                    c[u] = ldg_stream(reinterpret_cast<const uint4*>(w + n * words_per_row + wofs));
                    s[u] = bf16_bits_to_float(__ldg(scales + (long long)n * groups + g));
                    b[u] = bf16_bits_to_float(__ldg(biases + (long long)n * groups + g));
                } else {
                    c[u] = make_uint4(0, 0, 0, 0);
                    s[u] = 0.f;
                    b[u] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float A = BITS == 4 ? dot_chunk4(c[u], x2) : dot_chunk8(c[u], x2);
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

}  // namespace

cudaError_t launch_qmv(const void* x, const uint32_t* w, const void* scales, const void* biases,
                       void* y, int K, int N, int bits, cudaStream_t stream) {
    const int seg_k = bits == 4 ? 1024 : 512;
    const int nseg = (K + seg_k - 1) / seg_k;
    // as few passes over the segments as the warp limit allows, spread evenly
    const int passes = (nseg + kMaxWarps - 1) / kMaxWarps;
    const int warps = (nseg + passes - 1) / passes;
    const dim3 grid((N + kRows - 1) / kRows);
    const dim3 block(32 * warps);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* sb = static_cast<const uint16_t*>(scales);
    const auto* bb = static_cast<const uint16_t*>(biases);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    if (bits == 4)
        qmv_kernel<4><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N);
    else
        qmv_kernel<8><<<grid, block, 0, stream>>>(xb, w, sb, bb, yb, K, N);
    return cudaGetLastError();
}

}  // namespace mxq
