// Affine group-wise encoder: float weights -> packed codes, bf16 scales and
// biases (the stored format of mlxcel issue #1536, Baseline section: "affine
// 4-bit / group 64"; 8-bit codes are unsigned bytes; 2-, 3- and 6-bit codes
// continue the same little-endian bit stream per row, so 3- and 6-bit codes
// may straddle words; groups of 32 and 128 consecutive k use the same rule).
//
// Per (row n, group g of GROUP consecutive k): mn, mx = the group's minimum and
// maximum (-0 read as +0); s = bf16(RN(RN(mx - mn) / (2^bits - 1))) and
// b = bf16(mn), both rounded to nearest even; then every code is
// q = clamp(rint(RN(RN(w - b) / s)), 0, 2^bits - 1) against the stored bf16 s
// and b (q = 0 when s == 0).  Every decision is taken in binary32 with
// IEEE-rounded subtraction and division, so the result is the same bit for
// bit wherever the same rule is evaluated in binary32.
//
// One warp per row: each lane holds 8 consecutive values of a 256-wide block
// (two 16-byte loads), GROUP / 8 lanes make a group (4, 8 or 16), so a
// group's minimum and maximum take two to four shuffle steps and each lane
// packs its own codes (2, 3, 4, 6 or 8 bytes at 2, 3, 4, 6 or 8 bits).
// HBM-bound: 4 bytes read per weight, bits/8 written.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kEncWarps = 8;  // rows per CTA

template <int BITS, int GROUP>
__global__ void __launch_bounds__(kEncWarps * 32) quantize_kernel(const float* __restrict__ W,
                                                                 uint32_t* __restrict__ codes,
                                                                 uint16_t* __restrict__ scales,
                                                                 uint16_t* __restrict__ biases,
                                                                 int N, int K) {
    constexpr int kLevels = (1 << BITS) - 1;
    constexpr int kGroupLanes = GROUP / 8;
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * kEncWarps + (threadIdx.x >> 5);
    if (n >= N) return;  // the whole warp
    const float* row = W + (long long)n * K;
    const int groups = K / GROUP;
    // four 256-wide blocks per round: all their loads are issued before any
    // arithmetic, so each lane keeps 128 bytes in flight
    constexpr int kBlocks = 4;
    for (int kb = 0; kb < K; kb += 256 * kBlocks) {
        float v[kBlocks][8];
#pragma unroll
        for (int u = 0; u < kBlocks; ++u) {
            const int k = kb + u * 256 + lane * 8;
            if (k < K) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(row + k));
                const float4 b = __ldg(reinterpret_cast<const float4*>(row + k + 4));
                v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                v[u][4] = b.x; v[u][5] = b.y; v[u][6] = b.z; v[u][7] = b.w;
            }
        }
#pragma unroll
        for (int u = 0; u < kBlocks; ++u) {
            const int k0 = kb + u * 256;
            if (k0 >= K) break;  // warp-uniform
            const int k = k0 + lane * 8;
            const bool active = k < K;  // K % GROUP == 0: whole groups of lanes drop out
            float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
            if (active) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float t = __fadd_rn(v[u][i], 0.0f);  // -0 -> +0
                    mn = fminf(mn, t);
                    mx = fmaxf(mx, t);
                }
            }
#pragma unroll
            for (int off = 1; off < kGroupLanes; off <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            }
            if (!active) continue;
            const __nv_bfloat16 sb =
                __float2bfloat16_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)kLevels));
            const __nv_bfloat16 bb = __float2bfloat16_rn(mn);
            const float s = __bfloat162float(sb), b = __bfloat162float(bb);
            uint32_t q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float r = 0.f;
                if (s != 0.f)
                    r = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v[u][i], b), s)), 0.f), (float)kLevels);
                q[i] = (uint32_t)r;
            }
            if (BITS == 3 || BITS == 6) {
                // the lane's 8 codes are 3 or 6 whole bytes of the row's bit
                // stream, starting at byte k * BITS / 8 (k is a multiple of 8)
                uint64_t v = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) v |= (uint64_t)q[i] << (BITS * i);
                uint8_t* row = reinterpret_cast<uint8_t*>(codes) + (long long)n * (K / 8) * BITS;
                uint8_t* dst = row + (long long)(k / 8) * BITS;
#pragma unroll
                for (int i = 0; i < BITS; ++i) dst[i] = (uint8_t)(v >> (8 * i));
            } else if (BITS == 2) {
                uint32_t half = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) half |= q[i] << (2 * i);
                // row n has K / 8 halves of 16 bits; lane's k is a multiple of 8
                reinterpret_cast<uint16_t*>(codes)[(long long)n * (K / 8) + k / 8] = (uint16_t)half;
            } else if (BITS == 4) {
                uint32_t word = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) word |= q[i] << (4 * i);
                codes[(long long)n * (K / 8) + k / 8] = word;
            } else {
                uint2 words;
                words.x = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
                words.y = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
                *reinterpret_cast<uint2*>(codes + (long long)n * (K / 4) + k / 4) = words;
            }
            if ((lane & (kGroupLanes - 1)) == 0) {
                const long long gi = (long long)n * groups + k / GROUP;
                scales[gi] = __bfloat16_as_ushort(sb);
                biases[gi] = __bfloat16_as_ushort(bb);
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const float* W, uint32_t* codes, void* scales, void* biases, int N,
                            int K, int bits, int group, cudaStream_t stream) {
    const dim3 grid((N + kEncWarps - 1) / kEncWarps);
    const dim3 block(kEncWarps * 32);
    auto* s = static_cast<uint16_t*>(scales);
    auto* b = static_cast<uint16_t*>(biases);
#define MXQ_ENC_CASE(G)                                                                \
    case G:                                                                            \
        if (bits == 2)                                                                 \
            quantize_kernel<2, G><<<grid, block, 0, stream>>>(W, codes, s, b, N, K);   \
        else if (bits == 3)                                                            \
            quantize_kernel<3, G><<<grid, block, 0, stream>>>(W, codes, s, b, N, K);   \
        else if (bits == 6)                                                            \
            quantize_kernel<6, G><<<grid, block, 0, stream>>>(W, codes, s, b, N, K);   \
        else if (bits == 4)                                                            \
            quantize_kernel<4, G><<<grid, block, 0, stream>>>(W, codes, s, b, N, K);   \
        else                                                                           \
            quantize_kernel<8, G><<<grid, block, 0, stream>>>(W, codes, s, b, N, K);   \
        break;
    switch (group) {
        MXQ_ENC_CASE(32)
        MXQ_ENC_CASE(64)
        MXQ_ENC_CASE(128)
        default: return cudaErrorInvalidValue;
    }
#undef MXQ_ENC_CASE
    return cudaGetLastError();
}

}  // namespace mxq
