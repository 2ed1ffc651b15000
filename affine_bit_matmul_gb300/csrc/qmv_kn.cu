// Decode GEMV for the other operand layout: w stored [K, N], row k holding
// the packed codes of every output n (the same little-endian bit stream
// along n), groups of G consecutive n per scale/bias pair:
//
//     y[n] = sum_k x[k] * (s[k, n/G] * q[k, n] + b[k, n/G])
//
// (mlxcel PR #1562, What changed: the grouped GEMM is checked for both
// operand layouts; issue #1536, Diagnosis item 3: float accumulation at every
// width.)  HBM-bound like the [N, K] GEMV.
//
// Work split.  A cluster of S <= 8 CTAs owns 256 output columns; its CTAs
// take consecutive ranges of K.  In a CTA of 8 warps, lane l owns columns
// 32 * (l % 8) .. + 31 of the block and row slot l / 8, so one warp load
// covers four rows of 128 (4-bit) bytes and each lane keeps eight rows of
// codes in flight.  Per row a lane forms xs = x_k * s[k, g] once for its 32
// columns (all in one group) and accumulates xs * v_n in fp32 pairs
// (fma.rn.f32x2), where v_n = 1 + q_n * 2^-p is the code placed in a float
// mantissa by one byte permute; sum_k xs q_n = 2^p * (sum_k xs v_n - sum_k
// xs), and the bias term sum_k x_k b[k, g] is kept apart.  Partials are
// added in a fixed order: across the four row slots of a warp by shuffles,
// across warps through shared memory, across the cluster through
// distributed shared memory in rank order, so the result does not depend on
// timing.  No waits other than the two cluster barriers.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kKnWarps = 8;
constexpr int kKnThreads = kKnWarps * 32;
constexpr int kKnCols = 256;        // output columns per cluster
constexpr int kKnRowsPerStep = 32;  // rows a CTA covers per step: 8 warps x 4 row slots
constexpr int kKnMaxCluster = 8;

__device__ __forceinline__ uint32_t kn_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void kn_ffma2(float2& acc, float2 a, float2 b) {
    unsigned long long A = *reinterpret_cast<unsigned long long*>(&a);
    unsigned long long B = *reinterpret_cast<unsigned long long*>(&b);
    unsigned long long C = *reinterpret_cast<unsigned long long*>(&acc);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(C) : "l"(A), "l"(B));
    acc = *reinterpret_cast<float2*>(&C);
}

__device__ __forceinline__ void kn_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t kn_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float kn_ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Words of a lane's 32 codes in one row: 2, 4 or 8 at 2, 4 or 8 bits.
template <int BITS>
struct KnWords {
    uint32_t w[BITS];
};

template <int BITS>
__device__ __forceinline__ KnWords<BITS> kn_load(const uint32_t* p) {
    KnWords<BITS> r;
    if (BITS == 2) {
        uint2 v;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                     : "=r"(v.x), "=r"(v.y)
                     : "l"(p));
        r.w[0] = v.x;
        r.w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < BITS / 4; ++i) {
            uint4 v;
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "l"(p + 4 * i));
            r.w[4 * i] = v.x;
            r.w[4 * i + 1] = v.y;
            r.w[4 * i + 2] = v.z;
            r.w[4 * i + 3] = v.w;
        }
    }
    return r;
}

// acc[j] += (xs, xs) * (v_{2j}, v_{2j+1}) over the lane's 32 columns,
// v_n = 1 + q_n * 2^-7 (2- and 4-bit) or 1 + q_n * 2^-15 (8-bit).
template <int BITS>
__device__ __forceinline__ void kn_accumulate(const KnWords<BITS>& c, float xs, float2 (&acc)[16]) {
    const float2 xs2 = make_float2(xs, xs);
    if (BITS == 4) {
        // word j holds columns 8j .. 8j+7; bytes of lo / hi are the even / odd nibbles
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = (c.w[j] & 0x0F0F0F0Fu) | 0x80808080u;
            const uint32_t hi = ((c.w[j] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t sel = 0x7044u | (uint32_t(b) << 8);
                float2 v;
                v.x = __uint_as_float(kn_prmt(lo, 0x3F000000u, sel));
                v.y = __uint_as_float(kn_prmt(hi, 0x3F000000u, sel));
                kn_ffma2(acc[4 * j + b], xs2, v);
            }
        }
    } else if (BITS == 2) {
        // word j holds columns 16j .. 16j+15; byte i of plane t holds code 4i + t
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint32_t pe = ((c.w[j] >> (4 * t)) & 0x03030303u) | 0x80808080u;
                const uint32_t po = ((c.w[j] >> (4 * t + 2)) & 0x03030303u) | 0x80808080u;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t sel = 0x7044u | (uint32_t(i) << 8);
                    float2 v;
                    v.x = __uint_as_float(kn_prmt(pe, 0x3F000000u, sel));
                    v.y = __uint_as_float(kn_prmt(po, 0x3F000000u, sel));
                    kn_ffma2(acc[8 * j + 2 * i + t], xs2, v);
                }
            }
        }
    } else {
        // word j holds columns 4j .. 4j+3, one byte each
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float2 v;
                v.x = __uint_as_float(kn_prmt(c.w[j], 0x3F800000u, 0x7604u | (uint32_t(2 * b) << 4)));
                v.y = __uint_as_float(kn_prmt(c.w[j], 0x3F800000u, 0x7604u | (uint32_t(2 * b + 1) << 4)));
                kn_ffma2(acc[2 * j + b], xs2, v);
            }
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kKnThreads, 2)
    qmv_kn_kernel(const __nv_bfloat16* __restrict__ x, const uint32_t* __restrict__ w,
                  const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases,
                  __nv_bfloat16* __restrict__ y, int K, int N, int group, int rows_per_rank) {
    constexpr int kU = BITS == 8 ? 4 : 8;  // rows of codes in flight per lane
    constexpr float kUnscale = BITS == 8 ? 32768.f : 128.f;
    __shared__ float part[kKnWarps][kKnCols];
    __shared__ float cta_part[kKnCols];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = lane & 7;    // 32-column sub-block
    const int t = lane >> 3;   // row slot
    const int n0 = blockIdx.x * kKnCols + c * 32;
    const bool col_ok = n0 < N;  // N % 64 == 0: whole lanes
    const int rank = (int)kn_cluster_rank();
    const int k_begin = rank * rows_per_rank;
    const int k_end = min(K, k_begin + rows_per_rank);
    const int ng = N / group;
    const int g = n0 / group;
    const long long words_per_row = (long long)N * BITS / 32;
    const uint32_t* wcol = w + (long long)n0 * BITS / 32;
    const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);

    float2 acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = make_float2(0.f, 0.f);
    float XS = 0.f;  // sum_k xs_k over this lane's rows
    float XB = 0.f;  // sum_k x_k b[k, g]

    for (int kb = k_begin + warp * 4 + t; kb < k_end; kb += kKnRowsPerStep * kU) {
        KnWords<BITS> cw[kU];
        float xv[kU], sv[kU], bv[kU];
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            const int k = kb + i * kKnRowsPerStep;
            if (col_ok && k < k_end) {
                cw[i] = kn_load<BITS>(wcol + (long long)k * words_per_row);
                xv[i] = bf16_bits_to_float(__ldg(xb + k));
                sv[i] = bf16_bits_to_float(__ldg(scales + (long long)k * ng + g));
                bv[i] = bf16_bits_to_float(__ldg(biases + (long long)k * ng + g));
            } else {
#pragma unroll
                for (int j = 0; j < BITS; ++j) cw[i].w[j] = 0u;
                xv[i] = 0.f;
                sv[i] = 0.f;
                bv[i] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            // rows past the range have x = 0: they add exact zeros
            const float xs = xv[i] * sv[i];
            XS += xs;
            XB = fmaf(xv[i], bv[i], XB);
            kn_accumulate<BITS>(cw[i], xs, acc);
        }
    }

    // this lane's partial y over its rows, then the four row slots of the warp
    float yp[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        yp[2 * j] = fmaf(acc[j].x - XS, kUnscale, XB);
        yp[2 * j + 1] = fmaf(acc[j].y - XS, kUnscale, XB);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        yp[j] += __shfl_xor_sync(0xFFFFFFFFu, yp[j], 8);
        yp[j] += __shfl_xor_sync(0xFFFFFFFFu, yp[j], 16);
    }
    if (t == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) part[warp][c * 32 + j] = yp[j];
    }
    __syncthreads();
    {
        float s = 0.f;
#pragma unroll
        for (int wi = 0; wi < kKnWarps; ++wi) s += part[wi][threadIdx.x];
        cta_part[threadIdx.x] = s;
    }
    // every CTA's partial is written before rank 0 reads them; rank 0 adds
    // them in rank order
    kn_cluster_sync();
    if (rank == 0) {
        const int n = blockIdx.x * kKnCols + threadIdx.x;
        const uint32_t local = smem_u32(&cta_part[threadIdx.x]);
        float s = 0.f;
        const int S = (int)gridDim.y;
        for (int r = 0; r < S; ++r) s += kn_ld_cluster_f32(local, (uint32_t)r);
        if (n < N) y[n] = __float2bfloat16_rn(s);
    }
    // partials stay readable until rank 0 is done
    kn_cluster_sync();
}

}  // namespace

cudaError_t launch_qmv_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                          void* y, int K, int N, int bits, int group, int sms,
                          cudaStream_t stream) {
    const int col_blocks = (N + kKnCols - 1) / kKnCols;
    // enough CTAs for two per SM, at most 8 per cluster, and at least one
    // step of rows each
    int S = (2 * sms + col_blocks - 1) / col_blocks;
    if (S > kKnMaxCluster) S = kKnMaxCluster;
    const int max_by_k = (K + kKnRowsPerStep - 1) / kKnRowsPerStep;
    if (S > max_by_k) S = max_by_k;
    if (S < 1) S = 1;
    const int rows_per_rank = (K + S - 1) / S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(col_blocks, S, 1);
    cfg.blockDim = dim3(kKnThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* sb = static_cast<const uint16_t*>(scales);
    const auto* bb = static_cast<const uint16_t*>(biases);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    cudaError_t err;
    if (bits == 2)
        err = cudaLaunchKernelEx(&cfg, qmv_kn_kernel<2>, xb, w, sb, bb, yb, K, N, group, rows_per_rank);
    else if (bits == 4)
        err = cudaLaunchKernelEx(&cfg, qmv_kn_kernel<4>, xb, w, sb, bb, yb, K, N, group, rows_per_rank);
    else if (bits == 8)
        err = cudaLaunchKernelEx(&cfg, qmv_kn_kernel<8>, xb, w, sb, bb, yb, K, N, group, rows_per_rank);
    else
        return cudaErrorInvalidValue;
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mxq
