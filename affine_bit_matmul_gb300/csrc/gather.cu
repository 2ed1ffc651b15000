// Sorted mixture-of-experts: the per-call tile table for the grouped GEMM.
//
// mlxcel PR #1562 (Summary) describes the prior art: prepare_grouped_mm_data
// builds a per-expert problem table on the GPU before every grouped GEMM
// over rows sorted by expert.  Here one CTA:
//   1. validates the ids (range, order) and the source rows;
//   2. finds each expert's segment [start, end) of the sorted rows in one
//      pass over the row boundaries (no search: row r starts every expert in
//      (ids[r-1], ids[r]]);
//   3. cuts each segment into tiles of at most rows_per_tile rows of equal
//      size, and writes the tile list with a block-wide exclusive scan
//      (warp shuffles);
//   4. zeroes the y rows no tile covers (ids outside [0, E)), in both
//      outputs of the gate/up pair.
// Unsorted ids make the call produce an all-zero y and no tiles.
//
// When the activation rows are routed through row_src, a second kernel
// copies them into sorted order (x_sorted[r] = x[row_src[r]], zero for an
// invalid source) so that the GEMM reads every activation tile with TMA.
#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kPrepThreads = 1024;

__device__ void zero_rows(__nv_bfloat16* y, long long r0, long long r1, int N) {
    const long long total = (r1 - r0) * (long long)N;
    __nv_bfloat16* base = y + r0 * N;
    for (long long i = threadIdx.x; i < total; i += blockDim.x) base[i] = __float2bfloat16_rn(0.f);
}

// Block-wide exclusive scan of one int per thread (warp shuffles, then the
// warp totals); returns this thread's exclusive prefix, *total the sum.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += t;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? warp_sums[lane] : 0;
        int winc = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, winc, off);
            if (lane >= off) winc += t;
        }
        if (lane < nw) warp_sums[lane] = winc - w;  // exclusive
        if (lane == nw - 1) warp_sums[32] = winc;
    }
    __syncthreads();
    *total = warp_sums[32];
    return warp_sums[warp] + inc - v;
}

__global__ void __launch_bounds__(kPrepThreads) gather_prepass_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ row_src, int T, int B, int E,
    int N, int rows_per_tile, MTile* __restrict__ tiles, int* __restrict__ tile_count,
    int* __restrict__ seg_start, __nv_bfloat16* __restrict__ y, __nv_bfloat16* __restrict__ y2,
    int32_t* __restrict__ status) {
    __shared__ int flags;
    __shared__ int warp_sums[33];
    // the sorted copy of the activation rows (the next launch) does not read
    // anything this kernel writes: let it start now and run alongside
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        flags = 0;
        tile_count[1] = 0;  // the grouped GEMM's next-unclaimed-tile counter
    }
    __syncthreads();

    // 1. validate (eight rows per thread per round, all loads issued first)
    constexpr int kPer = 8;
    const int step = kPer * (int)blockDim.x;
    int f = 0;
    for (int base = 0; base < B; base += step) {
        int v[kPer], pv[kPer], sv[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int r = base + i * (int)blockDim.x + (int)threadIdx.x;
            v[i] = r < B ? ids[r] : 0;
            pv[i] = (r > 0 && r < B) ? ids[r - 1] : INT_MIN;
            sv[i] = (row_src && r < B) ? row_src[r] : 0;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int r = base + i * (int)blockDim.x + (int)threadIdx.x;
            if (r >= B) continue;
            if (v[i] < 0 || v[i] >= E) f |= MXQ_DEV_BAD_EXPERT_ID;
            if (pv[i] > v[i]) f |= MXQ_DEV_UNSORTED_IDS;
            if (row_src && (sv[i] < 0 || sv[i] >= T)) f |= MXQ_DEV_BAD_ROW_SRC;
        }
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    const int all = flags;
    if (threadIdx.x == 0 && status) *status = all;

    if (all & MXQ_DEV_UNSORTED_IDS) {
        if (threadIdx.x == 0) *tile_count = 0;
        zero_rows(y, 0, B, N);
        if (y2) zero_rows(y2, 0, B, N);
        return;
    }

    // 2. expert e's rows start at seg_start[e] = the first r with ids[r] >= e:
    // with the ids sorted, row r is that start for exactly the e in
    // (ids[r-1], ids[r]] (clamped to [0, E]), and r = B for the e above the
    // last id, so every entry of seg_start[0..E] is written once
    for (int base = 0; base <= B; base += step) {
        long long cur[kPer], prev[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int r = base + i * (int)blockDim.x + (int)threadIdx.x;
            cur[i] = r < B ? (long long)ids[r] : (long long)E;
            prev[i] = (r > 0 && r <= B) ? (long long)ids[r - 1] : -1;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int r = base + i * (int)blockDim.x + (int)threadIdx.x;
            if (r > B) continue;
            const long long e0 = prev[i] + 1 > 0 ? prev[i] + 1 : 0;
            const long long e1 = cur[i] < E ? cur[i] : E;
            for (long long e = e0; e <= e1; ++e) seg_start[e] = r;
        }
    }
    __syncthreads();

    // 3. tiles: each expert's segment cut into tiles of at most rows_per_tile
    // rows of equal size; a thread owns a contiguous range of experts, so the
    // scan keeps the tile list in expert order
    const int per = (E + kPrepThreads - 1) / kPrepThreads;
    const int e0 = min(E, (int)threadIdx.x * per);
    const int e1 = min(E, e0 + per);
    int my_tiles = 0;
    for (int e = e0; e < e1; ++e) {
        const int len = seg_start[e + 1] - seg_start[e];
        my_tiles += (len + rows_per_tile - 1) / rows_per_tile;
    }
    int total = 0;
    int out = block_exclusive_scan(my_tiles, warp_sums, &total);
    for (int e = e0; e < e1; ++e) {
        const int start = seg_start[e];
        const int len = seg_start[e + 1] - start;
        const int nt = (len + rows_per_tile - 1) / rows_per_tile;
        const int chunk = nt ? (len + nt - 1) / nt : 0;
        for (int j = 0; j < nt; ++j) {
            MTile t;
            t.e = e;
            t.row_start = start + j * chunk;
            t.rows = min(chunk, len - j * chunk);
            t.pad = 0;
            tiles[out++] = t;
        }
    }
    if (threadIdx.x == 0) *tile_count = total;
    // 4. rows before expert 0 (negative ids) and from expert E on (ids >= E)
    zero_rows(y, 0, seg_start[0], N);
    zero_rows(y, seg_start[E], B, N);
    if (y2) {
        zero_rows(y2, 0, seg_start[0], N);
        zero_rows(y2, seg_start[E], B, N);
    }
}

// One warp per sorted row, 16-byte copies.  It runs alongside the prepass
// (programmatic dependent launch) but does not finish before it: every
// thread ends in griddepcontrol.wait, so the launch after this one, which
// waits for this grid, also finds the tile list complete.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ row_src,
                                                          int T, int B, int K,
                                                          uint4* __restrict__ x_sorted) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r < B) {
        const int chunks = K / 8;  // 16-byte chunks per row (K % 8 == 0)
        const int src = row_src[r];
        uint4* dst = x_sorted + (long long)r * chunks;
        if (src < 0 || src >= T) {
            for (int c = threadIdx.x & 31; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        } else {
            const uint4* s = x + (long long)src * chunks;
            // four 16-byte loads in flight per lane before the stores
            int c = threadIdx.x & 31;
            for (; c + 96 < chunks; c += 128) {
                const uint4 a = __ldg(s + c), b = __ldg(s + c + 32), d = __ldg(s + c + 64),
                            e = __ldg(s + c + 96);
                dst[c] = a;
                dst[c + 32] = b;
                dst[c + 64] = d;
                dst[c + 96] = e;
            }
            for (; c < chunks; c += 32) dst[c] = __ldg(s + c);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* row_src, int T, int B, int K,
                               void* x_sorted, cudaStream_t stream) {
    // launched right after the prepass as a programmatic dependent launch:
    // it reads x and row_src and writes only x_sorted, none of which the
    // prepass touches, so it may overlap it; the GEMM after it is an
    // ordinary launch and waits for both
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((B + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gather_rows_kernel, static_cast<const uint4*>(x),
                                       row_src, T, B, K, static_cast<uint4*>(x_sorted));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gather_prepass(const int32_t* expert_ids, const int32_t* row_src, int T,
                                  int B, int E, int N, int rows_per_tile, MTile* tiles,
                                  int* tile_count, int* seg_start, void* y, void* y2,
                                  int32_t* status, cudaStream_t stream) {
    gather_prepass_kernel<<<1, kPrepThreads, 0, stream>>>(
        expert_ids, row_src, T, B, E, N, rows_per_tile, tiles, tile_count, seg_start,
        static_cast<__nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(y2), status);
    return cudaGetLastError();
}

}  // namespace mxq
