// Sorted mixture-of-experts: the per-call tile table for the grouped GEMM.
//
// mlxcel PR #1562 (Summary) describes the prior art: prepare_grouped_mm_data
// builds a per-expert problem table on the GPU before every grouped GEMM
// over rows sorted by expert.  Here one CTA:
//   1. validates the ids (range, order) and the source rows;
//   2. finds each expert's segment [start, end) of the sorted rows by binary
//      search;
//   3. cuts each segment into tiles of at most rows_per_tile rows of equal
//      size, and writes the tile list with a block-wide exclusive scan;
//   4. zeroes the y rows no tile covers (ids outside [0, E)).
// Unsorted ids make the call produce an all-zero y and no tiles.
//
// When the activation rows are routed through row_src, a second kernel
// copies them into sorted order (x_sorted[r] = x[row_src[r]], zero for an
// invalid source) so that the GEMM reads every activation tile with TMA.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kPrepThreads = 1024;

__device__ int lower_bound_ids(const int32_t* ids, int B, int v) {
    int lo = 0, hi = B;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ids[mid] < v) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ void zero_rows(__nv_bfloat16* y, long long r0, long long r1, int N) {
    const long long total = (r1 - r0) * (long long)N;
    __nv_bfloat16* base = y + r0 * N;
    for (long long i = threadIdx.x; i < total; i += blockDim.x) base[i] = __float2bfloat16_rn(0.f);
}

__global__ void __launch_bounds__(kPrepThreads) gather_prepass_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ row_src, int T, int B, int E,
    int N, int rows_per_tile, MTile* __restrict__ tiles, int* __restrict__ tile_count,
    __nv_bfloat16* __restrict__ y, int32_t* __restrict__ status) {
    __shared__ int flags;
    __shared__ int scan[kPrepThreads];
    __shared__ int seg_first, seg_last;
    if (threadIdx.x == 0) flags = 0;
    __syncthreads();

    int f = 0;
    for (int r = threadIdx.x; r < B; r += blockDim.x) {
        const int e = ids[r];
        if (e < 0 || e >= E) f |= MXQ_DEV_BAD_EXPERT_ID;
        if (r > 0 && ids[r - 1] > e) f |= MXQ_DEV_UNSORTED_IDS;
        if (row_src) {
            const int s = row_src[r];
            if (s < 0 || s >= T) f |= MXQ_DEV_BAD_ROW_SRC;
        }
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    const int all = flags;
    if (threadIdx.x == 0 && status) *status = all;

    if (all & MXQ_DEV_UNSORTED_IDS) {
        if (threadIdx.x == 0) *tile_count = 0;
        zero_rows(y, 0, B, N);
        return;
    }

    // experts owned by this thread: a contiguous range, so the scan keeps
    // the tile list in expert order
    const int per = (E + kPrepThreads - 1) / kPrepThreads;
    const int e0 = min(E, (int)threadIdx.x * per);
    const int e1 = min(E, e0 + per);
    int my_tiles = 0;
    for (int e = e0; e < e1; ++e) {
        const int len = lower_bound_ids(ids, B, e + 1) - lower_bound_ids(ids, B, e);
        my_tiles += (len + rows_per_tile - 1) / rows_per_tile;
    }
    scan[threadIdx.x] = my_tiles;
    __syncthreads();
    // inclusive Hillis-Steele scan
    for (int off = 1; off < kPrepThreads; off <<= 1) {
        const int v = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
        __syncthreads();
        scan[threadIdx.x] += v;
        __syncthreads();
    }
    int out = scan[threadIdx.x] - my_tiles;
    for (int e = e0; e < e1; ++e) {
        const int start = lower_bound_ids(ids, B, e);
        const int len = lower_bound_ids(ids, B, e + 1) - start;
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
    if (threadIdx.x == kPrepThreads - 1) *tile_count = scan[kPrepThreads - 1];
    if (threadIdx.x == 0) {
        seg_first = lower_bound_ids(ids, B, 0);
        seg_last = lower_bound_ids(ids, B, E);
    }
    __syncthreads();
    // rows before expert 0 (negative ids) and after expert E-1 (ids >= E)
    zero_rows(y, 0, seg_first, N);
    zero_rows(y, seg_last, B, N);
}

// One warp per sorted row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ row_src,
                                                          int T, int B, int K,
                                                          uint4* __restrict__ x_sorted) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= B) return;
    const int chunks = K / 8;  // 16-byte chunks per row (K % 64 == 0)
    const int src = row_src[r];
    uint4* dst = x_sorted + (long long)r * chunks;
    if (src < 0 || src >= T) {
        for (int c = threadIdx.x & 31; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* s = x + (long long)src * chunks;
    for (int c = threadIdx.x & 31; c < chunks; c += 32) dst[c] = __ldg(s + c);
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* row_src, int T, int B, int K,
                               void* x_sorted, cudaStream_t stream) {
    gather_rows_kernel<<<(B + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(x), row_src, T,
                                                        B, K, static_cast<uint4*>(x_sorted));
    return cudaGetLastError();
}

cudaError_t launch_gather_prepass(const int32_t* expert_ids, const int32_t* row_src, int T,
                                  int B, int E, int N, int rows_per_tile, MTile* tiles,
                                  int* tile_count, void* y, int32_t* status,
                                  cudaStream_t stream) {
    gather_prepass_kernel<<<1, kPrepThreads, 0, stream>>>(
        expert_ids, row_src, T, B, E, N, rows_per_tile, tiles, tile_count,
        static_cast<__nv_bfloat16*>(y), status);
    return cudaGetLastError();
}

}  // namespace mxq
