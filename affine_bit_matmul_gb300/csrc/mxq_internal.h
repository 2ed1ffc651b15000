// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mxq.h"

namespace mxq {

// The current device is compute capability 10.3 (MXQ_OK, *sms = its SM
// count; sms may be null), else MXQ_ERR_ARCH, or MXQ_ERR_CUDA if the runtime
// cannot say.  Cached per device.
mxq_status check_current_device(int* sms);

// The pipeline-wait budget, in SM clock cycles, for kernels launched now:
// the default (about one second) unless mxq_debug_set_wait_budget, or the
// MXQ_DEBUG_WAIT_BUDGET environment variable read at the first call, set a
// shorter one.
long long wait_budget_cycles();

// Scratch bytes a grouped call with these arguments needs: the tile table,
// plus the routed rows in sorted order when row_src is given.
size_t gather_scratch_bytes(int B, int E, int K, int N, int bits, int group_size,
                            bool has_row_src);

// One tile of output rows of the grouped (sorted mixture-of-experts) GEMM:
// rows [row_start, row_start + rows) of the sorted order, all of expert e.
struct MTile {
    int e;
    int row_start;
    int rows;
    int pad;
};

// Arguments of the tcgen05 GEMM kernel (dense and grouped forms).
struct QmmParams {
    const void* x;           // bf16 [T or M, K]
    const uint32_t* w;       // uint32 [E, N, K*bits/32]
    const uint16_t* scales;  // bf16 [E, N, K/group]
    const uint16_t* biases;  // bf16 [E, N, K/group]
    void* y;                 // bf16 [rows, N]
    const MTile* tiles;      // grouped form: tile list, or null (dense form)
    const int* tile_count;   // grouped form: number of valid tiles
    int32_t* status;         // MXQ_DEV_* bits, or null
    int x_rows;              // rows of the activation matrix the TMA reads
    int x_box_rows;          // rows per activation TMA box (multiple of 8, <= 256)
    int M;                   // dense form: rows of x and y
    int T;                   // grouped form: rows of x
    int E;                   // grouped form: experts
    int K, N;
    int group;               // k values per scale/bias pair: 32, 64 or 128
    int m_tile;              // dense form: rows per M tile (multiple of 16)
    int tmem_cols;           // tensor-memory columns allocated per CTA
    int splits;              // K splits = cluster size along z (1 = none)
    int kb_per_split;        // 64-wide K blocks per split
    long long w_expert_stride;   // words between experts
    long long sb_expert_stride;  // scale/bias entries between experts
    int persistent;          // 1: one CTA per SM walks the tiles (no K split)
    int m_tiles;             // dense persistent form: M tiles
    int grid_ctas;           // persistent form: CTAs launched
    int* tile_counter;       // persistent form: next unclaimed tile (zeroed before the
                             // launch), or null for a fixed gridDim.x stride
    // grouped form, gate/up pair: a second weight set of the same shape and
    // its output (sets = 2); the tiles of both sets share the activation rows
    int sets;                // 1 or 2
    const uint32_t* w1;
    const uint16_t* scales1;
    const uint16_t* biases1;
    void* y1;
    long long wait_budget;   // pipeline-wait budget in SM cycles (set by launch_qmm_tc)
};

// cuTensorMapEncodeTiled, looked up once through the runtime (null if the
// driver does not provide it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Decode GEMV; group = k values per scale/bias pair (32, 64 or 128).
cudaError_t launch_qmv(const void* x, const uint32_t* w, const void* scales, const void* biases,
                       void* y, int K, int N, int bits, int group, int sms, int32_t* status,
                       cudaStream_t stream);

// A few activation rows (M >= 2): one streaming GEMV per row, each row in
// its own grid row (cudaErrorNotSupported when the shape does not fit the
// streaming kernel).
cudaError_t launch_qmv_rows(const void* x, const uint32_t* w, const void* scales,
                            const void* biases, void* y, int M, int K, int N, int bits, int group,
                            int sms, int32_t* status, cudaStream_t stream);

// Dense or grouped tcgen05 GEMM; grid.y = number of M tiles (dense) or an
// upper bound on the number of tiles (grouped).
cudaError_t launch_qmm_tc(const QmmParams& p, int bits, int grid_m, int max_rows_per_tile,
                          cudaStream_t stream);

// The same GEMM with w stored [K, N] (codes and groups along n; 2-, 4- and
// 8-bit): dense (M tiles, K split over a cluster) or grouped (tile list).
cudaError_t launch_qmm_kn(const QmmParams& p, int bits, int grid_m, int max_rows_per_tile,
                          cudaStream_t stream);

// Grouped form, step 1: validate ids, find each expert's rows, build the
// tile list (count in tile_count[0]), zero tile_count[1] (the GEMM's tile
// counter) and the y rows that no tile covers.
// Step 2 (when row_src is given): copy the activation rows into sorted order.
// seg_start: device scratch of E + 1 ints (each expert's first sorted row).
// y2: the second output of the gate/up pair, or null.
cudaError_t launch_gather_prepass(const int32_t* expert_ids, const int32_t* row_src, int T,
                                  int B, int E, int N, int rows_per_tile, MTile* tiles,
                                  int* tile_count, int* seg_start, void* y, void* y2,
                                  int32_t* status, cudaStream_t stream);

// Grouped form with few rows (decode): one GEMV per sorted row (and weight
// set: sets = 2 adds w1, scales1, biases1 -> y1) against its expert's
// matrix, validating the ids itself (no tile table, no row copy).
// stream_form: the streaming GEMV with one grid row per sorted row and set
// (cudaErrorNotSupported when the shape does not fit it); otherwise the
// direct-load GEMV, grid (N / 16, B, sets).
cudaError_t launch_gather_qmv(const void* x, const uint32_t* w, const void* scales,
                              const void* biases, const uint32_t* w1, const void* scales1,
                              const void* biases1, const int32_t* expert_ids,
                              const int32_t* row_src, void* y, void* y1, int sets, int T, int B,
                              int E, int K, int N, int bits, int group, int sms,
                              bool stream_form, int32_t* status, cudaStream_t stream);

// Affine group-wise encoder (groups of 32, 64 or 128): float [N, K] ->
// codes, bf16 scales and biases.
cudaError_t launch_quantize(const float* W, uint32_t* codes, void* scales, void* biases, int N,
                            int K, int bits, int group, cudaStream_t stream);

// Decode GEMV for w stored [K, N] (codes and groups along n), 2/4/8-bit.
cudaError_t launch_qmv_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                          void* y, int K, int N, int bits, int group, int sms,
                          cudaStream_t stream);

cudaError_t launch_gather_rows(const void* x, const int32_t* row_src, int T, int B, int K,
                               void* x_sorted, cudaStream_t stream);

}  // namespace mxq
