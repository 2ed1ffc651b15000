// C ABI of the library: argument checks, tile and split planning, launches.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace {

constexpr int kTileN = 128;           // rows of w per CTA in the tensor-core kernel
constexpr int kMaxRowsPerTile = 256;  // MMA N limit
constexpr int kGatherRowsPerTile = 64;  // expert segments average ~36 rows
constexpr int kMinKBlocksPerSplit = 8;
// Grouped calls with at most one row per SM, and at most kGatherStreamWaves
// rows x weight sets per SM (a decode step: a few tokens x top_k), stream
// each row's expert matrix through the streaming GEMV; where the shape does
// not fit that kernel, calls with at most kGatherDecodeRows rows run one
// direct-load GEMV per row.  Larger calls run the tensor-core GEMM, which
// reads each expert once for all of its rows.
constexpr int kGatherDecodeRows = 32;
constexpr int kGatherStreamWaves = 2;
// Dense calls with at most this many activation rows run one streaming GEMV
// per row (measured: faster than the tensor-core GEMM at 2 rows, even at 4).
constexpr int kStreamRowsMax = 3;
constexpr int kMaxSplits = 8;             // portable cluster size
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int checked;  // 0 = not yet, 1 = ok, -1 = wrong arch
    int sms;
};
DeviceInfo g_dev[kMaxDevices];

mxq_status check_device(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MXQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MXQ_ERR_UNSUPPORTED;
    DeviceInfo& d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MXQ_ERR_CUDA;
        d.sms = count;
        d.checked = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (d.checked < 0) return MXQ_ERR_ARCH;
    if (sms) *sms = d.sms;
    return MXQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

mxq_status check_common(int K, int N, int bits, int group_size) {
    if (bits != 2 && bits != 3 && bits != 4 && bits != 6 && bits != 8) return MXQ_ERR_INVALID_ARG;
    if (group_size != 32 && group_size != 64 && group_size != 128) return MXQ_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || K % 64 != 0 || K % group_size != 0) return MXQ_ERR_INVALID_ARG;
    // rows of codes are whole 16-byte units (the tensor-core kernels copy
    // them with TMA): a multiple of 128 codes at 3 bits
    if (bits == 3 && K % 128 != 0) return MXQ_ERR_INVALID_ARG;
    return MXQ_OK;
}

// Dense GEMM plan: M tiles of equal size (multiple of 16, at most 256) and,
// when M and N give fewer tiles than SMs, a split of K over the CTAs of a
// cluster (at most 8, each with at least kMinKBlocksPerSplit 64-wide blocks).
struct DensePlan {
    int m_tiles, m_tile, tmem_cols, splits, kb_per_split;
};

DensePlan plan_dense(int M, int K, int N, int bits, int sms) {
    DensePlan pl;
    const int want_tiles = (M + kMaxRowsPerTile - 1) / kMaxRowsPerTile;
    const int per = (M + want_tiles - 1) / want_tiles;
    pl.m_tile = (per + 15) & ~15;                      // <= 256
    pl.m_tiles = (M + pl.m_tile - 1) / pl.m_tile;      // every tile has >= 1 row
    int cols = 32;
    while (cols < pl.m_tile) cols <<= 1;
    pl.tmem_cols = cols;
    const int n_tiles = (N + kTileN - 1) / kTileN;
    const int tiles = n_tiles * pl.m_tiles;
    const int KB = K / 64;
    const int slots = sms;
    int splits = 1;
    if (tiles < slots) {
        splits = slots / tiles;
        const int max_by_k = KB / kMinKBlocksPerSplit;
        if (splits > max_by_k) splits = max_by_k;
        if (splits > kMaxSplits) splits = kMaxSplits;
        if (splits < 1) splits = 1;
    }
    pl.kb_per_split = (KB + splits - 1) / splits;
    // a split starts on a 16-byte boundary of the code rows: 3-bit blocks
    // of 64 codes are 24 bytes, so splits of 3-bit codes hold an even number
    if (bits == 3 && (pl.kb_per_split & 1)) ++pl.kb_per_split;
    pl.splits = (KB + pl.kb_per_split - 1) / pl.kb_per_split;  // every split gets >= 1 block
    return pl;
}

// Tiles of the grouped tensor-core GEMM (at most 64 rows each), an upper bound.
size_t gather_max_tiles(int B, int E) { return (size_t)B / kGatherRowsPerTile + (size_t)E + 1; }

// Tile records, the tile count, each expert's first row; 256-byte aligned.
size_t gather_table_bytes(int B, int E) {
    return align_up(gather_max_tiles(B, E) * sizeof(mxq::MTile), 256) + 256 +
           align_up(((size_t)E + 1) * sizeof(int), 256);
}

// Pipeline-wait budget for kernels launched from now on; 0 until the first
// launch reads MXQ_DEBUG_WAIT_BUDGET.
std::atomic<long long> g_wait_budget{0};

long long clamp_budget(long long cycles) {
    return (cycles <= 0 || cycles > mxq::kWaitBudgetCycles) ? mxq::kWaitBudgetCycles : cycles;
}

}  // namespace

mxq_status mxq::check_current_device(int* sms) { return check_device(sms); }

long long mxq::wait_budget_cycles() {
    long long b = g_wait_budget.load(std::memory_order_relaxed);
    if (b == 0) {
        const char* env = std::getenv("MXQ_DEBUG_WAIT_BUDGET");
        long long expected = 0;
        g_wait_budget.compare_exchange_strong(expected,
                                              clamp_budget(env ? std::strtoll(env, nullptr, 10) : 0));
        b = g_wait_budget.load(std::memory_order_relaxed);
    }
    return b;
}

size_t mxq::gather_scratch_bytes(int B, int E, int K, int N, int bits, int group_size,
                                 bool has_row_src) {
    (void)N;
    (void)bits;
    (void)group_size;
    if (has_row_src) return gather_table_bytes(B, E) + align_up((size_t)B * K * 2, 256);
    return gather_table_bytes(B, E);
}

extern "C" {

const char* mxq_status_string(mxq_status s) {
    switch (s) {
        case MXQ_OK: return "ok";
        case MXQ_ERR_INVALID_ARG: return "invalid argument";
        case MXQ_ERR_MISALIGNED: return "misaligned pointer";
        case MXQ_ERR_UNSUPPORTED: return "unsupported";
        case MXQ_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
        case MXQ_ERR_CUDA: return "CUDA error";
        case MXQ_ERR_WORKSPACE: return "workspace missing or too small";
        case MXQ_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation entry point";
    }
    return "unknown status";
}

int mxq_version(void) { return 100; }

long long mxq_debug_set_wait_budget(long long cycles) {
    g_wait_budget.store(clamp_budget(cycles), std::memory_order_relaxed);
    return g_wait_budget.load(std::memory_order_relaxed);
}

mxq_status mxq_qmv(const void* x, const uint32_t* w, const void* scales, const void* biases,
                   void* y, int K, int N, int bits, int group_size, int32_t* dev_status,
                   void* stream) {
    mxq_status st = check_common(K, N, bits, group_size);
    if (st != MXQ_OK) return st;
    if (!x || !w || !scales || !biases || !y) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(dev_status, 4))
        return MXQ_ERR_MISALIGNED;
    int sms = 0;
    st = check_device(&sms);
    if (st != MXQ_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MXQ_ERR_CUDA;
    cudaError_t err =
        mxq::launch_qmv(x, w, scales, biases, y, K, N, bits, group_size, sms, dev_status, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

mxq_status mxq_qmm(const void* x, const uint32_t* w, const void* scales, const void* biases,
                   void* y, int M, int K, int N, int bits, int group_size, int32_t* dev_status,
                   void* stream) {
    mxq_status st = check_common(K, N, bits, group_size);
    if (st != MXQ_OK) return st;
    if (M <= 0) return MXQ_ERR_INVALID_ARG;
    if (!x || !w || !scales || !biases || !y) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(dev_status, 4))
        return MXQ_ERR_MISALIGNED;
    int sms = 0;
    st = check_device(&sms);
    if (st != MXQ_OK) return st;
    if (M == 1) {
        // one activation row: the streaming GEMV (same operation)
        cudaStream_t s1 = static_cast<cudaStream_t>(stream);
        if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s1) != cudaSuccess)
            return MXQ_ERR_CUDA;
        cudaError_t err =
            mxq::launch_qmv(x, w, scales, biases, y, K, N, bits, group_size, sms, dev_status, s1);
        return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
    }
    if (M <= kStreamRowsMax) {
        // two or three rows: one streaming GEMV per row (the matrix stays in
        // L2 between them) takes less time than a tensor-core tile's fill
        cudaStream_t s1 = static_cast<cudaStream_t>(stream);
        if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s1) != cudaSuccess)
            return MXQ_ERR_CUDA;
        cudaError_t err = mxq::launch_qmv_rows(x, w, scales, biases, y, M, K, N, bits, group_size,
                                               sms, dev_status, s1);
        if (err != cudaErrorNotSupported) return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
    }
    // enough tiles of at most 256 rows to fill every SM: the persistent
    // kernel (no K split; the next tile's loads overlap this tile's MMAs and
    // epilogue); otherwise the K split over thread-block clusters
    const int n_tiles = (N + 127) / 128;
    const int pm_tiles = (M + 255) / 256;
    const int pm_tile = (((M + pm_tiles - 1) / pm_tiles) + 15) & ~15;
    const bool persistent = (long long)n_tiles * pm_tiles >= sms;
    const DensePlan pl = plan_dense(M, K, N, bits, sms);
    if (pl.m_tiles > 65535) return MXQ_ERR_UNSUPPORTED;  // grid.y limit
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MXQ_ERR_CUDA;
    mxq::QmmParams p;
    std::memset(&p, 0, sizeof p);
    p.x = x;
    p.w = w;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.y = y;
    p.status = dev_status;
    p.M = M;
    p.T = M;
    p.E = 1;
    p.K = K;
    p.N = N;
    p.group = group_size;
    p.sets = 1;
    p.x_rows = M;
    p.x_box_rows = pl.m_tile;
    p.m_tile = pl.m_tile;
    p.tmem_cols = pl.tmem_cols;
    p.splits = pl.splits;
    p.kb_per_split = pl.kb_per_split;
    if (persistent) {
        p.persistent = 1;
        p.m_tile = pm_tile;
        p.x_box_rows = pm_tile;
        p.m_tiles = pm_tiles;
        p.splits = 1;
        p.kb_per_split = K / 64;
        const long long tiles = (long long)n_tiles * pm_tiles;
        p.grid_ctas = (int)(tiles < sms ? tiles : sms);
        cudaError_t err = mxq::launch_qmm_tc(p, bits, pm_tiles, pm_tile, s);
        return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
    }
    cudaError_t err = mxq::launch_qmm_tc(p, bits, pl.m_tiles, pl.m_tile, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

mxq_status mxq_qmv_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                      void* y, int K, int N, int bits, int group_size, int32_t* dev_status,
                      void* stream) {
    if (bits == 3 || bits == 6) return MXQ_ERR_UNSUPPORTED;
    if (bits != 2 && bits != 4 && bits != 8) return MXQ_ERR_INVALID_ARG;
    if (group_size != 32 && group_size != 64 && group_size != 128) return MXQ_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || N % 64 != 0 || N % group_size != 0) return MXQ_ERR_INVALID_ARG;
    if (!x || !w || !scales || !biases || !y) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(dev_status, 4))
        return MXQ_ERR_MISALIGNED;
    int sms = 0;
    mxq_status st = check_device(&sms);
    if (st != MXQ_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MXQ_ERR_CUDA;
    cudaError_t err = mxq::launch_qmv_kn(x, w, scales, biases, y, K, N, bits, group_size, sms, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

mxq_status mxq_qmm_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                      void* y, int M, int K, int N, int bits, int group_size, int32_t* dev_status,
                      void* stream) {
    if (bits == 3 || bits == 6) return MXQ_ERR_UNSUPPORTED;
    if (bits != 2 && bits != 4 && bits != 8) return MXQ_ERR_INVALID_ARG;
    if (group_size != 32 && group_size != 64 && group_size != 128) return MXQ_ERR_INVALID_ARG;
    if (M <= 0 || K <= 0 || N <= 0 || N % 64 != 0 || N % group_size != 0) return MXQ_ERR_INVALID_ARG;
    if (M > 1 && K % 8 != 0) return MXQ_ERR_INVALID_ARG;  // 16-byte activation rows for TMA
    if (!x || !w || !scales || !biases || !y) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(dev_status, 4))
        return MXQ_ERR_MISALIGNED;
    if (M == 1)  // one activation row: the [K, N] GEMV (same operation)
        return mxq_qmv_kn(x, w, scales, biases, y, K, N, bits, group_size, dev_status, stream);
    int sms = 0;
    mxq_status st = check_device(&sms);
    if (st != MXQ_OK) return st;
    const int K64 = (K + 63) / 64 * 64;
    const DensePlan pl = plan_dense(M, K64, N, bits, sms);
    if (pl.m_tiles > 65535) return MXQ_ERR_UNSUPPORTED;  // grid.y limit
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MXQ_ERR_CUDA;
    mxq::QmmParams p;
    std::memset(&p, 0, sizeof p);
    p.x = x;
    p.w = w;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.y = y;
    p.status = dev_status;
    p.M = M;
    p.T = M;
    p.E = 1;
    p.K = K;
    p.N = N;
    p.group = group_size;
    p.sets = 1;
    p.x_rows = M;
    p.x_box_rows = pl.m_tile;
    p.m_tile = pl.m_tile;
    p.tmem_cols = pl.tmem_cols;
    p.splits = pl.splits;
    p.kb_per_split = pl.kb_per_split;
    cudaError_t err = mxq::launch_qmm_kn(p, bits, pl.m_tiles, pl.m_tile, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

mxq_status mxq_quantize(const float* w, uint32_t* codes, void* scales, void* biases, int N,
                        int K, int bits, int group_size, void* stream) {
    mxq_status st = check_common(K, N, bits, group_size);
    if (st != MXQ_OK) return st;
    if (!w || !codes || !scales || !biases) return MXQ_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 2) || !aligned(biases, 2))
        return MXQ_ERR_MISALIGNED;
    st = check_device(nullptr);
    if (st != MXQ_OK) return st;
    cudaError_t err = mxq::launch_quantize(w, codes, scales, biases, N, K, bits, group_size,
                                           static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

size_t mxq_gather_workspace_bytes(int B, int E, int K, int N) {
    (void)N;
    if (B <= 0 || E <= 0 || K < 0) return 0;
    // tile table + count, then room for the activation rows in sorted order
    return gather_table_bytes(B, E) + align_up((size_t)B * K * 2, 256);
}

}  // extern "C"

namespace {

// The grouped call for one weight set, or for the gate/up pair (w1 != null:
// a second set of the same shape, written to y1).
mxq_status gather_call(const void* x, const uint32_t* w, const void* scales, const void* biases,
                       const uint32_t* w1, const void* scales1, const void* biases1,
                       const int32_t* expert_ids, const int32_t* row_src, void* y, void* y1, int T,
                       int B, int E, int K, int N, int bits, int group_size, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
    mxq_status st = check_common(K, N, bits, group_size);
    if (st != MXQ_OK) return st;
    if (T <= 0 || B <= 0 || E <= 0) return MXQ_ERR_INVALID_ARG;
    if (!row_src && T != B) return MXQ_ERR_INVALID_ARG;
    if (!x || !w || !scales || !biases || !expert_ids || !y) return MXQ_ERR_INVALID_ARG;
    const bool pair = w1 != nullptr;
    if (pair && (!scales1 || !biases1 || !y1)) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(expert_ids, 4) || !aligned(row_src, 4) ||
        !aligned(dev_status, 4) || !aligned(workspace, 256))
        return MXQ_ERR_MISALIGNED;
    if (pair && (!aligned(w1, 16) || !aligned(y1, 16) || !aligned(scales1, 2) ||
                 !aligned(biases1, 2)))
        return MXQ_ERR_MISALIGNED;
    const size_t need = mxq::gather_scratch_bytes(B, E, K, N, bits, group_size, row_src != nullptr);
    if (!workspace || workspace_bytes < need) return MXQ_ERR_WORKSPACE;
    if (gather_max_tiles(B, E) > 65535) return MXQ_ERR_UNSUPPORTED;  // grid.y limit
    int sms = 0;
    st = check_device(&sms);
    if (st != MXQ_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sets = pair ? 2 : 1;
    const bool stream_rows = B <= sms && (long long)B * sets <= (long long)kGatherStreamWaves * sms;
    if (stream_rows || B <= kGatherDecodeRows) {
        // a decode step: one GEMV per sorted row (and weight set) against its
        // expert's matrix, no tile table
        if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess)
            return MXQ_ERR_CUDA;
        cudaError_t err = cudaErrorNotSupported;
        if (stream_rows)
            err = mxq::launch_gather_qmv(x, w, scales, biases, w1, scales1, biases1, expert_ids,
                                         row_src, y, y1, sets, T, B, E, K, N, bits, group_size,
                                         sms, true, dev_status, s);
        if (err == cudaErrorNotSupported && B <= kGatherDecodeRows)
            err = mxq::launch_gather_qmv(x, w, scales, biases, w1, scales1, biases1, expert_ids,
                                         row_src, y, y1, sets, T, B, E, K, N, bits, group_size,
                                         sms, false, dev_status, s);
        if (err != cudaErrorNotSupported) return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
        // neither GEMV form fits: the tensor-core GEMM below
    }
    auto* tiles = static_cast<mxq::MTile*>(workspace);
    int* tile_count = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                             align_up(gather_max_tiles(B, E) * sizeof(mxq::MTile), 256));
    int* seg_start = tile_count + 256 / sizeof(int);
    char* rows_area = static_cast<char*>(workspace) + gather_table_bytes(B, E);
    const size_t max_tiles = gather_max_tiles(B, E);
    cudaError_t err = mxq::launch_gather_prepass(expert_ids, row_src, T, B, E, N,
                                                 kGatherRowsPerTile, tiles, tile_count, seg_start,
                                                 y, pair ? y1 : nullptr, dev_status, s);
    if (err != cudaSuccess) return MXQ_ERR_CUDA;
    const void* xa = x;
    if (row_src) {
        void* x_sorted = rows_area;
        err = mxq::launch_gather_rows(x, row_src, T, B, K, x_sorted, s);
        if (err != cudaSuccess) return MXQ_ERR_CUDA;
        xa = x_sorted;
    }
    mxq::QmmParams p;
    std::memset(&p, 0, sizeof p);
    p.x = xa;
    p.w = w;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.y = y;
    p.tiles = tiles;
    p.tile_count = tile_count;
    p.status = dev_status;
    p.x_rows = B;
    // one TMA box of a slot's 64 rows per 64-wide block (rows past the tile
    // are loaded and never used): fewer copies than 16-row boxes
    p.x_box_rows = kGatherRowsPerTile;
    p.M = B;
    p.T = T;
    p.E = E;
    p.K = K;
    p.N = N;
    p.group = group_size;
    p.m_tile = kGatherRowsPerTile;
    p.tmem_cols = kGatherRowsPerTile;
    p.splits = 1;
    p.kb_per_split = K / 64;
    p.w_expert_stride = (long long)N * K * bits / 32;
    p.sb_expert_stride = (long long)N * (K / group_size);
    // the gate/up pair: a second weight set and output, same tiles
    p.sets = sets;
    p.w1 = w1;
    p.scales1 = static_cast<const uint16_t*>(scales1);
    p.biases1 = static_cast<const uint16_t*>(biases1);
    p.y1 = y1;
    // 2- and 4-bit: two persistent CTAs per SM take tiles of (weight set) x
    // (tile list) x (n tiles) from a counter as they finish the previous one,
    // so the pipeline fills once per CTA and long and short tiles balance;
    // 3-, 6- and 8-bit (code slots too large for two CTAs per SM): one CTA
    // per tile and weight set
    if (bits == 2 || bits == 4) {
        const long long bound = (long long)max_tiles * ((N + 127) / 128) * sets;
        p.persistent = 1;
        p.grid_ctas = (int)(bound < 2LL * sms ? bound : 2LL * sms);
        p.tile_counter = tile_count + 1;  // tiles handed out as CTAs free up
    }
    err = mxq::launch_qmm_tc(p, bits, (int)max_tiles, kGatherRowsPerTile, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

}  // namespace

extern "C" {

mxq_status mxq_gather_qmm_kn(const void* x, const uint32_t* w, const void* scales,
                             const void* biases, const int32_t* expert_ids, const int32_t* row_src,
                             void* y, int T, int B, int E, int K, int N, int bits, int group_size,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             void* stream) {
    if (bits == 3 || bits == 6) return MXQ_ERR_UNSUPPORTED;
    if (bits != 2 && bits != 4 && bits != 8) return MXQ_ERR_INVALID_ARG;
    if (group_size != 32 && group_size != 64 && group_size != 128) return MXQ_ERR_INVALID_ARG;
    if (K <= 0 || K % 8 != 0 || N <= 0 || N % 64 != 0 || N % group_size != 0)
        return MXQ_ERR_INVALID_ARG;
    if (T <= 0 || B <= 0 || E <= 0) return MXQ_ERR_INVALID_ARG;
    if (!row_src && T != B) return MXQ_ERR_INVALID_ARG;
    if (!x || !w || !scales || !biases || !expert_ids || !y) return MXQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(biases, 2) || !aligned(expert_ids, 4) || !aligned(row_src, 4) ||
        !aligned(dev_status, 4) || !aligned(workspace, 256))
        return MXQ_ERR_MISALIGNED;
    const size_t need = mxq::gather_scratch_bytes(B, E, K, N, bits, group_size, row_src != nullptr);
    if (!workspace || workspace_bytes < need) return MXQ_ERR_WORKSPACE;
    if (gather_max_tiles(B, E) > 65535) return MXQ_ERR_UNSUPPORTED;  // grid.y limit
    mxq_status st = check_device(nullptr);
    if (st != MXQ_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto* tiles = static_cast<mxq::MTile*>(workspace);
    int* tile_count = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                             align_up(gather_max_tiles(B, E) * sizeof(mxq::MTile), 256));
    int* seg_start = tile_count + 256 / sizeof(int);
    char* rows_area = static_cast<char*>(workspace) + gather_table_bytes(B, E);
    const size_t max_tiles = gather_max_tiles(B, E);
    // the tile table (and zeroed rows for invalid ids), then the routed rows
    // in sorted order, then one CTA per (tile, 128 columns)
    cudaError_t err = mxq::launch_gather_prepass(expert_ids, row_src, T, B, E, N,
                                                 kGatherRowsPerTile, tiles, tile_count, seg_start,
                                                 y, nullptr, dev_status, s);
    if (err != cudaSuccess) return MXQ_ERR_CUDA;
    const void* xa = x;
    if (row_src) {
        err = mxq::launch_gather_rows(x, row_src, T, B, K, rows_area, s);
        if (err != cudaSuccess) return MXQ_ERR_CUDA;
        xa = rows_area;
    }
    mxq::QmmParams p;
    std::memset(&p, 0, sizeof p);
    p.x = xa;
    p.w = w;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.y = y;
    p.tiles = tiles;
    p.tile_count = tile_count;
    p.status = dev_status;
    p.x_rows = B;
    p.x_box_rows = 16;
    p.M = B;
    p.T = T;
    p.E = E;
    p.K = K;
    p.N = N;
    p.group = group_size;
    p.m_tile = kGatherRowsPerTile;
    p.tmem_cols = kGatherRowsPerTile;
    p.splits = 1;
    p.kb_per_split = (K + 63) / 64;
    p.sets = 1;
    p.w_expert_stride = (long long)K * N * bits / 32;
    p.sb_expert_stride = (long long)K * (N / group_size);
    err = mxq::launch_qmm_kn(p, bits, (int)max_tiles, kGatherRowsPerTile, s);
    return err == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

mxq_status mxq_gather_qmm(const void* x, const uint32_t* w, const void* scales,
                          const void* biases, const int32_t* expert_ids, const int32_t* row_src,
                          void* y, int T, int B, int E, int K, int N, int bits, int group_size,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          void* stream) {
    return gather_call(x, w, scales, biases, nullptr, nullptr, nullptr, expert_ids, row_src, y,
                       nullptr, T, B, E, K, N, bits, group_size, workspace, workspace_bytes,
                       dev_status, stream);
}

mxq_status mxq_gather_qmm_gateup(const void* x, const uint32_t* w_gate, const void* scales_gate,
                                 const void* biases_gate, const uint32_t* w_up,
                                 const void* scales_up, const void* biases_up,
                                 const int32_t* expert_ids, const int32_t* row_src, void* y_gate,
                                 void* y_up, int T, int B, int E, int K, int N, int bits,
                                 int group_size, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream) {
    if (!w_up) return MXQ_ERR_INVALID_ARG;
    return gather_call(x, w_gate, scales_gate, biases_gate, w_up, scales_up, biases_up,
                       expert_ids, row_src, y_gate, y_up, T, B, E, K, N, bits, group_size,
                       workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"
