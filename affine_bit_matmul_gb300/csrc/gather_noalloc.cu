// mxq_gather_qmm_noalloc: the sorted mixture-of-experts GEMM for callers that
// cannot hand the library a device workspace.
//
// mxq_gather_qmm needs scratch memory every call (the per-call tile table and,
// when rows are routed through row_src, the activation rows in sorted order).
// Some callers have no way to provide it: plain C hosts without a device
// allocator of their own, runtimes whose device memory is fully carved up
// before the serving loop starts, and code that must not allocate between
// steps (allocation can synchronise the device or fail under memory
// pressure).  This entry point takes the scratch from one fixed array in the
// library's own device memory instead, reserved when the library is loaded on
// a device, so neither the caller nor the library allocates anything at call
// time.
//
// Its price is that the scratch is shared: two calls whose execution overlaps
// on one device (different streams, or different host threads without
// ordering between them) use the same memory and corrupt each other's
// results.  Calls must be ordered, for example by issuing them all on one
// stream.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace {

// The fixed scratch.  Nothing in it needs to start at zero: each call writes
// every byte it later reads (the tile table and count in the first kernel,
// the sorted activation rows in the second).
__device__ __align__(256) unsigned char g_gather_scratch[MXQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the lookup may load the library's device code on that device).
mxq_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MXQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MXQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gather_scratch) != cudaSuccess || !p) return MXQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MXQ_OK;
}

}  // namespace

extern "C" mxq_status mxq_gather_qmm_noalloc(const void* x, const uint32_t* w,
                                             const void* scales, const void* biases,
                                             const int32_t* expert_ids, const int32_t* row_src,
                                             void* y, int T, int B, int E, int K, int N, int bits,
                                             int group_size, int32_t* dev_status, void* stream) {
    // the size check comes first, so an oversized request is refused before
    // anything touches a device
    const size_t need = mxq::gather_scratch_bytes(B, E, K, N, bits, group_size, row_src != nullptr);
    if (need > (size_t)MXQ_NOALLOC_SCRATCH_BYTES) return MXQ_ERR_SCRATCH_LIMIT;
    // a device of another architecture is reported as such before the
    // scratch lookup (which would fail there with a plain CUDA error)
    mxq_status st = mxq::check_current_device(nullptr);
    if (st != MXQ_OK) return st;
    void* scratch = nullptr;
    st = scratch_on_current_device(&scratch);
    if (st != MXQ_OK) return st;
    return mxq_gather_qmm(x, w, scales, biases, expert_ids, row_src, y, T, B, E, K, N, bits,
                          group_size, scratch, (size_t)MXQ_NOALLOC_SCRATCH_BYTES, dev_status,
                          stream);
}
