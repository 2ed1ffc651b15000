// Device helpers shared by the tensor-core GEMM kernels (codes stored
// [N, K] in qmm.cu, [K, N] in qmm_kn.cu): bf16 pair arithmetic, the code
// dequantisers, TMA tensor copies, cluster barriers and distributed shared
// memory, and whole-warp bounded waits.  Inline PTX written from the PTX ISA
// description of each instruction.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "mxq_device.cuh"

namespace mxq {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_bf16(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Sixteen 2-bit codes (one word, lowest k in the lowest two bits) -> eight
// bf16x2 words (k pairs 0-1, ..., 14-15) of s*q + b, one rounding each.
__device__ __forceinline__ void dequant_word2(uint32_t wd, uint32_t s2, uint32_t b2,
                                              uint32_t (&out)[8]) {
    // plane j holds codes j, 4 + j, 8 + j, 12 + j in its four bytes
    const uint32_t p0 = wd & 0x03030303u;
    const uint32_t p1 = (wd >> 2) & 0x03030303u;
    const uint32_t p2 = (wd >> 4) & 0x03030303u;
    const uint32_t p3 = (wd >> 6) & 0x03030303u;
    const uint32_t a01 = prmt(p0, p1, 0x5140u);    // q0 q1 q4 q5
    const uint32_t a23 = prmt(p2, p3, 0x5140u);    // q2 q3 q6 q7
    const uint32_t c01 = prmt(p0, p1, 0x7362u);    // q8 q9 q12 q13
    const uint32_t c23 = prmt(p2, p3, 0x7362u);    // q10 q11 q14 q15
    const uint32_t e[4] = {prmt(a01, a23, 0x5410u), prmt(a01, a23, 0x7632u),
                           prmt(c01, c23, 0x5410u), prmt(c01, c23, 0x7632u)};  // q0-3 ... q12-15
    // bf16 0x43qq = 128 + q exactly; subtracting 128 is exact
    const uint32_t k128 = 0x43004300u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = hfma2_bf16(hsub2_bf16(prmt(e[i], 0x43u, 0x4140u), k128), s2, b2);
        out[2 * i + 1] = hfma2_bf16(hsub2_bf16(prmt(e[i], 0x43u, 0x4342u), k128), s2, b2);
    }
}

// Eight 4-bit codes (one word, lowest k in the lowest nibble) -> four bf16x2
// words (k pairs 0-1, 2-3, 4-5, 6-7) of s*q + b, one rounding each.
__device__ __forceinline__ void dequant_word4(uint32_t wd, uint32_t s2, uint32_t b2,
                                              uint32_t (&out)[4]) {
    const uint32_t lo = wd & 0x0F0F0F0Fu;          // q0 q2 q4 q6
    const uint32_t hi = (wd >> 4) & 0x0F0F0F0Fu;   // q1 q3 q5 q7
    const uint32_t e0 = prmt(lo, hi, 0x5140u);     // q0 q1 q2 q3
    const uint32_t e1 = prmt(lo, hi, 0x7362u);     // q4 q5 q6 q7
    // bf16 0x43qq = 128 + q exactly (q < 128); subtracting 128 is exact
    const uint32_t k128 = 0x43004300u;
    out[0] = hfma2_bf16(hsub2_bf16(prmt(e0, 0x43u, 0x4140u), k128), s2, b2);
    out[1] = hfma2_bf16(hsub2_bf16(prmt(e0, 0x43u, 0x4342u), k128), s2, b2);
    out[2] = hfma2_bf16(hsub2_bf16(prmt(e1, 0x43u, 0x4140u), k128), s2, b2);
    out[3] = hfma2_bf16(hsub2_bf16(prmt(e1, 0x43u, 0x4342u), k128), s2, b2);
}

// Four 8-bit codes (lowest k in the lowest byte) -> two bf16x2 words.  The
// code is exact in fp32 (2^23 + q, minus 2^23), s*q + b is one fp32 FMA
// (s*q is exact), then rounded to bf16.
__device__ __forceinline__ void dequant_word8(uint32_t wd, float s, float b, uint32_t (&out)[2]) {
    const float m = 8388608.f;
    const float q0 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7440u)) - m;
    const float q1 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7441u)) - m;
    const float q2 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7442u)) - m;
    const float q3 = __uint_as_float(prmt(wd, 0x4B000000u, 0x7443u)) - m;
    out[0] = cvt_bf16x2(fmaf(s, q0, b), fmaf(s, q1, b));
    out[1] = cvt_bf16x2(fmaf(s, q2, b), fmaf(s, q3, b));
}


__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}


__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Bring a tensor map into the descriptor cache ahead of its first use.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// L2 cache policies for the copies below: lines a copy brings in are the
// first (evict_first) or the last (evict_last) candidates for eviction.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// Ask L2 to fetch one box of a tensor map (a hint: it reads nothing into the
// CTA and orders nothing).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// Programmatic dependent launch: a kernel launched with it may start while
// the previous kernel on the stream finishes; it must call pdl_wait() before
// it reads or writes anything the previous kernel may touch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// One lane of the (converged) warp returns true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
        "elect.sync r|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Tests up to three barrier phases with one round trip.
__device__ __forceinline__ bool mbar_try_wait3(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                               uint64_t* c, uint32_t pc) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p, q, r;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 q, [%3], %4;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 r, [%5], %6;\n\t"
        "and.pred p, p, q;\n\t"
        "and.pred p, p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(a)), "r"(pa), "r"(smem_u32(b)), "r"(pb), "r"(smem_u32(c)), "r"(pc)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait3(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                           uint64_t* c, uint32_t pc, long long budget) {
    if (budget < kWaitBudgetCycles)  // a short budget: exact, non-blocking polls
        return mbar_wait(a, pa, budget) && mbar_wait(b, pb, budget) && mbar_wait(c, pc, budget);
    if (mbar_try_wait3(a, pa, b, pb, c, pc)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait3(a, pa, b, pb, c, pc)) {
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

// Position in a ring of n slots: the slot of the current item and the parity
// of its round (round = item / n), advanced without divisions.
struct Ring {
    int n, slot;
    uint32_t parity;
    __device__ explicit Ring(int n_) : n(n_), slot(0), parity(0) {}
    __device__ void next() {
        if (++slot == n) {
            slot = 0;
            parity ^= 1u;
        }
    }
};

// Whole-warp waits: every lane polls with its own bounded budget, then the
// warp agrees on the outcome, so the warp stays converged for elect.sync even
// when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, long long budget) {
    const bool ok = mbar_wait(bar, parity, budget);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool warp_wait3(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                           uint64_t* c, uint32_t pc, long long budget) {
    const bool ok = mbar_wait3(a, pa, b, pb, c, pc, budget);
    return __all_sync(0xffffffffu, ok);
}


// try_wait that lets the thread sleep in hardware until the phase completes
// (or the hint, in ns, runs out), so waiting warps take no issue slots from
// the warps doing the work.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try_wait_s(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait that sleeps: the first poll does not suspend, then the
// budget is checked before every suspending poll, so a budget shorter than
// one poll gives up at the first wait that is not already satisfied.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, long long budget) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    do {
        if (clock64() - t0 > budget) return false;
    } while (!mbar_try_wait_s(bar, parity, kSuspendNs));
    return true;
}

__device__ __forceinline__ bool warp_wait_sleep(uint64_t* bar, uint32_t parity, long long budget) {
    const bool ok = mbar_wait_sleep(bar, parity, budget);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace mxq
