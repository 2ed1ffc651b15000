// Device-side helpers for the sm_103a kernels: mbarriers with bounded waits,
// cp.async, tcgen05 (tensor memory, UMMA descriptors, MMA issue and loads).
// All inline PTX is written from the PTX ISA description of each instruction.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace mxq {

// ----------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// A pipeline wait gives up after a budget of SM clock cycles; the kernel
// then records MXQ_DEV_TIMEOUT and winds down.  The budget is a kernel
// argument: this default (about one second at 2 GHz), or a shorter one set
// with mxq_debug_set_wait_budget to exercise the give-up path.  A CTA's waits
// for the copies and MMAs it issued itself (before it exits or frees tensor
// memory) always take the default, so no asynchronous write outlives it.
constexpr long long kWaitBudgetCycles = 2000000000LL;

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// One poll under a budget: try_wait may hold the thread for a while in
// hardware, so a budget shorter than the default polls with test_wait and
// is kept to the cycle.
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity, long long budget) {
    return budget < kWaitBudgetCycles ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity);
}

// Waits for the phase with the given parity to complete.  Returns false if
// the budget ran out (the caller then stops its pipeline role).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          long long budget = kWaitBudgetCycles) {
    if (mbar_poll(bar, parity, budget)) return true;
    const long long t0 = clock64();
    while (!mbar_poll(bar, parity, budget)) {
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

// Waits (default budget) until the copies issued into the last n slots of a
// ring have landed: copy g of the ring (g < issued) completes phase g / slots
// of barrier full[g % slots].  A producer calls this before it leaves, also
// after giving up, so that no copy writes shared memory after the CTA exits.
__device__ __forceinline__ bool drain_ring(uint64_t* full, int slots, long long issued, int n) {
    bool all = true;
    for (long long g = issued - 1; g >= 0 && g >= issued - n; --g)
        all = mbar_wait(&full[g % slots], (uint32_t)((g / slots) & 1)) && all;
    return all;
}

// ----------------------------------------------------------------- cp.async

// 16-byte global->shared copy; src_bytes = 0 fills the destination with zeros
// without reading global memory.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor cores read operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzled canonical layout: 8-row x 128-byte atoms, atoms stacked
// 1024 bytes apart along M/N.  Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29, unused for swizzled K-major), stride byte
// offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0,
// swizzle mode "128B" = 2 (61-63).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;            // LBO (ignored): 16 bytes
    d |= (uint64_t)(1024u >> 4) << 32;  // SBO: 1024 bytes between 8-row atoms
    d |= (uint64_t)1u << 46;            // version
    d |= (uint64_t)2u << 61;            // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16: bf16 A and B, fp32 D, both operands
// K-major, tile M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(uint32_t M, uint32_t N) {
    return (1u << 4)               // D format: f32
           | (1u << 7)             // A format: bf16
           | (1u << 10)            // B format: bf16
           | ((N >> 3) << 17)      // N / 8
           | ((M >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same MMA with the A operand read from tensor memory (row i of A in lane i,
// K along the columns, two bf16 per 32-bit column).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: column col + j of this thread's
// lane <- register j.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on an mbarrier once every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: register j <- column col + j of
// this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- bf16

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) {
    return __uint_as_float(h16 << 16);
}

}  // namespace mxq
