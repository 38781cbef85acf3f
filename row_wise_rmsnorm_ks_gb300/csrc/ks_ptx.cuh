// Inline-PTX helpers for the staged row kernel: mbarriers, bulk global->shared copies with an
// L2 evict-first policy, and a bounded wait. sm_90 and later (compiled here for sm_103a).
#pragma once

#include <stdint.h>

namespace ks {

// Device-side fault word: bit 0 is set by a wait that gave up. Each translation unit that
// includes this header has its own copy (no relocatable device code); the host reads and clears
// all of them through ks_device_faults().
static __device__ unsigned int g_fault_flags = 0;

constexpr unsigned int kFaultWaitTimeout = 1u;
// A wait gives up after this long (nanoseconds of %globaltimer); a healthy wait lasts about a
// microsecond.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Programmatic dependent launch. Every row kernel calls grid_dependency_wait() before its first
// global-memory access: when the kernel was launched with the programmatic-serialization
// attribute it waits there until the preceding kernel in the stream has completed and its writes
// are visible; otherwise it returns at once. allow_dependents_launch() lets a kernel queued
// after this one (and launched with the attribute) be scheduled early; that kernel still waits
// for this one to finish before touching memory.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after kWaitLimitNs. Returns false on
// time-out (the caller records the fault and leaves the row loop).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// A hint to the copy engine: bring `bytes` (a multiple of 16, the address 16-byte aligned) of
// global memory into L2, with no completion to wait for and no register or shared-memory cost.
// Later loads of those bytes hit L2 if the lines are still there, and go to DRAM otherwise.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The address of this CTA's shared variable `p` in the shared memory of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

// An 8-byte store into a cluster peer's shared memory (addresses from cluster_map) that completes
// as 8 transaction bytes on the peer's mbarrier `bar`: no fence, no cluster barrier; the peer sees
// the bytes once its wait on that barrier's phase returns.
__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
                 ::"r"(addr), "r"(a), "r"(b), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

}  // namespace ks
