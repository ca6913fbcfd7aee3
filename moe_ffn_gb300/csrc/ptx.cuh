// ptx.cuh — inline-PTX wrappers for sm_103a: mbarriers, 1-D bulk TMA copies,
// programmatic dependent launch, bounded waits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace qmoe {

// Device error codes: the first one recorded wins; read and cleared by
// qmoe_device_status().
enum : unsigned {
    DEV_OK = 0,
    DEV_TIMEOUT_FULL = 1,
    DEV_TIMEOUT_EMPTY = 2,
    DEV_ROUTE_RANGE = 5,  // an expert index was clamped (internal invariant)
    DEV_X_RANGE = 6       // an activation of magnitude >= 2^106
};

// The device control block, one per device (a global of the library): the
// error word, the limit of every bounded wait, and a fault-injection setting
// for tests (a CTA that never arrives at the grid barriers, so that the
// other CTAs' bounded waits run out).  The host sets the last two only
// through qmoe_set_fault_injection; by default waits give up after 2 s.
struct DevCtl {
    unsigned code;                // 0, or the first error code recorded
    int skip_arrive_cta;          // -1: none
    unsigned long long wait_ns;   // limit of a bounded wait, nanoseconds
};
constexpr unsigned long long DEFAULT_WAIT_NS = 2000000000ull;

__device__ __forceinline__ void record_error(DevCtl* c, unsigned code) {
    atomicCAS(&c->code, 0u, code);
}
__device__ __forceinline__ unsigned long long wait_limit(const DevCtl* c) {
    return __ldcg(&c->wait_ns);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on a barrier phase.  Returns false (and records `code` in the
// device error word) if the phase has not completed within the wait limit
// (2 s unless a test shortened it).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, DevCtl* err,
                                                  unsigned code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    const unsigned long long lim = wait_limit(err);
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_ns() - t0 > lim) {
            record_error(err, code);
            return false;
        }
    }
}

// L2 policy for streamed weights: evict first, so activations and
// re-read operands keep their L2 lines.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for operands several CTAs re-read (evict last).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  Every kernel triggers its dependents right
// after its own wait: the next launch on the stream is then scheduled while
// this one runs, and its CTAs start (and stream their weights) as soon as
// they fit; its own griddepcontrol.wait holds back every read of this
// launch's outputs until this grid has completed and its writes are
// visible.  Triggering at the very start was measured slower on the GEMV
// sweep: the next launch's copies then compete with this launch's own.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over the first `nthreads` threads (consumer warps).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 2-D tiled TMA load of the box at (x, y) of the tensor map `tmap` (the
// address of a __grid_constant__ kernel parameter) into shared memory,
// completing `bar`'s transaction bytes.  x times the element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Named barrier that also ANDs a flag over its participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Arrive on a named barrier without waiting for it to complete.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace qmoe
