// pipeline.cuh -- shared-memory staging primitives for sm_100-family GPUs:
// mbarriers with bounded waits, 1-D bulk (TMA) copies global -> shared, and
// the device error word that a timed-out wait raises.
#pragma once

#include <stdint.h>

namespace qg {

// A wait that is still pending after this many try_wait polls gives up
// (each poll may suspend the thread for a hardware-defined interval).
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr int kErrTimeout = -7;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Wait for the phase of the given parity to complete; false after `limit`
// polls (kSpinLimit unless a test asks for a short wait).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit = kSpinLimit) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// As mbar_wait, but also gives up early once *abort is set (checked every
// 256 tries), and sets *abort itself when it runs out of tries, so that one
// timed-out wait ends the other waits of the block quickly.  Polls without
// sleeping: for the waits on a pipeline's critical path.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                                   uint32_t limit = kSpinLimit) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    return false;
}

// As mbar_wait_or_abort, for long waits off the critical path (a warp that
// waits for a whole tile): between tries the thread sleeps kBackoffNs, so it
// takes almost no issue slots from the warps that work meanwhile.
constexpr uint32_t kBackoffNs = 256;
constexpr uint32_t kBackoffLimit = 1u << 24;   // ~4 s of 256 ns sleeps
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t it = 0; it < kBackoffLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 15u) == 15u && *abort) return false;
        __nanosleep(kBackoffNs);
    }
    *abort = 1u;
    return false;
}

// 1-D bulk copy of `bytes` (multiple of 16) from global `src` (16-byte
// aligned) to shared `dst` (16-byte aligned); completion is counted on `bar`.
// The data is marked first to leave L2: these are streamed weights, read
// once per call, and a decode step streams several times L2's capacity, so
// without the hint they evict the activations and outputs that the next
// kernels read (measured: the six-matrix decode step 4607 -> 4754 GB/s).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "{.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "pol;}" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream is still
// running; it must execute griddep_wait() before it reads anything that
// kernel wrote or writes anything that kernel reads (the wait returns once
// the previous grid has completed and its memory is visible).  Work that
// depends on neither (streaming the weights into shared memory) can be
// issued before the wait.  griddep_launch_dependents() lets the next such
// kernel start early.  Both are no-ops for a kernel launched normally.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Record a kernel-side failure (a wait that gave up) in the device error word
// `err` (one int per device, read and cleared by qg_device_status()).
__device__ __forceinline__ void raise_device_error(int *err, int code) {
    if (err != nullptr) atomicExch(err, code);
}

}  // namespace qg
