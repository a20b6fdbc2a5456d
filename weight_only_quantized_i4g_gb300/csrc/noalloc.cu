// noalloc.cu -- qgemv_i4g_noalloc: the fmt=4 decode GEMV for callers that
// cannot allocate device memory.
//
// qgemv_i4g needs a caller workspace when a row is too long for one thread
// block (the reduction is split across blocks and summed in a second pass).
// Some callers cannot provide one: an inference engine whose device memory is
// planned once at start-up and handed out by its own allocator, or host code
// that must not call cudaMalloc on the decode path because that call can
// block until the device is idle.  This entry point takes its scratch from a
// fixed array that lives in the library's device image instead, so it
// allocates nothing.  The array is shared by every call on a device and keeps
// the previous call's contents; calls whose kernels overlap on the GPU
// (several streams, or several host threads) race on it and must be ordered
// by the caller.
#include "../../include/qgemv.h"
#include "launch.h"

namespace qg {

// Scratch for the split partial sums: [splits, S, O] floats.  Every element
// that the summing pass reads is written by the same call first, so nothing
// has to be cleared between calls.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;   // 4 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch array in the current context.  In host code
// `g_noalloc_scratch` names a host-side stand-in, not device memory, so the
// address is looked up with cudaGetSymbolAddress, with the caller's device
// current, the first time a context calls, and cached per context: a context
// made after cudaDeviceReset, or a driver-API context of the caller's own,
// gets its own address rather than a stale one.
int noalloc_scratch(void **out) {
    static PerContext<void *> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error_detail("qgemv_i4g_noalloc: no current device (%s)", cudaGetErrorString(e));
        cudaGetLastError();
        return kECuda;
    }
    return cache.get(out, [dev](void **p) {
        void *a = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&a, g_noalloc_scratch);
        if (r != cudaSuccess || a == nullptr) {
            set_error_detail("qgemv_i4g_noalloc: cannot locate the scratch array on device %d (%s)", dev,
                             cudaGetErrorString(r));
            cudaGetLastError();
            return (int)kECuda;
        }
        *p = a;
        return (int)kOk;
    });
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" int qgemv_i4g_noalloc(float *y, const float *x, const uint8_t *w, const float *scales, int S,
                                 int I, int O, int gs, qg_stream_t stream) {
    const char *fn = "qgemv_i4g_noalloc";
    if (S < 1 || I < 1 || O < 1) {
        set_error_detail("%s: S, I and O must be >= 1 (got %d, %d, %d)", fn, S, I, O);
        return kEInval;
    }
    if (gs < 2 || (gs & 1)) {
        set_error_detail("%s: gs = %d, must be even and >= 2", fn, gs);
        return kEGs;
    }
    if (!y || !x || !w || !scales) {
        set_error_detail("%s: y, x, w and scales must be non-NULL", fn);
        return kEInval;
    }
    if ((uintptr_t)y % 4 || (uintptr_t)x % 4 || (uintptr_t)scales % 4) {
        set_error_detail("%s: y, x and scales must be 4-byte aligned", fn);
        return kEAlign;
    }
    const size_t need = qg_workspace_bytes(QG_FMT_I4G, S, I, O, gs);
    if (need > kNoAllocScratchBytes) {
        set_error_detail("%s: this shape needs %zu bytes of split-reduction scratch, more than the "
                         "%zu bytes this entry point has (use qgemv_i4g with a workspace)",
                         fn, need, kNoAllocScratchBytes);
        return kEWorkspace;
    }
    void *scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc != kOk) return rc;
    cudaGetLastError();
    return run_gemv_i4g(y, x, w, scales, S, I, O, gs, scratch, kNoAllocScratchBytes,
                        reinterpret_cast<cudaStream_t>(stream));
}
