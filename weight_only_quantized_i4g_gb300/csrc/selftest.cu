// selftest.cu -- qg_selftest_wait_timeout: one bounded barrier wait of the
// staging pipeline made to run out on purpose, so that the failure path the
// kernels share (give up, record QG_ETIMEOUT in the device error word, end
// the block's other waits, land the copies in flight, leave) runs on a GPU
// under test.  Nothing faults: the stall is a batch that is never issued.
#include "../../include/qgemv.h"
#include "launch.h"
#include "pipeline.cuh"

namespace qg {

int *device_error_word();   // cs_common.cu

constexpr uint32_t kSelftestBytes = 4096;
static __device__ __align__(128) uint8_t g_selftest_src[kSelftestBytes];   // copy source (zeros)
static __device__ int g_selftest_seen;                                     // what the block observed
static __device__ unsigned g_chain_word;                                   // counted by the launch chain

// Two warps.  Warp 0 (producer) streams one batch into the ring slot with a
// bulk copy and waits for the consumer to release the slot; warp 1 (consumer)
// takes that batch, then waits for a second batch that is never issued.  Both
// use the library's bounded waits with `limit` polls: the consumer gives up,
// raises QG_ETIMEOUT and sets the block's abort flag; the producer's wait ends
// on that flag; before leaving it waits (bounded) for its copy's phase, so no
// copy is in flight when the block exits.  Bits of g_selftest_seen: 1 the
// consumer gave up on the missing batch, 2 the producer's wait ended on the
// abort flag, 4 the first batch landed.
__global__ void __launch_bounds__(64) selftest_wait_timeout_kernel(uint32_t limit, int *err) {
    __shared__ __align__(128) uint8_t slot[kSelftestBytes];
    __shared__ uint64_t full, empty;
    __shared__ uint32_t abort_flag;
    volatile uint32_t *abort_word = &abort_flag;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&full, 1);
        mbar_init(&empty, 1);
        *abort_word = 0u;
        g_selftest_seen = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&full, kSelftestBytes);
            bulk_copy_g2s(slot, g_selftest_src, kSelftestBytes, &full);
            // the consumer releases phase 0 of `empty` after the first batch and
            // then waits for a second one; phase 1 never completes
            bool ok = mbar_wait_or_abort(&empty, 0u, abort_word, limit);
            if (ok) ok = mbar_wait_or_abort(&empty, 1u, abort_word, limit);
            if (!ok && *abort_word) atomicOr(&g_selftest_seen, 2);
            if (mbar_wait(&full, 0u, limit)) atomicOr(&g_selftest_seen, 4);   // the copy has landed
        }
        return;
    }
    // consumer: batch 0 (phase 0 of `full`), then batch 1, which is never issued
    if (!mbar_wait_or_abort(&full, 0u, abort_word, limit)) {
        if (lane == 0) raise_device_error(err, kErrTimeout);
        return;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty);
    if (!mbar_wait_or_abort(&full, 1u, abort_word, limit)) {
        if (lane == 0) {
            raise_device_error(err, kErrTimeout);
            *abort_word = 1u;
            atomicOr(&g_selftest_seen, 1);
        }
        return;
    }
}

// One link of the launch chain: let the next launch start, wait for the
// previous one, count.
__global__ void selftest_pdl_chain_kernel() {
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) g_chain_word += 1u;
}

}  // namespace qg

using namespace qg;

extern "C" int qg_selftest_pdl_chain(int blocks, int threads, int launches, qg_stream_t stream) {
    if (blocks < 1 || blocks > 65535 || threads < 32 || threads > 1024 || threads % 32 != 0 || launches < 1 ||
        launches > 100000) {
        set_error_detail("qg_selftest_pdl_chain: blocks in [1, 65535], threads in [32, 1024] (a multiple of 32), "
                         "launches in [1, 100000] (got %d, %d, %d)", blocks, threads, launches);
        return kEInval;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    for (int i = 0; i < launches; ++i) {
        cudaLaunchKernelEx(&cfg, selftest_pdl_chain_kernel);
        count_launch();
    }
    return check_launch("qg_selftest_pdl_chain");
}

extern "C" int qg_selftest_wait_timeout(int spin_limit, int *observed) {
    if (observed == nullptr) {
        set_error_detail("qg_selftest_wait_timeout: observed must be non-NULL");
        return kEInval;
    }
    if (spin_limit < 1 || (uint32_t)spin_limit > kSpinLimit) {
        set_error_detail("qg_selftest_wait_timeout: spin_limit must be in [1, %u] (got %d)", kSpinLimit, spin_limit);
        return kEInval;
    }
    int *err = device_error_word();
    if (err == nullptr) {
        set_error_detail("qg_selftest_wait_timeout: no device error word (no current device?)");
        return kECuda;
    }
    selftest_wait_timeout_kernel<<<1, 64>>>((uint32_t)spin_limit, err);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(observed, g_selftest_seen, sizeof(int));
    if (e != cudaSuccess) {
        set_error_detail("qg_selftest_wait_timeout: %s", cudaGetErrorString(e));
        return kECuda;
    }
    return kOk;
}
