// cs_common.cu -- host helpers of the column-stationary GEMVs: launch plans,
// the split-K reduction kernel, the per-device SM count and error details.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "gemv_cs.cuh"
#include "launch.h"

namespace qg {

// ---------------------------------------------------------------------------
// error detail (thread-local, read by qg_last_error)
// ---------------------------------------------------------------------------
static thread_local char g_detail[512];

void set_error_detail(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
}

const char *error_detail() { return g_detail; }

int check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_detail("%s: %s", what, cudaGetErrorString(e));
        return kECuda;
    }
    return kOk;
}

// ---------------------------------------------------------------------------
// SM count of the current device, cached per device ordinal
// ---------------------------------------------------------------------------
int num_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;  // no device: plan for a GB300
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
static int round_up(int a, int b) { return (a + b - 1) / b * b; }
static int cdiv(int a, int b) { return (a + b - 1) / b; }

CsPlan cs_plan(int units, int O, int u, int rb, int regs_per_thread) {
    const int nsm = num_sms();
    CsPlan pl;
    // columns: as few blocks per row as the thread limit allows
    const int per_block_max = kCsMaxThreads * u;
    int splits = cdiv(units, per_block_max);
    pl.nrowb = cdiv(O, rb);
    // short-O / long-I: split the row further until the grid covers the SMs,
    // keeping at least two warps of units per block
    if (pl.nrowb * splits < nsm) {
        const int want = cdiv(2 * nsm, pl.nrowb);
        const int most = units / (64 * u);
        if (most > splits) splits = want < most ? want : most;
    }
    if (splits < 1) splits = 1;
    pl.splits = splits;
    pl.units_per_split = cdiv(units, splits);
    pl.threads = round_up(cdiv(pl.units_per_split, u), 32);
    if (pl.threads > kCsMaxThreads) pl.threads = kCsMaxThreads;
    pl.units_per_split = pl.threads * u < pl.units_per_split ? pl.threads * u : pl.units_per_split;
    // rows: enough blocks to be resident at once, each walking several batches
    int regs = regs_per_thread < 32 ? 32 : regs_per_thread;
    int by_regs = 65536 / (regs * pl.threads);
    int by_threads = 2048 / pl.threads;
    int per_sm = by_regs < by_threads ? by_regs : by_threads;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 16) per_sm = 16;
    const long resident = (long)nsm * per_sm / (splits > 0 ? splits : 1);
    pl.grid_x = pl.nrowb < resident ? pl.nrowb : (int)(resident > 0 ? resident : 1);
    return pl;
}

// ---------------------------------------------------------------------------
// split-K reduction
// ---------------------------------------------------------------------------
__global__ void splitk_reduce_kernel(float *__restrict__ y, const float *__restrict__ ws, int splits,
                                     size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int k = 0; k < splits; ++k) acc += ws[(size_t)k * n + i];
        y[i] = acc;
    }
}

void launch_splitk_reduce(float *y, const float *ws, int splits, int S, int O, cudaStream_t st) {
    const size_t n = (size_t)S * O;
    int blocks = (int)((n + 255) / 256);
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    splitk_reduce_kernel<<<blocks, 256, 0, st>>>(y, ws, splits, n);
}

}  // namespace qg
