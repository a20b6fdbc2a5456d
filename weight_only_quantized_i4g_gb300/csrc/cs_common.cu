// cs_common.cu -- host helpers of the column-stationary GEMVs: launch plans,
// the split-K reduction kernel, the per-device SM count and error details.
#include <stdarg.h>
#include <stdio.h>

#include <cmath>
#include <mutex>

#include <cuda.h>

#include "gemv_cs.cuh"
#include "gemv_tma.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qg {

// One error word per device: kernels that give up waiting set it; the host
// reads and clears it with qg_device_status().  The stamps build keeps the
// kernels' timeline stamps after it (common.cuh).
#ifdef QG_STAMPS
__device__ __align__(16) int g_device_error[kStampOffsetInts + 2 * kStampSlots * kStampBlocks];
#else
__device__ int g_device_error = 0;
#endif

unsigned long long current_context_id() {
    typedef CUresult (*GetCurrentFn)(CUcontext *);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long *);
    static std::once_flag once;
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
        cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

void set_max_dynamic_smem(const void *kernel, int bytes) {
    struct Entry { unsigned long long ctx; const void *fn; };
    static std::mutex mu;
    static Entry table[512];
    static int n = 0, next = 0;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(mu);
    if (ctx != 0)
        for (int i = 0; i < n; ++i)
            if (table[i].ctx == ctx && table[i].fn == kernel) return;
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaGetLastError();
    const unsigned long long id = ctx != 0 ? ctx : current_context_id();
    if (id == 0) return;
    table[next] = Entry{id, kernel};
    next = (next + 1) % 512;
    if (n < 512) ++n;
}

int stamps_take(unsigned long long *host, int max_blocks) {
#ifdef QG_STAMPS
    const int nb = max_blocks < kStampBlocks ? max_blocks : kStampBlocks;
    void *p = nullptr;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_device_error);
    unsigned long long *area =
        p != nullptr ? reinterpret_cast<unsigned long long *>(static_cast<int *>(p) + kStampOffsetInts) : nullptr;
    if (e == cudaSuccess)
        e = cudaMemcpy(host, area, (size_t)nb * kStampSlots * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(area, 0, (size_t)kStampBlocks * kStampSlots * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        set_error_detail("qg_stamps_take: %s", cudaGetErrorString(e));
        return kECuda;
    }
    return kOk;
#else
    (void)host;
    (void)max_blocks;
    set_error_detail("qg_stamps_take: this library was built without stamps (the stamps build is "
                     "libqgemv_stamps.so, from _build.py --stamps)");
    return kEInval;
#endif
}

int *device_error_word() {
    static PerContext<int *> cache;
    int *w = nullptr;
    const int rc = cache.get(&w, [](int **out) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return (int)kECuda;
        }
        *out = static_cast<int *>(p);
        return (int)kOk;
    });
    return rc == kOk ? w : nullptr;
}

int read_device_error(int *status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) {
        set_error_detail("qg_device_status: %s", cudaGetErrorString(e));
        return kECuda;
    }
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
        if (e != cudaSuccess) {
            set_error_detail("qg_device_status: %s", cudaGetErrorString(e));
            return kECuda;
        }
    }
    *status = v;
    return kOk;
}

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
// plan of the staged (TMA) kernel
// ---------------------------------------------------------------------------
bool tma_plan(const TmaGeom &g, int S, int O, int RB, int NV, int U_max, TmaPlan *pl, int max_per_sm,
              int one_block_slots) {
    int U = 1, splits = 1;
    // unit slots per block: consumer threads / token groups
    int max_thr = tma_max_consumer_warps(S, 1) * 32 / g.tg;
    if (g.units > max_thr) {
        max_thr = tma_max_consumer_warps(S, 2) * 32 / g.tg;
        if (g.units <= max_thr * U_max) {
            U = cdiv(g.units, max_thr);
        } else {
            U = U_max;
            splits = cdiv(g.units, max_thr * U);
        }
    }
    int ups = cdiv(g.units, splits);
    if (splits > 1) {
        ups = round_up(ups, g.granule);
        splits = cdiv(g.units, ups);
    }
    if (cdiv(ups, U) > max_thr) return false;
    const uint32_t seg = splits == 1 ? g.rowbytes : (uint32_t)(ups / g.granule) * g.granule_bytes;
    if (seg % 16 != 0 || g.rowbytes % 16 != 0 || g.arowbytes % 4 != 0) return false;
    const int nc = cdiv(cdiv(ups, U) * g.tg, 32);
    const uint32_t stage_w = (uint32_t)round_up((int)(RB * seg), 128);
    const uint32_t stage_a = (uint32_t)round_up((int)(RB * g.arowbytes), 128);
    const uint32_t red_stage = (uint32_t)(nc * NV * 4);
    const uint32_t per_slot = stage_w + stage_a + red_stage + 16;
    // aim for about 16 consumer warps per SM, up to 8 blocks; then as many
    // ring slots (2..6) as that share of the 228 KB of shared memory holds
    int nst = 0;
    int target = 16 / nc;
    if (target < 1) target = 1;
    if (target > max_per_sm) target = max_per_sm;
    for (; target >= 1; --target) {
        long budget = 233472L / target - 1024;
        if (budget > 232448) budget = 232448;
        nst = (int)(budget / per_slot);
        if (nst > 6) nst = 6;
        if (target == 1 && nst > one_block_slots) nst = one_block_slots;
        if (nst >= 2) break;
    }
    if (nst < 2) return false;
    pl->per_sm = target;
    pl->rb = RB;
    pl->units = g.units;
    pl->U = U;
    pl->nc = nc;
    pl->splits = splits;
    pl->units_per_split = ups;
    pl->nrowb = cdiv(O, RB);
    pl->nst = nst;
    pl->L.stage_w = stage_w;
    pl->L.stage_a = stage_a;
    pl->L.red_off = (uint32_t)nst * (stage_w + stage_a);
    pl->L.bar_off = (uint32_t)round_up((int)(pl->L.red_off + nst * red_stage), 16);
    pl->L.total = pl->L.bar_off + 16u * (uint32_t)nst;
    return true;
}

bool tma_plan_rows(const TmaGeom &g, int S, int O, int U_max, TmaPlan *pl) {
    // A small matrix (a few MB) is over in a few microseconds, and every
    // block loads the whole activation row: with several blocks per SM that
    // load rivals the weights the SM streams (fmt=4 2048x7168 with f32 x:
    // 28 KB of x per block against 54 KB of weights per SM).  One block per
    // SM with 8-row batches measured 30% faster there (6.2 -> 4.3 us); 4- and
    // 2-row batches were slower (5.1, 6.2 us).  A matrix with fewer 8-row
    // batches than SMs (under 1216 rows) takes 4-row batches on the same plan
    // (Q2_0 640x2560: 3.25 -> 2.85 us) before the general plan below.
    if (S <= 2 && (double)O * (g.rowbytes + g.arowbytes) < 32e6) {
        for (int rb = 8; rb >= 4; rb /= 2) {
            TmaPlan t;
            if (tma_plan(g, S, O, rb, next_pow2(rb * S), U_max, &t, 1, 6) && (long)t.nrowb * t.splits >= num_sms()) {
                *pl = t;
                return true;
            }
        }
    }
    const int cands[3] = {8, 4, 2};
    bool have = false, have_bal = false;
    TmaPlan last, bal;
    double bal_eff = 0.0;
    for (int i = 0; i < 3; ++i) {
        const int rb = cands[i];
        if (S > 2 && rb == 8) continue;
        TmaPlan t;
        if (!tma_plan(g, S, O, rb, next_pow2(rb * S), U_max, &t)) continue;
        if (rb == 2 && t.U > 1) continue;
        last = t;
        have = true;
        // Batches per resident block: at least three to overlap, and an even
        // last wave (a block with one batch more than the mean sets the time).
        const double resident = (double)num_sms() * t.per_sm;
        const double waves = (double)t.nrowb * t.splits / resident;
        if (waves >= 3.0) {
            const double eff = waves / std::ceil(waves);
            if (eff >= 0.92) {
                *pl = t;
                return true;
            }
            if (!have_bal || eff > bal_eff) {
                bal = t;
                bal_eff = eff;
                have_bal = true;
            }
        }
    }
    if (have_bal) *pl = bal;
    else if (have) *pl = last;
    return have;
}

// ---------------------------------------------------------------------------
// split-K reduction
// ---------------------------------------------------------------------------
__global__ void splitk_reduce_kernel(float *__restrict__ y, const float *__restrict__ ws, int splits,
                                     size_t n) {
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();   // ws is the previous kernel's output
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
    // Launched as a programmatic dependent of the GEMV that fills ws: it
    // starts early and waits in the kernel (griddep_wait) for that GEMV.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, y, ws, splits, n);
    count_launch();
}

}  // namespace qg
