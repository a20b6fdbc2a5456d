// launch.h -- internal interface between the C ABI (abi.cu) and the kernels.
// Arguments reaching these functions have been validated by abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace qg {

// Status codes mirror qg_status in include/qgemv.h.
enum { kOk = 0, kEInval = -1, kEGs = -2, kEShape = -3, kEAlign = -4, kEWorkspace = -5, kECuda = -6 };

// Records a refusal / error detail for qg_last_error() (thread-local).
void set_error_detail(const char *fmt, ...);

// Reports launch errors of the kernels just enqueued.
int check_launch(const char *what);

// Kernel launches of this library in this process (qg_launch_count()); every
// launch site counts itself.
inline std::atomic<unsigned long long> g_launches{0};
inline void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Reads and clears this device's kernel error word (0 or a qg status).
int read_device_error(int *status);

// Stamps build: copies min(max_blocks, kStampBlocks) blocks' timeline stamps
// to host and clears them (qg_stamps_take); kEInval in other builds.
int stamps_take(unsigned long long *host, int max_blocks);

// A process-unique id of the CUDA context current on this thread (the
// driver's context id), 0 when no context is current or the driver cannot
// say.  Device addresses of the library's __device__ variables and kernel
// attributes belong to a context, not to a device ordinal: after
// cudaDeviceReset the runtime creates a new primary context, and a caller
// may make its own driver-API context current.  Host caches of either are
// therefore keyed on this id.
unsigned long long current_context_id();

// One cached value per context, for up to kSlots contexts (the oldest entry
// is reused after that).  get() returns the value of the current context,
// computing it with fill(&value) -> status the first time that context asks;
// fill runs with the context current and under the cache's lock.
template <class T, int kSlots = 16>
class PerContext {
  public:
    template <class Fill>
    int get(T *out, Fill fill) {
        std::lock_guard<std::mutex> lk(mu_);
        unsigned long long id = current_context_id();
        if (id != 0)
            for (int i = 0; i < kSlots; ++i)
                if (ids_[i] == id) {
                    *out = vals_[i];
                    return kOk;
                }
        T v{};
        const int rc = fill(&v);
        if (rc != kOk) return rc;
        if (id == 0) id = current_context_id();   // fill may have created the primary context
        if (id != 0) {
            ids_[next_] = id;
            vals_[next_] = v;
            next_ = (next_ + 1) % kSlots;
        }
        *out = v;
        return kOk;
    }

  private:
    std::mutex mu_;
    unsigned long long ids_[kSlots] = {};
    T vals_[kSlots] = {};
    int next_ = 0;
};

// Sets a kernel's dynamic shared-memory limit (bytes) in the current context,
// once per (context, kernel).  The record lives in one table of this library
// (not in a static of a template function: those are merged across every
// loaded copy of a library by the dynamic loader, so a second copy -- such as
// the bounds-checking build in a test process -- would see the first copy's
// kernels as configured and skip its own).
void set_max_dynamic_smem(const void *kernel, int bytes);

size_t ws_i4g(int S, int I, int O, int gs);
size_t ws_fp8b128(int S, int I, int O);
size_t ws_fp8ue8m0(int S, int I, int O);
size_t ws_mq4v2(int S, int I, int O);
size_t ws_mq4v1(int S, int I, int O);
size_t ws_mq4c(int S, int I, int O);
size_t ws_q2_0(int S, int I, int O);

int run_gemv_i4g(float *y, const float *x, const uint8_t *w, const float *scales, int S, int I, int O,
                 int gs, void *ws, size_t ws_bytes, cudaStream_t st);
int run_gemv_fp8b128(float *y, const uint16_t *x, const uint8_t *w, const float *scale_inv, int S,
                     int I, int O, void *ws, size_t ws_bytes, cudaStream_t st);
int run_gemv_fp8ue8m0(float *y, const uint16_t *x, const uint8_t *w, const uint8_t *scale_e8m0, int S,
                      int I, int O, void *ws, size_t ws_bytes, cudaStream_t st);
int run_gemv_mq4v2(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st);
int run_gemv_mq4v1(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st);
int run_gemv_mq4c(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                  size_t ws_bytes, cudaStream_t st);
int run_gemv_q2_0(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                  size_t ws_bytes, cudaStream_t st);


// Routed experts: n_slots GEMVs of one shape in one launch; `table` is a
// device array of {weights, scales} pointer pairs (qg_expert), `ids` a device
// array of n_slots expert ids, slot r reads x + r * x_stride (elements).
int run_gemv_moe_i4g(float *y, const float *x, size_t x_stride, const void *table, int n_experts,
                     const int *ids, int n_slots, int S, int I, int O, int gs, cudaStream_t st);
int run_gemv_moe_fp8b128(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                         const int *ids, int n_slots, int S, int I, int O, cudaStream_t st);
int run_gemv_moe_fp8ue8m0(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                          const int *ids, int n_slots, int S, int I, int O, cudaStream_t st);
int run_gemv_moe_mq4v2(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                       const int *ids, int n_slots, int S, int I, int O, cudaStream_t st);
int run_gemv_moe_mq4v1(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                       const int *ids, int n_slots, int S, int I, int O, cudaStream_t st);
int run_gemv_moe_mq4c(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                      const int *ids, int n_slots, int S, int I, int O, cudaStream_t st);

// Routed-expert prefill on the tensor cores: up to kMoeGroupsPerLaunch groups
// of token-sorted rows in one launch (row0[g], rows[g] > 0 relative to X and
// Y; w[g], scales[g] the group's weights).  *taken is false when the shapes
// or pointers do not suit the tensor-core kernel (nothing is launched).
constexpr int kMoeGroupsPerLaunch = 64;
size_t ws_gemm_moe_i4g(const int *rows, int n, int M, int I, int O, int gs);
size_t ws_gemm_moe_fp8(const int *rows, int n, int M, int I, int O);
size_t ws_gemm_moe_mq4(const int *rows, int n, int M, int I, int O);
int run_gemm_moe_i4g_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                        const float *const *scales, int n, int M, int I, int O, int gs, void *ws, size_t ws_bytes,
                        cudaStream_t st, bool *taken);
int run_gemm_moe_fp8b128_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                            const float *const *scales, int n, int M, int I, int O, void *ws, size_t ws_bytes,
                            cudaStream_t st, bool *taken);
int run_gemm_moe_fp8ue8m0_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                             const float *const *scales, int n, int M, int I, int O, void *ws, size_t ws_bytes,
                             cudaStream_t st, bool *taken);
int run_gemm_moe_mq4v2_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                          int n, int M, int I, int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);
int run_gemm_moe_mq4v1_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                          int n, int M, int I, int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);
int run_gemm_moe_mq4c_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                         int n, int M, int I, int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);

int run_quantize_i4g(uint8_t *wq, float *scales, const float *w, int O, int I, int gs, cudaStream_t st);
int run_encode_mq4v2(uint8_t *blocks, const float *w, int O, int I, cudaStream_t st);
int run_encode_mq4_one_header(uint8_t *blocks, const float *w, int O, int I, bool fp16_header, cudaStream_t st);
int run_fwht256(float *out, const float *in, const int8_t *signs, size_t nblocks, cudaStream_t st);

}  // namespace qg
