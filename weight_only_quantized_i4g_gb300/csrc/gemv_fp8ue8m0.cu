// gemv_fp8ue8m0.cu -- fmt=7 decode GEMV with UE8M0 block scales: one byte per
// 128x128 block, the power of two 2^(e - 127) (the kernels are in gemv_fp8.cuh).
#include "gemv_fp8.cuh"

namespace qg {

size_t ws_fp8ue8m0(int S, int I, int O) { return ws_fp8(S, I, O); }

int run_gemv_fp8ue8m0(float *y, const uint16_t *x, const uint8_t *w, const uint8_t *scale_e8m0, int S, int I,
                      int O, void *ws, size_t ws_bytes, cudaStream_t st) {
    return run_gemv_fp8<ScaleE8M0>(y, x, w, scale_e8m0, S, I, O, ws, ws_bytes, st, "qgemv_fp8ue8m0");
}

int run_gemv_moe_fp8ue8m0(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                          const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    return run_gemv_moe_fp8<ScaleE8M0>(y, x, x_stride, table, n_experts, ids, n_slots, S, I, O, st);
}

}  // namespace qg
