// gemv_fp8b128.cu -- fmt=7 decode GEMV with f32 block scales (the kernels are
// in gemv_fp8.cuh).
#include "gemv_fp8.cuh"

namespace qg {

size_t ws_fp8b128(int S, int I, int O) { return ws_fp8(S, I, O); }

int run_gemv_fp8b128(float *y, const uint16_t *x, const uint8_t *w, const float *scale_inv, int S, int I,
                     int O, void *ws, size_t ws_bytes, cudaStream_t st) {
    return run_gemv_fp8<ScaleF32>(y, x, w, scale_inv, S, I, O, ws, ws_bytes, st, "qgemv_fp8b128");
}

int run_gemv_moe_fp8b128(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                         const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    return run_gemv_moe_fp8<ScaleF32>(y, x, x_stride, table, n_experts, ids, n_slots, S, I, O, st);
}

}  // namespace qg
