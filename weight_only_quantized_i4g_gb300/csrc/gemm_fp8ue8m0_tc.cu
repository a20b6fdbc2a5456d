// gemm_fp8ue8m0_tc.cu -- fmt=7 prefill GEMM with UE8M0 block scales on the
// tensor cores (the policy is in gemm_fp8_tc.cuh).
#include "gemm_fp8_tc.cuh"

namespace qg {

size_t ws_gemm_fp8ue8m0(int M, int I, int O) { return ws_gemm_fp8(M, I, O); }

int run_gemm_fp8ue8m0_tc(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0, int M, int I,
                         int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    return run_gemm_fp8_tc<ScaleE8M0>(Y, X, w, scale_e8m0, M, I, O, ws, ws_bytes, st, taken);
}

int run_gemm_moe_fp8ue8m0_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                             const float *const *scales, int n, int M, int I, int O, void *ws, size_t ws_bytes,
                             cudaStream_t st, bool *taken) {
    return run_gemm_moe_fp8_tc<ScaleE8M0>(Y, X, row0, rows, w, scales, n, M, I, O, ws, ws_bytes, st, taken);
}

}  // namespace qg
