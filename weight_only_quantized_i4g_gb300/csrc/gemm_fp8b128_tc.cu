// gemm_fp8b128_tc.cu -- fmt=7 prefill GEMM with f32 block scales on the tensor
// cores (the policy is in gemm_fp8_tc.cuh).
#include "gemm_fp8_tc.cuh"

namespace qg {

size_t ws_gemm_fp8b128(int M, int I, int O) { return ws_gemm_fp8(M, I, O); }

int run_gemm_fp8b128_tc(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv, int M, int I,
                        int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    return run_gemm_fp8_tc<ScaleF32>(Y, X, w, scale_inv, M, I, O, ws, ws_bytes, st, taken);
}

}  // namespace qg
