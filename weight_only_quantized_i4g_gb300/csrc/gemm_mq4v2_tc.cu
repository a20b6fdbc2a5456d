// gemm_mq4v2_tc.cu -- MQ4-V2 (hipfire qt=44) batched-prefill dequant-GEMM on the tensor cores
// (the format policy is in gemm_mq4_tc.cuh, the kernel in gemm_tc.cuh).
#include "gemm_mq4_tc.cuh"

namespace qg {

size_t ws_gemm_mq4v2(int M, int I, int O) { return ws_gemm_mq4(M, I, O); }

int run_gemm_mq4v2_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                      size_t ws_bytes, cudaStream_t st, bool *taken) {
    return run_gemm_mq4_tc<44>(Y, X, blocks, M, I, O, ws, ws_bytes, st, taken, "qgemm_mq4v2");
}

size_t ws_gemm_moe_mq4(const int *rows, int n, int M, int I, int O) { return ws_gemm_moe_mq4_impl(rows, n, M, I, O); }

int run_gemm_moe_mq4v2_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                          int n, int M, int I, int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    return run_gemm_moe_mq4_tc<44>(Y, X, row0, rows, w, n, M, I, O, ws, ws_bytes, st, taken);
}

}  // namespace qg
