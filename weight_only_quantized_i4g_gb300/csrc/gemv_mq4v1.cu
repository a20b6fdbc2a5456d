// gemv_mq4v1.cu -- decode GEMV for MQ4 v1 (hipfire qt=13): f32 scale and zero per 256-weight block
// (the kernels are in gemv_mq4.cuh).
#include "gemv_mq4.cuh"

namespace qg {

size_t ws_mq4v1(int S, int I, int O) { return ws_mq4(S, I, O); }

int run_gemv_mq4v1(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st) {
    return run_gemv_mq4<13>(y, x, blocks, S, I, O, ws, ws_bytes, st, "qgemv_mq4v1");
}


int run_gemv_moe_mq4v1(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                        const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    return run_gemv_moe_mq4<13>(y, x, x_stride, table, n_experts, ids, n_slots, S, I, O, st);
}

}  // namespace qg
