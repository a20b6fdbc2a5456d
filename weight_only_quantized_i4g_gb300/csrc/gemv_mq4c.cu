// gemv_mq4c.cu -- decode GEMV for MQ4C pad (hipfire qt=45): fp16 scale and zero per 256-weight block
// (the kernels are in gemv_mq4.cuh).
#include "gemv_mq4.cuh"

namespace qg {

size_t ws_mq4c(int S, int I, int O) { return ws_mq4(S, I, O); }

int run_gemv_mq4c(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st) {
    return run_gemv_mq4<45>(y, x, blocks, S, I, O, ws, ws_bytes, st, "qgemv_mq4c");
}


int run_gemv_moe_mq4c(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                        const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    return run_gemv_moe_mq4<45>(y, x, x_stride, table, n_experts, ids, n_slots, S, I, O, st);
}

}  // namespace qg
