// gemv_mq4v2.cu -- decode GEMV for MQ4-V2 (hipfire qt=44): fp16 scale and zero per 128-weight half
// (the kernels are in gemv_mq4.cuh).
#include "gemv_mq4.cuh"

namespace qg {

size_t ws_mq4v2(int S, int I, int O) { return ws_mq4(S, I, O); }

int run_gemv_mq4v2(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st) {
    return run_gemv_mq4<44>(y, x, blocks, S, I, O, ws, ws_bytes, st, "qgemv_mq4v2");
}


int run_gemv_moe_mq4v2(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                        const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    return run_gemv_moe_mq4<44>(y, x, x_stride, table, n_experts, ids, n_slots, S, I, O, st);
}

}  // namespace qg
