// gemm_i4g.cu -- fmt=4 batched-prefill dequant-GEMM, general kernel.
//
// Y[m, o] = sum_i X[m, i] * (n(o,i) - 8) * scale[o, i/gs]   (colibri PR #457,
// section 4: the large-batch path takes the same grouped layout as the GEMV).
//
// This kernel covers every shape and alignment with CUDA cores: a 64x64
// output tile per block, K in steps of 32; the weight tile is dequantized to
// f32 in shared memory, the activation tile widened from bf16 to f32, and
// each thread accumulates a 4x4 sub-tile in f32.  The tensor-core kernel
// (gemm_i4g_tc.cu) takes the aligned shapes.
#include "common.cuh"
#include "launch.h"

namespace qg {

constexpr int kGT = 64;   // tile edge (rows of W and rows of X)
constexpr int kGK = 32;   // K step

__global__ void __launch_bounds__(256)
gemm_i4g_general_kernel(float *__restrict__ Y, const uint16_t *__restrict__ X, const uint8_t *__restrict__ w,
                        const float *__restrict__ scales, int M, int I, int O, int gs) {
    __shared__ float Ws[kGK][kGT + 1];   // [k][o]
    __shared__ float Xs[kGK][kGT + 1];   // [k][m]
    const int o0 = blockIdx.x * kGT, m0 = blockIdx.y * kGT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads, 4x4 each
    const size_t rb = ((size_t)I + 1) / 2;
    const int ng = (I + gs - 1) / gs;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < I; k0 += kGK) {
        for (int e = threadIdx.x; e < kGK * kGT; e += blockDim.x) {
            const int kk = e % kGK, r = e / kGK;
            const int i = k0 + kk;
            const int o = o0 + r, m = m0 + r;
            float wv = 0.f, xv = 0.f;
            if (o < O && i < I) {
                const uint8_t b = w[(size_t)o * rb + (i >> 1)];
                const int q = (int)((i & 1) ? (b >> 4) : (b & 0xF)) - 8;
                wv = (float)q * scales[(size_t)o * ng + i / gs];
            }
            if (m < M && i < I) xv = bf16_bits_to_f32(X[(size_t)m * I + i]);
            Ws[kk][r] = wv;
            Xs[kk][r] = xv;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kGK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                a[t] = Xs[kk][ty * 4 + t];
                b[t] = Ws[kk][tx * 4 + t];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int m = m0 + ty * 4 + r;
        if (m >= M) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int o = o0 + tx * 4 + c;
            if (o < O) Y[(size_t)m * O + o] = acc[r][c];
        }
    }
}

int run_gemm_i4g_general(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I,
                         int O, int gs, cudaStream_t st) {
    dim3 grid((O + kGT - 1) / kGT, (M + kGT - 1) / kGT);
    gemm_i4g_general_kernel<<<grid, 256, 0, st>>>(Y, X, w, scales, M, I, O, gs);
    return check_launch("qgemm_i4g (general kernel)");
}

}  // namespace qg
