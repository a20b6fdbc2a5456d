// gemm_general.cu -- batched-prefill dequant-GEMM, general kernel, for the
// three weight formats:
//
//   Y[m, o] = sum_i X[m, i] * w(o, i)       X bf16 [M, I], Y f32 [M, O]
//
//   fmt=4   w = (n(o,i) - 8) * scale[o, i/gs]      colibri PR #457, sections 3, 4
//   fmt=7   w = e4m3(code) * scale_inv[o/128, i/128]  colibri PR #528, "Design"
//   MQ4-V2  w = q * scale[h] + zero[h]              hipfire "MQ4 V2", sections 2, 4
//   MQ4 v1, MQ4C pad: one header per 256 weights    hipfire "MQ4 V2", sections 1b, 1e
//
// This kernel covers every shape and alignment with CUDA cores: a 64x64
// output tile per block, K in steps of 32; the weight tile is dequantized to
// f32 in shared memory, the activation tile widened from bf16 to f32, and
// each thread accumulates a 4x4 sub-tile in f32.  The tensor-core kernel
// (gemm_tc.cuh) takes the aligned shapes.
#include "common.cuh"
#include "launch.h"

namespace qg {
namespace {

constexpr int kGT = 64;   // tile edge (rows of W and rows of X)
constexpr int kGK = 32;   // K step

struct WeightI4G {
    const uint8_t *w;
    const float *scales;
    size_t rb;
    int gs, ng;
    __device__ float operator()(int o, int i) const {
        const uint8_t b = w[(size_t)o * rb + (i >> 1)];
        const int q = (int)((i & 1) ? (b >> 4) : (b & 0xF)) - 8;
        return (float)q * scales[(size_t)o * ng + i / gs];
    }
};

template <class SC>
struct WeightFp8 {
    const uint8_t *w;
    const typename SC::T *scale_inv;
    int I, nbi;
    __device__ float operator()(int o, int i) const {
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)w[(size_t)o * I + i]));
        return f16_bits_to_f32((uint16_t)h2) * SC::get(scale_inv, (size_t)(o >> 7) * nbi + (i >> 7));
    }
};

// HK = 44: MQ4-V2 (fp16 pair per half), 45: MQ4C pad (one fp16 pair), 13:
// MQ4 v1 (f32 scale and zero).
template <int HK>
struct WeightMq4 {
    const uint8_t *blocks;
    int nb;   // blocks per row, I / 256
    __device__ float operator()(int o, int i) const {
        const uint8_t *b = blocks + ((size_t)o * nb + (i >> 8)) * 136;
        const int j = i & 255;
        const uint8_t p = b[8 + (j >> 1)];
        const float q = (float)((j & 1) ? (p >> 4) : (p & 0xF));
        if (HK == 13) {
            const float *h = reinterpret_cast<const float *>(b);   // blocks are 8-byte aligned
            return fmaf(q, h[0], h[1]);
        }
        const uint8_t *h = b + (HK == 44 ? 4 * (j >> 7) : 0);
        const uint16_t sc = (uint16_t)(h[0] | (h[1] << 8)), ze = (uint16_t)(h[2] | (h[3] << 8));
        return fmaf(q, f16_bits_to_f32(sc), f16_bits_to_f32(ze));
    }
};

template <class W>
__global__ void __launch_bounds__(256)
gemm_general_kernel(float *__restrict__ Y, const uint16_t *__restrict__ X, W wat, int M, int I, int O) {
    __shared__ float Ws[kGK][kGT + 1];   // [k][o]
    __shared__ float Xs[kGK][kGT + 1];   // [k][m]
    const int o0 = blockIdx.x * kGT, m0 = blockIdx.y * kGT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads, 4x4 each
    float acc[4][4] = {};
    for (int k0 = 0; k0 < I; k0 += kGK) {
        for (int e = threadIdx.x; e < kGK * kGT; e += blockDim.x) {
            const int kk = e % kGK, r = e / kGK;
            const int i = k0 + kk;
            const int o = o0 + r, m = m0 + r;
            Ws[kk][r] = (o < O && i < I) ? wat(o, i) : 0.f;
            Xs[kk][r] = (m < M && i < I) ? bf16_bits_to_f32(X[(size_t)m * I + i]) : 0.f;
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

template <class W>
int launch_general(float *Y, const uint16_t *X, const W &wat, int M, int I, int O, cudaStream_t st,
                   const char *what) {
    dim3 grid((O + kGT - 1) / kGT, (M + kGT - 1) / kGT);
    gemm_general_kernel<W><<<grid, 256, 0, st>>>(Y, X, wat, M, I, O);
    count_launch();
    return check_launch(what);
}

}  // namespace

int run_gemm_i4g_general(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I,
                         int O, int gs, cudaStream_t st) {
    const WeightI4G wat{w, scales, ((size_t)I + 1) / 2, gs, (I + gs - 1) / gs};
    return launch_general(Y, X, wat, M, I, O, st, "qgemm_i4g (general kernel)");
}

int run_gemm_fp8b128_general(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv, int M,
                             int I, int O, cudaStream_t st) {
    const WeightFp8<ScaleF32> wat{w, scale_inv, I, (I + 127) / 128};
    return launch_general(Y, X, wat, M, I, O, st, ScaleF32::kGemmGeneral);
}

int run_gemm_fp8ue8m0_general(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0, int M,
                              int I, int O, cudaStream_t st) {
    const WeightFp8<ScaleE8M0> wat{w, scale_e8m0, I, (I + 127) / 128};
    return launch_general(Y, X, wat, M, I, O, st, ScaleE8M0::kGemmGeneral);
}

int run_gemm_mq4v2_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                           cudaStream_t st) {
    const WeightMq4<44> wat{blocks, I / 256};
    return launch_general(Y, X, wat, M, I, O, st, "qgemm_mq4v2 (general kernel)");
}

int run_gemm_mq4v1_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                           cudaStream_t st) {
    const WeightMq4<13> wat{blocks, I / 256};
    return launch_general(Y, X, wat, M, I, O, st, "qgemm_mq4v1 (general kernel)");
}

int run_gemm_mq4c_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                          cudaStream_t st) {
    const WeightMq4<45> wat{blocks, I / 256};
    return launch_general(Y, X, wat, M, I, O, st, "qgemm_mq4c (general kernel)");
}

}  // namespace qg
