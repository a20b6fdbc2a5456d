// gemm_fp8_tc.cuh -- fmt=7 (FP8-e4m3, 128x128 block scales) batched-prefill
// dequant-GEMM on the tensor cores: the format policy of the kernel in
// gemm_tc.cuh, templated on the block-scale encoding SC (f32 or UE8M0;
// instantiated by gemm_fp8b128_tc.cu and gemm_fp8ue8m0_tc.cu).
//
// colibri PR #528 "fmt=7: fp8-e4m3-b128 passthrough weight format", section
// "Design": W[o, i] = e4m3(code) * scale_inv[o/128, i/128] (a multiply), and
// Y[m, o] = sum_i X[m, i] * W[o, i].  Here each weight is formed in f32 (the
// e4m3 value is exact in f16 and f32; one rounding of the product), scaled by
// the row's power of two and rounded to fp16 for the MMA.  A NaN code stays
// NaN and makes its output column NaN through the MMA.
//
// One dequantizing thread takes 32 codes of its row per K step (two 16-byte
// loads).  A 128-row tile lies inside one block row of scale_inv and a K
// step inside one block column, so the thread needs one scale per step.
#pragma once
#include "gemm_tc.cuh"

namespace qg {
namespace tc {

// Two e4m3 codes (the low and high byte of `two`) -> f16x2 of code * s,
// low byte in the low half.
__device__ __forceinline__ uint32_t e4m3x2_scaled_f16x2(uint16_t two, uint64_t s2) {
    uint32_t r;
    asm("{\n\t.reg .b32 h2;\n\t.reg .f16 fl, fh;\n\t.reg .f32 a, b;\n\t.reg .b64 t;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, %1;\n\t"
        "mov.b32 {fl, fh}, h2;\n\t"
        "cvt.f32.f16 a, fl;\n\t"
        "cvt.f32.f16 b, fh;\n\t"
        "mov.b64 t, {a, b};\n\t"
        "mul.rn.f32x2 t, t, %2;\n\t"
        "mov.b64 {a, b}, t;\n\t"
        "cvt.rn.f16x2.f32 %0, b, a;\n\t}"
        : "=r"(r)
        : "h"(two), "l"(s2));
    return r;
}

// Args::scales carries the block scales as SC::T (bytes for UE8M0).
template <class SC>
struct PolicyFp8 {
    static constexpr const char *kName = SC::kGemmTc;
    static __device__ __forceinline__ const typename SC::T *scales_of(const float *scales) {
        return reinterpret_cast<const typename SC::T *>(scales);
    }
    // Bound on |w| over row o, |e4m3| <= 448: 448 max_k |scale_inv[o/128, k]|
    // (the same for every row of a 128-row block).  Called by a whole warp.
    static __device__ __forceinline__ float row_bound(const Args &a, const uint8_t *, const float *scales, int o,
                                                      int lane) {
        const typename SC::T *src = scales_of(scales) + (size_t)(o >> 7) * a.nbi;
        float b = 0.f;
#pragma unroll 4
        for (int k = lane; k < a.nbi; k += 32) b = fmaxf(b, fabsf(SC::get(src, k)));
        return 448.f * warp_max(b);
    }
    struct Fetch {
        uint4 q0, q1;
        float s;
    };
    struct Row {
        const uint8_t *w;
        const typename SC::T *s;
    };
    static __device__ __forceinline__ void row_begin(const Args &a, const uint8_t *w, const float *scales, int o,
                                                     int kq, int, Row &r) {
        const bool in = o < a.O;
        r.w = in ? w + (size_t)o * (size_t)a.rowbytes + kq * 32 : nullptr;
        r.s = in ? scales_of(scales) + (size_t)(o >> 7) * a.nbi : nullptr;
    }
    static __device__ __forceinline__ void clear(Fetch &f) {
        f.q0 = make_uint4(0u, 0u, 0u, 0u);
        f.q1 = f.q0;
        f.s = 0.f;
    }
    static __device__ __forceinline__ void fetch(const Args &, Row &r, int pk, int, bool skip, Fetch &f) {
        if (r.w && !skip) {
            const uint8_t *p = r.w + (size_t)pk * kBK;
            f.q0 = ldg_w16(p);
            f.q1 = ldg_w16(p + 16);
            f.s = SC::get(r.s, pk);
        }
    }
    static __device__ __forceinline__ void dequant(const Fetch &f, float p2, uint32_t (&col)[16]) {
        const float s = f.s * p2;
        const uint64_t s2 = f32_pair(s, s);
        const uint32_t wv[8] = {f.q0.x, f.q0.y, f.q0.z, f.q0.w, f.q1.x, f.q1.y, f.q1.z, f.q1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            col[2 * j] = e4m3x2_scaled_f16x2((uint16_t)wv[j], s2);
            col[2 * j + 1] = e4m3x2_scaled_f16x2((uint16_t)(wv[j] >> 16), s2);
        }
    }
};

}  // namespace tc

// Shapes the tensor-core kernel takes: K in whole 64-steps (a last step of
// 64), 16-byte aligned w (rows of I bytes then start on 16-byte boundaries)
// and a TMA-aligned X.
inline bool gemm_fp8_tc_ok(const uint16_t *X, const uint8_t *w, int I) {
    return I % tc::kBKBox == 0 && (uintptr_t)X % 16 == 0 && (uintptr_t)w % 16 == 0;
}

inline size_t ws_gemm_fp8(int M, int I, int O) {
    if (I % tc::kBKBox != 0) return 0;
    return tc::choose_plan(M, I, O).ws_bytes;
}

template <class SC>
int run_gemm_fp8_tc(float *Y, const uint16_t *X, const uint8_t *w, const typename SC::T *scale_inv, int M, int I,
                    int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    *taken = false;
    if (!gemm_fp8_tc_ok(X, w, I)) return kOk;
    *taken = true;
    const tc::Plan p = tc::choose_plan(M, I, O);
    if (ws == nullptr || ws_bytes < p.ws_bytes) {
        set_error_detail("%s: this shape needs a workspace of %zu bytes (got %zu)", SC::kGemm, p.ws_bytes,
                         ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    tc::Args args{};
    args.w = w;
    args.scales = reinterpret_cast<const float *>(scale_inv);   // read back as SC::T by the policy
    args.nbi = (I + tc::kBK - 1) / tc::kBK;
    args.rowbytes = I;
    return tc::launch_plan<tc::PolicyFp8<SC>>(p, Y, X, args, M, I, O, ws, st);
}

template <class SC>
int run_gemm_moe_fp8_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                        const float *const *scales, int n, int M, int I, int O, void *ws, size_t ws_bytes,
                        cudaStream_t st, bool *taken) {
    *taken = false;
    for (int g = 0; g < n; ++g)
        if (!gemm_fp8_tc_ok(X, w[g], I)) return kOk;
    *taken = true;
    tc::Args args{};
    args.nbi = (I + tc::kBK - 1) / tc::kBK;
    args.rowbytes = I;
    return tc::launch_grouped<tc::PolicyFp8<SC>>(Y, X, args, row0, rows, w, scales, n, M, I, O, ws, ws_bytes, st);
}

}  // namespace qg
