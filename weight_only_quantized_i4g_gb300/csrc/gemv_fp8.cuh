// gemv_fp8.cuh -- fmt=7 FP8-e4m3 decode GEMV with 128x128 block scales,
// templated on the scale encoding SC (instantiated by gemv_fp8b128.cu for f32
// scales and gemv_fp8ue8m0.cu for UE8M0 scales).
//
// Format (colibri PR #528, "Design"): O*I raw OCP E4M3-FN codes, row-major;
// one scale per 128x128 block, [ceil(O/128), ceil(I/128)] in row-major block
// order, either f32 (the encoding the page implements) or UE8M0 (the page's
// DeepSeek-V4 encoding: one byte per block, a power-of-two exponent):
//     W[o,i] = e4m3(code) * scale[o/128, i/128]   (multiply, not divide)
// The only NaN codes are 0x7F and 0xFF; a NaN weight propagates to its row.
//
// Decode: the hardware e4m3x2 -> f16x2 conversion (exact for every code:
// each E4M3-FN value, subnormals included, is an f16 value, and the NaN codes
// convert to NaN), then f16 -> f32 (exact).  A unit (4*NW codes, NW <= 4)
// lies inside one 128-column block, so the block scale multiplies the unit's
// partial sum.
//
// Paths, fastest first: staged (gemv_tma.cuh; 16-byte aligned w and x,
// I % 16 == 0), direct (gemv_cs.cuh; 16- or 8-byte global loads), general.
#pragma once
#include "gemv_cs.cuh"
#include "gemv_tma.cuh"
#include "launch.h"

namespace qg {


__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_codes));
    float a, b;
    asm("{.reg .f16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi;}"
        : "=f"(a), "=f"(b) : "r"(h2));
    return make_float2(a, b);
}

template <class SC>
struct FmtFp8 {
    static constexpr int kElemsPerWord = 4;
    static constexpr int kPairsPerWord = 2;
    struct Params {
        const uint16_t *x;
        const uint8_t *w;
        const typename SC::T *scale_inv;
        int I, O, nbi;
    };
    struct ThreadConst { int ib; };  // 128-column block of the thread's unit
    typedef float Aux;

    __device__ static ThreadConst thread_const(const Params &, int u, int XU) {
        return ThreadConst{(u * XU) >> 7};
    }
    __device__ static const void *unit_ptr(const Params &p, int o, int u, int XU) {
        return p.w + (size_t)o * p.I + (size_t)u * XU;
    }
    __device__ static Aux unit_aux(const Params &p, int o, int, ThreadConst tc) {
        return SC::get(p.scale_inv, (size_t)(o >> 7) * p.nbi + tc.ib);
    }
    __device__ static Aux zero_aux() { return 0.f; }
    // the unit's block scale lies inside the [ceil(O/128), ceil(I/128)] array
    __device__ static bool aux_ok(const Params &p, int o, ThreadConst tc) {
        return tc.ib >= 0 && tc.ib < p.nbi && (o >> 7) < (p.O + 127) / 128;
    }

    // xs: natural element order, f32
    template <int XU>
    __device__ static void load_x(const Params &p, int s, int u, float (&xs)[XU], float &xsum) {
        xsum = 0.f;
#pragma unroll
        for (int k = 0; k < XU; ++k)
            xs[k] = u >= 0 ? bf16_bits_to_f32(p.x[(size_t)s * p.I + (size_t)u * XU + k]) : 0.f;
    }

    template <int S, int NW, int XU>
    __device__ static void accumulate(const Words<NW> &wd, Aux sc, const float (&xs)[S][XU],
                                      const float (&)[S], float *part) {
        float2 d[NW * 2];
#pragma unroll
        for (int wq = 0; wq < NW; ++wq) {
            d[2 * wq] = e4m3x2_to_f32x2(wd.w[wq]);
            d[2 * wq + 1] = e4m3x2_to_f32x2(wd.w[wq] >> 16);
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NW * 2; ++i)
                acc = __ffma2_rn(d[i], make_float2(xs[s][2 * i], xs[s][2 * i + 1]), acc);
            part[s] = fmaf(sc, acc.x + acc.y, part[s]);
        }
    }

    // ---- staged (TMA) kernel -------------------------------------------------
    struct TConst { uint32_t uoff; int ib; };   // unit byte offset, 128-column block
    struct StageConst { float sc; };            // the batch's block scale for that column block
    // routed experts: 16-byte aligned codes for the staged copies; the block
    // scales are read one at a time from global memory
    __device__ static bool expert_ok(const Params &, const void *w, const float *scales) {
        return w != nullptr && scales != nullptr && ((uintptr_t)w % 16 == 0) &&
               ((uintptr_t)scales % alignof(typename SC::T) == 0);
    }
    __device__ static Params with_expert(Params p, const void *w, const float *scales, size_t x_off) {
        p.w = static_cast<const uint8_t *>(w);
        p.scale_inv = reinterpret_cast<const typename SC::T *>(scales);
        p.x += x_off;
        return p;
    }

    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.I; }
    __device__ static uint32_t aux_row_bytes(const Params &) { return 0u; }
    __device__ static uint32_t seg_byte(const Params &, int u, int XU) { return (uint32_t)(u * XU); }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.w + (size_t)o * p.I + col;
    }
    __device__ static const void *a_src(const Params &, int) { return nullptr; }
    __device__ static TConst tconst(const Params &, int u, int XU, uint32_t seg_col) {
        return TConst{(uint32_t)(u * XU) - seg_col, (u * XU) >> 7};
    }
    // rows of a batch share one 128-row block (the batch size divides 128)
    __device__ static StageConst stage_const(const Params &p, int o0, TConst tc) {
        return StageConst{o0 < p.O ? SC::get(p.scale_inv, (size_t)(o0 >> 7) * p.nbi + tc.ib) : 0.f};
    }
    template <int NW>
    __device__ static Words<NW> lds_unit(uint32_t a) { return lds_at<NW, true>(a); }
    __device__ static float aux(uint32_t, uint32_t, TConst, StageConst sc) { return sc.sc; }

    // xp[i] = {x[2i], x[2i+1]} of the unit, widened from bf16 (16-byte vector loads)
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        xsum = 0.f;
#pragma unroll
        for (int v = 0; v < XU / 8; ++v) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (u >= 0) q = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + v);
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                xp[4 * v + i] = pack2(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xFFFF0000u));
        }
    }

    struct ThreadScale {};
    template <int U, int S, int NP>
    __device__ static ThreadScale prepare_x(uint64_t (&)[U][S][NP], float (&)[U][S]) { return ThreadScale{}; }

    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, float sc, const uint64_t (&xp)[S][NP],
                                      const float (&)[S], ThreadScale, float *part) {
        uint64_t d[NW * 2];
#pragma unroll
        for (int wq = 0; wq < NW; ++wq) {
            d[2 * wq] = decode_e4m3x2(wd.w[wq]);
            d[2 * wq + 1] = decode_e4m3x2(wd.w[wq] >> 16);
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            uint64_t acc = fmul2(d[0], xp[s][0]);
#pragma unroll
            for (int i = 1; i < NW * 2; ++i) ffma2(acc, d[i], xp[s][i]);
            const float2 a = unpack2(acc);
            part[s] = fmaf(sc, a.x + a.y, part[s]);
        }
    }
};

// ---------------------------------------------------------------------------
// General kernel: any shape and alignment.  One warp per row.
// ---------------------------------------------------------------------------
// One token: the products in fma.rn.f32.f16.  The e4m3 pair converts to an
// exact fp16 pair (one cvt); the bf16 activations are carried as fp16 pairs
// scaled by 2^A, A putting the thread's largest finite |x| in [2^14, 2^15)
// (bf16's 8-bit significand fits fp16's 11; values more than 2^29 below that
// maximum lose bits as fp16 subnormals, more than 2^40 below it become zero).  fp16 x fp16 products are exact in f32,
// so the sum differs from the f32 form only in rounding order; the 2^-A goes
// back with the block scale.  Three instructions per weight pair instead of
// four (cvt, two f16 -> f32 cvts, f32x2 FMA), and half the x registers.
template <class SC>
struct FmtFp8H : FmtFp8<SC> {
    typedef typename FmtFp8<SC>::Params Params;
    static constexpr int kPairsPerWord = 1;     // one 64-bit register = two fp16 pairs per word

    // raw bf16 pairs in memory order: xp[w] = (x[4w], x[4w+1]) | (x[4w+2], x[4w+3]) << 32
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        static_assert(NP == XU / 4, "four activations per 64-bit register");
        xsum = 0.f;
#pragma unroll
        for (int v = 0; v < XU / 8; ++v) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (u >= 0) q = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + v);
            xp[2 * v] = (uint64_t)q.x | ((uint64_t)q.y << 32);
            xp[2 * v + 1] = (uint64_t)q.z | ((uint64_t)q.w << 32);
        }
    }

    typedef Pow2Pair ThreadScale;   // 2^-A as two factors

    __device__ static uint32_t bf16x2_to_scaled_f16x2(uint32_t b, float k1, float k2) {
        const float lo = __uint_as_float(b << 16) * k1 * k2, hi = __uint_as_float(b & 0xFFFF0000u) * k1 * k2;
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }

    template <int U, int S, int NP>
    __device__ static ThreadScale prepare_x(uint64_t (&xp)[U][S][NP], float (&)[U][S]) {
        uint32_t m = 0;   // largest finite |x| as a bf16 magnitude pattern
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int s = 0; s < S; ++s)
#pragma unroll
                for (int i = 0; i < NP; ++i)
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint32_t v = (uint32_t)(xp[j][s][i] >> (16 * h)) & 0x7FFFu;
                        if (v < 0x7F80u && v > m) m = v;
                    }
        int F = (int)(m >> 7);
        if (F < 1) F = 1;
        const int A = 141 - F;                       // in [-113, 140]
        const float k1 = pow2i(A >> 1), k2 = pow2i(A - (A >> 1));
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int s = 0; s < S; ++s)
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const uint32_t lo = (uint32_t)xp[j][s][i], hi = (uint32_t)(xp[j][s][i] >> 32);
                    xp[j][s][i] = (uint64_t)bf16x2_to_scaled_f16x2(lo, k1, k2) |
                                  ((uint64_t)bf16x2_to_scaled_f16x2(hi, k1, k2) << 32);
                }
        const int c = -A;
        return Pow2Pair{pow2i(c >> 1), pow2i(c - (c >> 1))};
    }

    __device__ static uint32_t e4m3x2_to_f16x2(uint32_t two) {
        uint32_t h;
        asm("{.reg .b16 lo, hi;\n\t"
            "mov.b32 {lo, hi}, %1;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, lo;}" : "=r"(h) : "r"(two));
        return h;
    }

    __device__ static void fma_mixed2(float &a0, float &a1, uint32_t w2, uint32_t x2) {
        asm("{.reg .f16 wl, wh, xl, xh;\n\t"
            "mov.b32 {wl, wh}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
            "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(w2), "r"(x2));
    }

    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, float sc, const uint64_t (&xp)[S][NP],
                                      const float (&)[S], ThreadScale ts, float *part) {
        uint32_t h[NW][2];
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            h[w][0] = e4m3x2_to_f16x2(wd.w[w]);
            h[w][1] = e4m3x2_to_f16x2(wd.w[w] >> 16);
        }
        const float scs = sc * ts.p1;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                fma_mixed2(a0, a1, h[w][0], (uint32_t)xp[s][w]);
                fma_mixed2(a0, a1, h[w][1], (uint32_t)(xp[s][w] >> 32));
            }
            part[s] = fmaf(scs, (a0 + a1) * ts.p2, part[s]);
        }
    }
};

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    return e4m3x2_to_f32x2((uint32_t)c).x;
}

template <class SC, int S>
__global__ void __launch_bounds__(256)
gemv_fp8_general_kernel(float *__restrict__ y, const uint16_t *__restrict__ x, const uint8_t *__restrict__ w,
                        const typename SC::T *__restrict__ scale_inv, int I, int O) {
    const int lane = threadIdx.x & 31;
    const int nbi = (I + 127) / 128;
    for (int o = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); o < O;
         o += gridDim.x * (blockDim.x >> 5)) {
        float acc[S];
#pragma unroll
        for (int s = 0; s < S; ++s) acc[s] = 0.f;
        const uint8_t *wr = w + (size_t)o * I;
        const size_t sb = (size_t)(o >> 7) * nbi;
        for (int i = lane; i < I; i += 32) {
            const float wv = e4m3_to_f32(wr[i]) * SC::get(scale_inv, sb + (i >> 7));
#pragma unroll
            for (int s = 0; s < S; ++s) acc[s] = fmaf(wv, bf16_bits_to_f32(x[(size_t)s * I + i]), acc[s]);
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const float t = warp_sum(acc[s]);
            if (lane == 0) y[(size_t)s * O + o] = t;
        }
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
namespace fp8 {

inline int fp8_nw(int S) { return S <= 4 ? 4 : 2; }       // activation registers 4*NW*S <= 64
inline int fp8_rb(int S, int U) { return S <= 2 ? (U == 1 ? 8 : 4) : 4; }

inline bool fp8_fast_ok(const uint16_t *x, const uint8_t *w, int I, int S) {
    const int nw = fp8_nw(S);
    return (I % (4 * nw) == 0) && ((uintptr_t)w % (4 * nw) == 0) && ((uintptr_t)x % 2 == 0);
}


inline bool fp8_tma_ok(const uint16_t *x, const uint8_t *w, int I, int S) {
    return fp8_fast_ok(x, w, I, S) && (I % 16 == 0) && ((uintptr_t)w % 16 == 0) && ((uintptr_t)x % 16 == 0);
}

inline bool fp8_tma_plan(int S, int I, int O, TmaPlan *pl) {
    const int nw = fp8_nw(S);
    TmaGeom g;
    g.units = I / (4 * nw);
    g.granule = 4 / nw;                          // 16 bytes of weights
    g.rowbytes = (uint32_t)I;
    g.granule_bytes = 16;
    g.arowbytes = 0;
    return tma_plan_rows(g, S, O, S == 1 ? 3 : 1, pl);
}

inline CsPlan fp8_plan(int S, int I, int O, int *U_out) {
    const int nw = fp8_nw(S);
    const int units = I / (4 * nw);
    // up to three units per thread at S = 1 (at S > 1 more than one spills
    // registers); longer rows split across blocks
    const int U = S == 1 ? (units > 2 * kCsMaxThreads ? 3 : units > kCsMaxThreads ? 2 : 1) : 1;
    *U_out = U;
    const int regs = 40 + 4 * nw * S * U + fp8_rb(S, U) * U * (nw + 1) + 2 * fp8_rb(S, U) * S;
    return cs_plan(units, O, U, fp8_rb(S, U), regs);
}

template <class SC, int S, int NW, int U>
void launch_cs_fp8(const typename FmtFp8<SC>::Params &p, float *out, const CsPlan &pl, int units, cudaStream_t st) {
    constexpr int RB = S <= 2 ? (U == 1 ? 8 : 4) : 4;
    dim3 grid(pl.grid_x, pl.splits);
    gemv_cs_kernel<FmtFp8<SC>, S, NW, U, RB><<<grid, pl.threads, 0, st>>>(p, out, units, pl.units_per_split,
                                                                         pl.nrowb, device_error_word());
    count_launch();
}

template <class SC, int S>
void launch_cs_fp8_s(const typename FmtFp8<SC>::Params &p, float *out, const CsPlan &pl, int units, int U,
                     cudaStream_t st) {
    constexpr int NW = S <= 4 ? 4 : 2;
    if constexpr (S == 1) {
        if (U == 2) {
            launch_cs_fp8<SC, S, NW, 2>(p, out, pl, units, st);
            return;
        }
        if (U == 3) {
            launch_cs_fp8<SC, S, NW, 3>(p, out, pl, units, st);
            return;
        }
    }
    (void)U;
    launch_cs_fp8<SC, S, NW, 1>(p, out, pl, units, st);
}

template <class SC, int S, int RB>
void launch_tma_fp8_u(const typename FmtFp8<SC>::Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    constexpr int NW = S <= 4 ? 4 : 2;
    if constexpr (S == 1) {
        if (pl.U == 2) {
            launch_tma<FmtFp8H<SC>, S, NW, 2, RB>(p, out, pl, st, moe);
            return;
        }
        if (pl.U == 3) {
            launch_tma<FmtFp8H<SC>, S, NW, 3, RB>(p, out, pl, st, moe);
            return;
        }
        launch_tma<FmtFp8H<SC>, S, NW, 1, RB>(p, out, pl, st, moe);
    } else {
        launch_tma<FmtFp8<SC>, S, NW, 1, RB>(p, out, pl, st, moe);
    }
}

template <class SC, int S>
void launch_tma_fp8_s(const typename FmtFp8<SC>::Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    if constexpr (S <= 2) {
        if (pl.rb == 8) {
            launch_tma_fp8_u<SC, S, 8>(p, out, pl, st, moe);
            return;
        }
    }
    if (pl.rb == 2) {
        if constexpr (S == 1) launch_tma<FmtFp8H<SC>, S, 4, 1, 2>(p, out, pl, st, moe);
        else launch_tma<FmtFp8<SC>, S, (S <= 4 ? 4 : 2), 1, 2>(p, out, pl, st, moe);
        return;
    }
    launch_tma_fp8_u<SC, S, 4>(p, out, pl, st, moe);
}

template <class SC>
int gemv_fp8_chunk(float *y, const uint16_t *x, const uint8_t *w, const typename SC::T *scale_inv, int S, int I,
                   int O, void *ws, size_t ws_bytes, cudaStream_t st, const char *name) {
    typename FmtFp8<SC>::Params p;
    p.x = x; p.w = w; p.scale_inv = scale_inv; p.I = I; p.O = O; p.nbi = (I + 127) / 128;

    TmaPlan tp;
    if (fp8_tma_ok(x, w, I, S) && fp8_tma_plan(S, I, O, &tp)) {
        const size_t need = tp.splits > 1 ? (size_t)tp.splits * S * O * sizeof(float) : 0;
        if (need > 0 && (ws == nullptr || ws_bytes < need)) {
            set_error_detail("%s: this shape splits the reduction and needs %zu bytes of "
                             "workspace (got %zu)", name, need, ws == nullptr ? (size_t)0 : ws_bytes);
            return kEWorkspace;
        }
        float *out = tp.splits > 1 ? static_cast<float *>(ws) : y;
        switch (S) {
#define QG_CASE(SS) case SS: launch_tma_fp8_s<SC, SS>(p, out, tp, st); break;
            QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
        }
        if (tp.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), tp.splits, S, O, st);
        return check_launch(name);
    }

    if (!fp8_fast_ok(x, w, I, S)) {
        const int blocks_needed = (O + 7) / 8;
        const int cap = num_sms() * 16;
        const int grid = blocks_needed < cap ? blocks_needed : cap;
        switch (S) {
#define QG_CASE(SS) case SS: gemv_fp8_general_kernel<SC, SS><<<grid, 256, 0, st>>>(y, x, w, scale_inv, I, O); count_launch(); break;
            QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
        }
        return check_launch(name);
    }
    int U = 1;
    const CsPlan pl = fp8_plan(S, I, O, &U);
    const int units = I / (4 * fp8_nw(S));
    const size_t need = cs_ws_bytes(pl, S, O);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) {
        set_error_detail("%s: this shape splits the reduction and needs %zu bytes of "
                         "workspace (got %zu)", name, need, ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    float *out = pl.splits > 1 ? static_cast<float *>(ws) : y;
    switch (S) {
#define QG_CASE(SS) case SS: launch_cs_fp8_s<SC, SS>(p, out, pl, units, U, st); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    if (pl.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), pl.splits, S, O, st);
    return check_launch(name);
}

}  // namespace fp8
using namespace fp8;

inline size_t ws_fp8(int S, int I, int O) {
    const int s = S < 8 ? S : 8;
    if (I % (4 * fp8_nw(s)) != 0) return 0;
    // the larger of the staged and the direct plan (the pointers decide the path)
    size_t need = 0;
    TmaPlan tp;
    if (I % 16 == 0 && fp8_tma_plan(s, I, O, &tp) && tp.splits > 1) need = (size_t)tp.splits * s * O * sizeof(float);
    int U = 1;
    const size_t cs = cs_ws_bytes(fp8_plan(s, I, O, &U), s, O);
    return need > cs ? need : cs;
}

template <class SC>
int run_gemv_fp8(float *y, const uint16_t *x, const uint8_t *w, const typename SC::T *scale_inv, int S, int I,
                 int O, void *ws, size_t ws_bytes, cudaStream_t st, const char *name) {
    for (int s0 = 0; s0 < S; s0 += 8) {
        const int sc = S - s0 < 8 ? S - s0 : 8;
        const int rc = gemv_fp8_chunk<SC>(y + (size_t)s0 * O, x + (size_t)s0 * I, w, scale_inv, sc, I, O, ws,
                                          ws_bytes, st, name);
        if (rc != kOk) return rc;
    }
    return kOk;
}


// Routed experts (fmt=7): every slot on the staged kernel, one launch.
template <class SC>
int run_gemv_moe_fp8(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                         const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    const uint8_t *probe = reinterpret_cast<const uint8_t *>(uintptr_t(256));   // stands for any 16-byte aligned expert
    TmaPlan tp;
    if (!fp8_tma_ok(x, probe, I, S) || !fp8_tma_plan(S, I, moe_plan_rows(O, n_slots), &tp) || tp.splits != 1) {
        set_error_detail("qgemv_moe: fmt=7 routed experts need I %% 16 == 0, a 16-byte aligned x and rows "
                         "short enough for one block (I = %d)", I);
        return kEShape;
    }
    typename FmtFp8<SC>::Params p;
    p.x = x; p.w = nullptr; p.scale_inv = nullptr; p.I = I; p.O = O; p.nbi = (I + 127) / 128;
    tp.nrowb = (O + tp.rb - 1) / tp.rb;            // the plan sized the launch for all slots' rows
    const MoeLaunch m{MoeSlots{static_cast<const ExpertW *>(table), ids, n_experts, x_stride}, n_slots};
    switch (S) {
#define QG_CASE(SS) case SS: launch_tma_fp8_s<SC, SS>(p, y, tp, st, &m); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    return check_launch("qgemv_moe");
}

}  // namespace qg
