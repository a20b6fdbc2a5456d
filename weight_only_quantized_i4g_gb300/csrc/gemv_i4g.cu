// gemv_i4g.cu -- fmt=4 grouped-int4 decode GEMV.
//
// Format (colibri PR #457, sections 3 and 11): row-major packed nibbles, row o
// is (I+1)/2 bytes; element i is in byte i/2, low nibble for even i; the
// stored nibble n means n - 8; f32 scales [O, ceil(I/gs)], one per gs
// consecutive elements of a row, applied to every term of its group:
//     y[s,o] = sum_i (n(o,i) - 8) * scale[o, i/gs] * x[s,i]
//
// A thread's unit is 4*NW bytes = 8*NW consecutive elements inside one group
// (gs % (8*NW) == 0), so one scale multiplies the unit's partial sum.
// Decode: for a 32-bit word of 8 nibbles, OR-ing a masked nibble into the bit
// pattern of 2^23 gives the float 2^23 + n*16^p exactly (p = position of the
// nibble in its 16-bit half); subtracting 2^23 + 8*16^p (exact) leaves
// (n - 8)*16^p, and the matching activation is pre-scaled by 16^-p (exact).
// Two elements at a time with packed f32x2 add and fma.
//
// Paths, fastest first:
//   mma      gemv_mma.cuh: nibbles as fp16 operands of the warp-level MMA,
//            f32 activations as an fp16 high and low part (two MMA columns
//            per token, four tokens per launch); needs 16-byte aligned w, x
//            and scales, I % 64 == 0, gs 64 or 128 and ceil(I/gs) % 4 == 0
//   staged   gemv_tma.cuh: bulk copies of whole rows (and their scales) into
//            a shared-memory ring; needs 16-byte aligned w, x and scales,
//            I % 32 == 0, gs a multiple of the unit and ceil(I/gs) % 4 == 0
//   direct   gemv_cs.cuh: the same decode with 16-, 8- or 4-byte global loads
//   general  any shape and alignment, byte loads
#include "gemv_cs.cuh"
#include "gemv_mma.cuh"
#include "gemv_tma.cuh"
#include "launch.h"

namespace qg {

struct FmtI4G {
    static constexpr int kElemsPerWord = 8;
    static constexpr int kPairsPerWord = 4;
    struct Params {
        const float *x;
        const uint8_t *w;
        const float *scales;
        int I, O, gs, ng;
        size_t rb;
    };
    // ---- direct (column-stationary) kernel ---------------------------------
    struct ThreadConst { int g; };   // group of the thread's unit
    typedef float Aux;               // the row's scale for that group

    __device__ static ThreadConst thread_const(const Params &p, int u, int XU) {
        return ThreadConst{(u * XU) / p.gs};
    }
    __device__ static const void *unit_ptr(const Params &p, int o, int u, int XU) {
        return p.w + (size_t)o * p.rb + (size_t)u * (XU / 2);
    }
    __device__ static Aux unit_aux(const Params &p, int o, int /*u*/, ThreadConst tc) {
        return ld_nc_f32(p.scales + (size_t)o * p.ng + tc.g);
    }
    __device__ static Aux zero_aux() { return 0.f; }
    // the unit's group scale lies inside the row's scales (bounds-checking build)
    __device__ static bool aux_ok(const Params &p, int, ThreadConst tc) { return tc.g >= 0 && tc.g < p.ng; }

    // xs layout: pair i = 4*w + q holds elements (8w + q, 8w + q + 4), both
    // scaled by 16^-q, at xs[2i], xs[2i+1].
    template <int XU>
    __device__ static void load_x(const Params &p, int s, int u, float (&xs)[XU], float &xsum) {
        xsum = 0.f;
#pragma unroll
        for (int wq = 0; wq < XU / 8; ++wq) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float sc = q == 0 ? 1.f : q == 1 ? 0.0625f : q == 2 ? 0.00390625f : 0.000244140625f;
                float a = 0.f, b = 0.f;
                if (u >= 0) {
                    const float *xp = p.x + (size_t)s * p.I + (size_t)u * XU + 8 * wq;
                    a = xp[q] * sc;
                    b = xp[q + 4] * sc;
                }
                xs[2 * (4 * wq + q)] = a;
                xs[2 * (4 * wq + q) + 1] = b;
            }
        }
    }

    template <int S, int NW, int XU>
    __device__ static void accumulate(const Words<NW> &wd, Aux sc, const float (&xs)[S][XU],
                                      const float (&)[S], float *part) {
        constexpr uint32_t kMagic = 0x4B000000u;   // 2^23
        float2 d[NW * 4];
#pragma unroll
        for (int wq = 0; wq < NW; ++wq) {
            const uint32_t lo = wd.w[wq];
            const uint32_t hi = lo >> 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t m = 0xFu << (4 * q);
                const float c = -(8388608.f + 8.f * (float)(1u << (4 * q)));
                float2 f = make_float2(__uint_as_float((lo & m) | kMagic), __uint_as_float((hi & m) | kMagic));
                d[4 * wq + q] = __fadd2_rn(f, make_float2(c, c));
            }
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NW * 4; ++i)
                acc = __ffma2_rn(d[i], make_float2(xs[s][2 * i], xs[s][2 * i + 1]), acc);
            part[s] = fmaf(sc, acc.x + acc.y, part[s]);
        }
    }

    // ---- staged (TMA) kernel -------------------------------------------------
    struct TConst { uint32_t uoff; uint32_t goff; };   // unit byte offset, scale byte offset
    struct StageConst {};
    // routed experts: the staged copies want both arrays 16-byte aligned
    __device__ static bool expert_ok(const Params &, const void *w, const float *scales) {
        return w != nullptr && scales != nullptr && ((uintptr_t)w % 16 == 0) && ((uintptr_t)scales % 16 == 0);
    }
    __device__ static Params with_expert(Params p, const void *w, const float *scales, size_t x_off) {
        p.w = static_cast<const uint8_t *>(w);
        p.scales = scales;
        p.x += x_off;
        return p;
    }

    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.rb; }
    __device__ static uint32_t aux_row_bytes(const Params &p) { return (uint32_t)p.ng * 4u; }
    __device__ static uint32_t seg_byte(const Params &, int u, int XU) { return (uint32_t)(u * (XU / 2)); }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.w + (size_t)o * p.rb + col;
    }
    __device__ static const void *a_src(const Params &p, int o) { return p.scales + (size_t)o * p.ng; }
    __device__ static TConst tconst(const Params &p, int u, int XU, uint32_t seg_col) {
        return TConst{(uint32_t)(u * (XU / 2)) - seg_col, 4u * (uint32_t)((u * XU) / p.gs)};
    }
    __device__ static StageConst stage_const(const Params &, int, TConst) { return StageConst{}; }
    template <int NW>
    __device__ static Words<NW> lds_unit(uint32_t a) { return lds_at<NW, true>(a); }
    __device__ static float aux(uint32_t, uint32_t row_a, TConst tc, StageConst) {
        return lds_f32_at(row_a + tc.goff);
    }


    // Activation pairs in the order nibbles_as_denormals produces weights:
    // for a word pair (2i, 2i+1) of the unit, xp[8i+q] = {x[16i+q], x[16i+8+q]}
    // and xp[8i+4+q] = {x[16i+4+q], x[16i+12+q]}; for a single-word unit
    // (NW = 1) xp[q] = {x[q], x[q+4]}.  Raw values here; prepare_x scales.
    // xsum = the unit's activation sum (the -8 offset of the nibbles).
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        float e[XU];
#pragma unroll
        for (int v = 0; v < XU / 4; ++v) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            if (u >= 0) a = __ldg(reinterpret_cast<const float4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + v);
            e[4 * v] = a.x; e[4 * v + 1] = a.y; e[4 * v + 2] = a.z; e[4 * v + 3] = a.w;
        }
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < XU; ++k) sum += e[k];
        xsum = sum;
        if constexpr (XU == 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q) xp[q] = pack2(e[q], e[q + 4]);
        } else {
#pragma unroll
            for (int i = 0; i < XU / 16; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    xp[8 * i + q] = pack2(e[16 * i + q], e[16 * i + 8 + q]);
                    xp[8 * i + 4 + q] = pack2(e[16 * i + 4 + q], e[16 * i + 12 + q]);
                }
        }
    }

    typedef Pow2Pair ThreadScale;
    template <int U, int S, int NP>
    __device__ static ThreadScale prepare_x(uint64_t (&xp)[U][S][NP], float (&)[U][S]) {
        return prescale_for_denormals<U, S, NP>(xp);
    }

    // sum (n - 8) * x over the unit = 2^c * sum(n * x * 2^-c) - 8 * xsum
    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, float sc, const uint64_t (&xp)[S][NP],
                                      const float (&xsum)[S], ThreadScale ts, float *part) {
        uint64_t d[NP];
        if constexpr (NW == 1) {
            const uint64_t ab = pack2(__uint_as_float(wd.w[0]), __uint_as_float(wd.w[0] >> 16));
#pragma unroll
            for (int q = 0; q < 4; ++q) d[q] = ab & ((uint64_t)(0xFu << (4 * q)) * 0x0000000100000001ull);
        } else {
#pragma unroll
            for (int i = 0; i < NW / 2; ++i) {
                uint64_t di[8];
                nibbles_as_denormals(((uint64_t)wd.w[2 * i + 1] << 32) | wd.w[2 * i], di);
#pragma unroll
                for (int k = 0; k < 8; ++k) d[8 * i + k] = di[k];
            }
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            uint64_t acc = fmul2(d[0], xp[s][0]);
#pragma unroll
            for (int i = 1; i < NP; ++i) ffma2(acc, d[i], xp[s][i]);
            const float2 u = unpack2(acc);
            const float t = fmaf((u.x + u.y) * ts.p1, ts.p2, -8.f * xsum[s]);
            part[s] = fmaf(sc, t, part[s]);
        }
    }
};

// Warp-MMA decode (gemv_mma.cuh).  A scale unit is one 64-weight span, which
// lies inside one group (gs = 64 or 128).  The C operand starts every unit's
// sum at -8 sum(x), so D = sum((n - 8) x) and acc += scale * D.  Each token
// takes two MMA columns: x = high + low, both fp16 (x * 2^k rounded to fp16,
// and the rounding remainder rounded to fp16), which keeps 22 significant
// bits of the f32 activation.
template <int LG>   // gs = 64 << LG
struct MmaI4G {
    static constexpr bool kHiLo = true;
    static constexpr bool kNeg8 = true;
    static constexpr int kSpansPerUnit = 1;
    static constexpr bool kFenceUnits = true;
    static constexpr int kMaxConsumerWarps = 14;   // 7168 columns; 136 registers a thread
    static constexpr int kRedStride = 4;           // four tokens per launch
    typedef FmtI4G::Params Params;
    typedef float Side;
    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.rb; }
    __device__ static uint32_t aux_row_bytes(const Params &p) { return (uint32_t)p.ng * 4u; }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) { return p.w + (size_t)o * p.rb + col; }
    __device__ static const void *a_src(const Params &p, int o) { return p.scales + (size_t)o * p.ng; }
    __host__ __device__ static uint32_t span_byte(int sp) { return 32u * (uint32_t)sp; }
    __device__ static uint32_t span_off(int sp_local) { return 32u * (uint32_t)sp_local; }
    static constexpr int kXWords = 8;   // eight f32 activations
    __device__ static const void *x_src(const Params &p, int tok, int col) { return p.x + (size_t)tok * p.I + col; }
    __device__ static float abs_max8(const uint32_t (&w)[8]) {
        float m = fabsf(__uint_as_float(w[0]));
#pragma unroll
        for (int e = 1; e < 8; ++e) m = fmaxf(m, fabsf(__uint_as_float(w[e])));
        return m;
    }
    __device__ static uint64_t pair(const uint32_t (&w)[8], int i) {
        return (uint64_t)w[2 * i] | ((uint64_t)w[2 * i + 1] << 32);
    }
    // byte offset of unit u's group scale in the staged scale row (a group
    // is 2^LG spans; the warp's first span is a multiple of 8)
    __device__ static uint32_t side_off(int sp_abs0, int, int u) {
        return ((uint32_t)(sp_abs0 >> LG) + (uint32_t)(u >> LG)) << 2;
    }
    __device__ static Side side(uint32_t, uint32_t row_a, uint32_t off) { return lds_f32_at(row_a + off); }
    __device__ static void apply(float (&acc)[4], const float (&d)[4], Side s0, Side s1, const float (&)[2]) {
        acc[0] = fmaf(s0, d[0], acc[0]);
        acc[1] = fmaf(s0, d[1], acc[1]);
        acc[2] = fmaf(s1, d[2], acc[2]);
        acc[3] = fmaf(s1, d[3], acc[3]);
    }
};

// ---------------------------------------------------------------------------
// General kernel: any I, any even gs, any alignment.  One warp per row; lanes
// walk the elements; byte loads.
// ---------------------------------------------------------------------------
template <int S>
__global__ void __launch_bounds__(256)
gemv_i4g_general_kernel(float *__restrict__ y, const float *__restrict__ x, const uint8_t *__restrict__ w,
                        const float *__restrict__ scales, int I, int O, int gs) {
    const int lane = threadIdx.x & 31;
    const size_t rb = ((size_t)I + 1) / 2;
    const int ng = (I + gs - 1) / gs;
    for (int o = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); o < O;
         o += gridDim.x * (blockDim.x >> 5)) {
        float acc[S];
#pragma unroll
        for (int s = 0; s < S; ++s) acc[s] = 0.f;
        const uint8_t *wr = w + (size_t)o * rb;
        const float *sr = scales + (size_t)o * ng;
        for (int i = lane; i < I; i += 32) {
            const uint8_t b = wr[i >> 1];
            const int q = (int)((i & 1) ? (b >> 4) : (b & 0xF)) - 8;
            const float wv = (float)q * sr[i / gs];
#pragma unroll
            for (int s = 0; s < S; ++s) acc[s] = fmaf(wv, x[(size_t)s * I + i], acc[s]);
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
namespace {

// words per unit for S tokens: keep the activation registers (8*NW*S) <= 64;
// at one or two tokens 8-byte units (16 weights) rather than 16-byte ones:
// twice the threads share the decode that follows the activation load, which
// is what a call on a matrix of a few MB waits for (measured on GB300:
// 2048x7168 4.38 -> 4.03 us, 7168x2048 4.33 -> 3.99 us)
int i4g_nw(int S) { return S <= 4 ? 2 : 1; }
int i4g_rb(int S, int U) { return S <= 2 ? (U == 1 ? 8 : 4) : 4; }

bool i4g_fast_ok(const float *x, const uint8_t *w, int I, int gs, int S) {
    const int nw = i4g_nw(S);
    const int ue = 8 * nw;                       // elements per unit
    return (I % ue == 0) && (gs % ue == 0) && ((uintptr_t)w % (4 * nw) == 0) &&
           ((uintptr_t)x % 4 == 0);
}

bool i4g_tma_ok(const float *x, const uint8_t *w, const float *scales, int I, int gs, int S) {
    const int ng = (I + gs - 1) / gs;
    return i4g_fast_ok(x, w, I, gs, S) && (I % 32 == 0) && (ng % 4 == 0) && ((uintptr_t)w % 16 == 0) &&
           ((uintptr_t)x % 16 == 0) && ((uintptr_t)scales % 16 == 0);
}

bool i4g_mma_ok(const float *x, const uint8_t *w, const float *scales, int I, int gs) {
    const int ng = (I + gs - 1) / gs;
    return (I % 64 == 0) && (gs == 64 || gs == 128) && (ng % 4 == 0) && ((uintptr_t)w % 16 == 0) &&
           ((uintptr_t)x % 16 == 0) && ((uintptr_t)scales % 16 == 0);
}

// S <= 4 tokens per launch (two MMA columns each)
bool i4g_mma_plan(int S, int I, int O, int gs, MmaPlan *pl) {
    return mma_plan(I / 64, 8, (uint32_t)(I / 2), (uint32_t)((I + gs - 1) / gs) * 4u, 4u, S, O, 16,
                    MmaI4G<0>::kMaxConsumerWarps, MmaI4G<0>::kRedStride, [](int sp) { return 32u * (uint32_t)sp; },
                    pl);
}

bool i4g_tma_plan(int S, int I, int O, int gs, TmaPlan *pl) {
    const int nw = i4g_nw(S);
    TmaGeom g;
    g.units = I / (8 * nw);
    g.granule = 4 / nw;                          // 16 bytes of weights
    g.rowbytes = (uint32_t)(I / 2);
    g.granule_bytes = 16;
    g.arowbytes = (uint32_t)((I + gs - 1) / gs) * 4u;
    return tma_plan_rows(g, S, O, S == 1 ? 2 : 1, pl);
}

CsPlan i4g_plan(int S, int I, int O, int *U_out) {
    const int nw = i4g_nw(S);
    const int units = I / (8 * nw);
    // up to two units per thread at S = 1 (more, or more than one at S > 1,
    // spills registers); longer rows split across blocks
    const int U = (S == 1 && units > kCsMaxThreads) ? 2 : 1;
    *U_out = U;
    const int regs = 40 + 8 * nw * S * U + i4g_rb(S, U) * U * (nw + 1) + 2 * i4g_rb(S, U) * S;
    return cs_plan(units, O, U, i4g_rb(S, U), regs);
}

template <int S, int NW, int U>
void launch_cs_i4g(const FmtI4G::Params &p, float *out, const CsPlan &pl, int units, cudaStream_t st) {
    constexpr int RB = S <= 2 ? (U == 1 ? 8 : 4) : 4;
    dim3 grid(pl.grid_x, pl.splits);
    gemv_cs_kernel<FmtI4G, S, NW, U, RB><<<grid, pl.threads, 0, st>>>(p, out, units, pl.units_per_split,
                                                                     pl.nrowb, device_error_word());
    count_launch();
}

template <int S>
void launch_cs_i4g_s(const FmtI4G::Params &p, float *out, const CsPlan &pl, int units, int U, cudaStream_t st) {
    constexpr int NW = S <= 4 ? 2 : 1;
    if constexpr (S == 1) {
        if (U == 2) {
            launch_cs_i4g<S, NW, 2>(p, out, pl, units, st);
            return;
        }
    }
    (void)U;
    launch_cs_i4g<S, NW, 1>(p, out, pl, units, st);
}

template <int S, int RB>
void launch_tma_i4g_u(const FmtI4G::Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    constexpr int NW = S <= 4 ? 2 : 1;
    if constexpr (S == 1) {
        if (pl.U == 2) {
            launch_tma<FmtI4G, S, NW, 2, RB>(p, out, pl, st, moe);
            return;
        }
    }
    launch_tma<FmtI4G, S, NW, 1, RB>(p, out, pl, st, moe);
}

template <int S>
void launch_tma_i4g_s(const FmtI4G::Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    if constexpr (S <= 2) {
        if (pl.rb == 8) {
            launch_tma_i4g_u<S, 8>(p, out, pl, st, moe);
            return;
        }
    }
    if (pl.rb == 2) {
        launch_tma<FmtI4G, S, (S <= 4 ? 2 : 1), 1, 2>(p, out, pl, st, moe);
        return;
    }
    launch_tma_i4g_u<S, 4>(p, out, pl, st, moe);
}

int gemv_i4g_chunk(float *y, const float *x, const uint8_t *w, const float *scales, int S, int I, int O,
                   int gs, void *ws, size_t ws_bytes, cudaStream_t st) {
    FmtI4G::Params p;
    p.x = x; p.w = w; p.scales = scales; p.I = I; p.O = O; p.gs = gs;
    p.ng = (I + gs - 1) / gs; p.rb = ((size_t)I + 1) / 2;

    TmaPlan tp;
    if (i4g_tma_ok(x, w, scales, I, gs, S) && i4g_tma_plan(S, I, O, gs, &tp)) {
        const size_t need = tp.splits > 1 ? (size_t)tp.splits * S * O * sizeof(float) : 0;
        if (need > 0 && (ws == nullptr || ws_bytes < need)) {
            set_error_detail("qgemv_i4g: this shape splits the reduction and needs %zu bytes of workspace "
                             "(got %zu)", need, ws == nullptr ? (size_t)0 : ws_bytes);
            return kEWorkspace;
        }
        float *out = tp.splits > 1 ? static_cast<float *>(ws) : y;
        switch (S) {
#define QG_CASE(SS) case SS: launch_tma_i4g_s<SS>(p, out, tp, st); break;
            QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
        }
        if (tp.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), tp.splits, S, O, st);
        return check_launch("qgemv_i4g");
    }

    if (!i4g_fast_ok(x, w, I, gs, S)) {
        const int blocks_needed = (O + 7) / 8;
        const int cap = num_sms() * 16;
        const int grid = blocks_needed < cap ? blocks_needed : cap;
        switch (S) {
#define QG_CASE(SS) case SS: gemv_i4g_general_kernel<SS><<<grid, 256, 0, st>>>(y, x, w, scales, I, O, gs); count_launch(); break;
            QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
        }
        return check_launch("qgemv_i4g (general kernel)");
    }
    int U = 1;
    const CsPlan pl = i4g_plan(S, I, O, &U);
    const int units = I / (8 * i4g_nw(S));
    const size_t need = cs_ws_bytes(pl, S, O);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) {
        set_error_detail("qgemv_i4g: this shape splits the reduction and needs %zu bytes of workspace "
                         "(got %zu)", need, ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    float *out = pl.splits > 1 ? static_cast<float *>(ws) : y;
    switch (S) {
#define QG_CASE(SS) case SS: launch_cs_i4g_s<SS>(p, out, pl, units, U, st); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    if (pl.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), pl.splits, S, O, st);
    return check_launch("qgemv_i4g");
}

}  // namespace

// The fmt=4 decode planners above, exported (host code) for the test suite's
// checks of the shared-memory layouts they choose over a sweep of shapes.
bool plan_i4g_mma(int S, int I, int O, int gs, MmaPlan *pl) { return i4g_mma_plan(S, I, O, gs, pl); }
bool plan_i4g_tma(int S, int I, int O, int gs, TmaPlan *pl) { return i4g_tma_plan(S, I, O, gs, pl); }

size_t ws_i4g(int S, int I, int O, int gs) {
    const int s = S < 8 ? S : 8;
    size_t mma_need = 0;
    MmaPlan mp;
    if (I % 64 == 0 && (gs == 64 || gs == 128) && ((I + gs - 1) / gs) % 4 == 0 &&
        i4g_mma_plan(s < 4 ? s : 4, I, O, gs, &mp) && mp.splits > 1)
        mma_need = (size_t)mp.splits * (s < 4 ? s : 4) * O * sizeof(float);
    if (I % (8 * i4g_nw(s)) != 0 || gs % (8 * i4g_nw(s)) != 0) return 0;  // general kernel: none
    // the larger of the staged and the direct plan (the pointers decide the path)
    size_t need = 0;
    TmaPlan tp;
    if (I % 32 == 0 && ((I + gs - 1) / gs) % 4 == 0 && i4g_tma_plan(s, I, O, gs, &tp) && tp.splits > 1)
        need = (size_t)tp.splits * s * O * sizeof(float);
    int U = 1;
    const size_t cs = cs_ws_bytes(i4g_plan(s, I, O, &U), s, O);
    return std::max(mma_need, need > cs ? need : cs);
}

int run_gemv_i4g(float *y, const float *x, const uint8_t *w, const float *scales, int S, int I, int O,
                 int gs, void *ws, size_t ws_bytes, cudaStream_t st) {
    // The warp-MMA kernel from two tokens on; at one token the staged kernel
    // is faster on the 8 MB decode shapes (measured on GB300: 2048x7168 4.3
    // against 5.8 us, 7168x2048 4.35 against 4.9).
    if (S > 1 && i4g_mma_ok(x, w, scales, I, gs)) {
        FmtI4G::Params p;
        p.w = w; p.scales = scales; p.I = I; p.O = O; p.gs = gs;
        p.ng = (I + gs - 1) / gs; p.rb = ((size_t)I + 1) / 2;
        for (int s0 = 0; s0 < S; s0 += 4) {
            const int sc = S - s0 < 4 ? S - s0 : 4;
            MmaPlan mp;
            if (!i4g_mma_plan(sc, I, O, gs, &mp)) break;   // the staged / direct paths below
            const size_t need = mp.splits > 1 ? (size_t)mp.splits * sc * O * sizeof(float) : 0;
            if (need > 0 && (ws == nullptr || ws_bytes < need)) {
                set_error_detail("qgemv_i4g: this shape splits the reduction and needs %zu bytes of workspace "
                                 "(got %zu)", need, ws == nullptr ? (size_t)0 : ws_bytes);
                return kEWorkspace;
            }
            p.x = x + (size_t)s0 * I;
            float *yc = y + (size_t)s0 * O;
            float *out = mp.splits > 1 ? static_cast<float *>(ws) : yc;
            if (gs == 64) launch_mma<MmaI4G<0>, kMmaSpansPerWarp, 16>(p, out, mp, st);
            else launch_mma<MmaI4G<1>, kMmaSpansPerWarp, 16>(p, out, mp, st);
            if (mp.splits > 1) launch_splitk_reduce(yc, static_cast<float *>(ws), mp.splits, sc, O, st);
            const int rc = check_launch("qgemv_i4g");
            if (rc != kOk) return rc;
            if (s0 + sc >= S) return kOk;
        }
    }
    for (int s0 = 0; s0 < S; s0 += 8) {
        const int sc = S - s0 < 8 ? S - s0 : 8;
        const int rc = gemv_i4g_chunk(y + (size_t)s0 * O, x + (size_t)s0 * I, w, scales, sc, I, O, gs, ws,
                                      ws_bytes, st);
        if (rc != kOk) return rc;
    }
    return kOk;
}


// Routed experts (fmt=4): every slot on the staged kernel, one launch.
int run_gemv_moe_i4g(float *y, const float *x, size_t x_stride, const void *table, int n_experts,
                     const int *ids, int n_slots, int S, int I, int O, int gs, cudaStream_t st) {
    const uint8_t *probe = reinterpret_cast<const uint8_t *>(uintptr_t(256));   // stands for any 16-byte aligned expert
    TmaPlan tp;
    if (!i4g_tma_ok(x, probe, reinterpret_cast<const float *>(probe), I, gs, S) ||
        !i4g_tma_plan(S, I, moe_plan_rows(O, n_slots), gs, &tp) || tp.splits != 1) {
        set_error_detail("qgemv_moe: fmt=4 routed experts need I %% 32 == 0, gs %% 32 == 0, ceil(I/gs) %% 4 == 0, "
                         "a 16-byte aligned x and rows short enough for one block (I = %d, gs = %d)", I, gs);
        return kEShape;
    }
    FmtI4G::Params p;
    p.x = x; p.w = nullptr; p.scales = nullptr; p.I = I; p.O = O; p.gs = gs;
    p.ng = (I + gs - 1) / gs; p.rb = ((size_t)I + 1) / 2;
    tp.nrowb = (O + tp.rb - 1) / tp.rb;            // the plan sized the launch for all slots' rows
    const MoeLaunch m{MoeSlots{static_cast<const ExpertW *>(table), ids, n_experts, x_stride}, n_slots};
    switch (S) {
#define QG_CASE(SS) case SS: launch_tma_i4g_s<SS>(p, y, tp, st, &m); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    return check_launch("qgemv_moe");
}

}  // namespace qg
