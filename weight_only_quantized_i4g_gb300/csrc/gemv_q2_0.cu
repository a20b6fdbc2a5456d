// gemv_q2_0.cu -- decode GEMV for the Q2_0 codec (the ggml Q2_0 layout the
// strata review checks in "convert_k256_q2_0.cpp vs ref_quant.cpp", 2.5):
// 18 bytes per 64 weights, an fp16 d at bytes [0,2) and 2-bit codes at
// [2,18), weight e of the block in byte 2 + e/4 at bit 2*(e%4);
//     w_e = (code_e - 1) * d.
//
// Batch 1 with 16-byte aligned x and blocks and I % 512 == 0 (rows of whole
// 16-byte lines): the staged kernel (gemv_tma.cuh, FmtQ2T below).  Otherwise
// a direct column-stationary kernel (gemv_cs.cuh): a unit is 8 weights, the two
// code bytes 2 + 2h, 3 + 2h of a block (h = 0..7) -- blocks of 18 bytes keep
// units 2-byte aligned only, so a unit is one 16-bit load.  Per unit and
// token: sum_k code_k x_k in f32 (codes exact), then d * (that - sum_k x_k).
#include "gemv_cs.cuh"
#include "gemv_tma.cuh"
#include "launch.h"

namespace qg {

struct FmtQ2 {
    static constexpr int kElemsPerWord = 8;   // 8 codes in the low 16 bits of each loaded word
    struct Params {
        const uint16_t *x;
        const uint8_t *blocks;
        int I, O;
        size_t rowbytes;
    };
    struct ThreadConst { int uoff; int doff; };   // bytes of the unit's codes and of its block's d in a row
    typedef float Aux;                           // d of the unit's block

    __device__ static ThreadConst thread_const(const Params &, int u, int) {
        const int b = u >> 3, h = u & 7;
        return ThreadConst{18 * b + 2 + 2 * h, 18 * b};
    }
    __device__ static const void *unit_ptr(const Params &p, int o, int u, int) {
        return p.blocks + (size_t)o * p.rowbytes + 18 * (u >> 3) + 2 + 2 * (u & 7);
    }
    __device__ static Aux unit_aux(const Params &p, int o, int, ThreadConst tc) {
        uint16_t h;
        asm("ld.global.nc.u16 %0, [%1];" : "=h"(h) : "l"(p.blocks + (size_t)o * p.rowbytes + tc.doff));
        return f16_bits_to_f32(h);
    }
    __device__ static Aux zero_aux() { return 0.f; }
    // the unit's d lies inside the row (bounds-checking build)
    __device__ static bool aux_ok(const Params &p, int, ThreadConst tc) {
        return tc.doff >= 0 && (size_t)tc.doff + 2 <= p.rowbytes;
    }
    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.rowbytes; }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.blocks + (size_t)o * p.rowbytes + col;
    }
    template <int NW>
    __device__ static Words<NW> load_unit(const void *ptr) {
        static_assert(NW == 1, "a Q2_0 unit is one 16-bit load");
        uint16_t h;
        asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(h) : "l"(ptr));
        Words<NW> w;
        w.w[0] = h;
        return w;
    }
    template <int XU>
    __device__ static void load_x(const Params &p, int s, int u, float (&xs)[XU], float &xsum) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < XU; ++k) {
            xs[k] = u >= 0 ? bf16_bits_to_f32(p.x[(size_t)s * p.I + (size_t)u * XU + k]) : 0.f;
            sum += xs[k];
        }
        xsum = sum;
    }
    // part[s] += d * (sum_k code_k x_k - sum_k x_k)
    template <int S, int NW, int XU>
    __device__ static void accumulate(const Words<NW> &wd, Aux d, const float (&xs)[S][XU], const float (&xsum)[S],
                                      float *part) {
        float c[XU];
#pragma unroll
        for (int k = 0; k < XU; ++k) c[k] = (float)((wd.w[0] >> (2 * k)) & 3u);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float a = 0.f;
#pragma unroll
            for (int k = 0; k < XU; ++k) a = fmaf(c[k], xs[s][k], a);
            part[s] = fmaf(d, a - xsum[s], part[s]);
        }
    }
};

namespace {

// Staged path at one token.  A unit is 32 weights: the 8 code bytes of half a
// block (2-byte aligned in shared memory: four 16-bit loads make two words).
// In each 32-bit word (16 codes, byte j holding codes 4j..4j+3 at bits 0, 2,
// 4, 6) the masks 0x00030003 << 2k on the word and on the word shifted down by
// 8 leave pairs of codes (element e and e + 8 of the word, k = e % 4) as the
// fp16 subnormals code * 4^k * 2^-24 (exact); each multiplies, in
// fma.rn.f32.f16, its activations held as fp16 pairs pre-scaled by
// 2^(A - 2k), A putting the thread's largest |x| in [2^14, 2^15): every
// product is code * x * 2^(A - 24) exactly, accumulated in f32.  Then
// part += d * (2^(24 - A) * sum - sum_x).
struct FmtQ2T : FmtQ2 {
    static constexpr int kElemsPerWord = 16;
    static constexpr int kPairsPerWord = 4;    // four 64-bit registers = eight fp16 pairs per word
    struct TConst { uint32_t uoff; uint32_t doff; };
    struct StageConst {};
    typedef float Aux;

    __device__ static bool expert_ok(const Params &, const void *w, const float *) {
        return w != nullptr && ((uintptr_t)w % 16 == 0);
    }
    __device__ static Params with_expert(Params p, const void *w, const float *, size_t x_off) {
        p.blocks = static_cast<const uint8_t *>(w);
        p.x += x_off;
        return p;
    }
    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.rowbytes; }
    __device__ static uint32_t aux_row_bytes(const Params &) { return 0u; }
    // a segment starts at a granule of 8 blocks (144 bytes, whole 16-byte lines)
    __device__ static uint32_t seg_byte(const Params &, int u, int) { return 18u * (uint32_t)(u >> 1); }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.blocks + (size_t)o * p.rowbytes + col;
    }
    __device__ static const void *a_src(const Params &, int) { return nullptr; }
    __device__ static TConst tconst(const Params &, int u, int, uint32_t seg_col) {
        const uint32_t b = (uint32_t)(u >> 1), h = (uint32_t)(u & 1);
        return TConst{18u * b + 2u + 8u * h - seg_col, 18u * b - seg_col};
    }
    __device__ static StageConst stage_const(const Params &, int, TConst) { return StageConst{}; }
    template <int NW>
    __device__ static Words<NW> lds_unit(uint32_t a) {
        static_assert(NW == 2, "a staged Q2_0 unit is 8 code bytes");
        uint16_t h0, h1, h2, h3;
        asm volatile("ld.shared.u16 %0, [%4];\n\tld.shared.u16 %1, [%4+2];\n\t"
                     "ld.shared.u16 %2, [%4+4];\n\tld.shared.u16 %3, [%4+6];"
                     : "=h"(h0), "=h"(h1), "=h"(h2), "=h"(h3) : "r"(a));
        Words<NW> w;
        w.w[0] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        w.w[1] = (uint32_t)h2 | ((uint32_t)h3 << 16);
        return w;
    }
    __device__ static Aux aux(uint32_t row_w, uint32_t, TConst tc, StageConst) {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(row_w + tc.doff));
        return f16_bits_to_f32(h);
    }

    // Raw bf16 pairs in slot order: for word w of the unit, register 4w + q
    // holds pair e = 2q (low half) and e = 2q + 1 (high half), pair e being
    // (x[16w + e], x[16w + e + 8]); xsum = the unit's activation sum.
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        static_assert(XU == 32 && NP == 8, "32 weights per unit");
        uint32_t raw[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (u >= 0) q = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + v);
            raw[4 * v] = q.x; raw[4 * v + 1] = q.y; raw[4 * v + 2] = q.z; raw[4 * v + 3] = q.w;
        }
        auto bf = [&](int j) { return (raw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu; };
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) sum += __uint_as_float(bf(j) << 16);
        xsum = sum;
#pragma unroll
        for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e0 = 2 * q, e1 = 2 * q + 1;
                const uint32_t p0 = bf(16 * w + e0) | (bf(16 * w + e0 + 8) << 16);
                const uint32_t p1 = bf(16 * w + e1) | (bf(16 * w + e1 + 8) << 16);
                xp[4 * w + q] = (uint64_t)p0 | ((uint64_t)p1 << 32);
            }
    }

    typedef Pow2Pair ThreadScale;   // 2^(24 - A) as two factors

    __device__ static uint32_t bf16x2_scaled(uint32_t b, float k1, float k2) {
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
        const int A = 141 - F;                       // max |x| * 2^A < 2^15
        float k1[4], k2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int kk = A - 2 * k;                // in [-119, 140]
            k1[k] = pow2i(kk >> 1);
            k2[k] = pow2i(kk - (kk >> 1));
        }
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int s = 0; s < S; ++s)
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const int q = i & 3;             // pairs 2q (position 2(q%2)) and 2q + 1
                    const int klo = 2 * (q & 1), khi = klo + 1;
                    const uint32_t lo = (uint32_t)xp[j][s][i], hi = (uint32_t)(xp[j][s][i] >> 32);
                    xp[j][s][i] = (uint64_t)bf16x2_scaled(lo, k1[klo], k2[klo]) |
                                  ((uint64_t)bf16x2_scaled(hi, k1[khi], k2[khi]) << 32);
                }
        const int c = F - 117;                       // 24 - A
        return Pow2Pair{pow2i(c >> 1), pow2i(c - (c >> 1))};
    }

    __device__ static void fma_mixed2(float &a0, float &a1, uint32_t n2, uint32_t x2) {
        asm("{.reg .f16 nl, nh, xl, xh;\n\t"
            "mov.b32 {nl, nh}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.f16 %0, nl, xl, %0;\n\t"
            "fma.rn.f32.f16 %1, nh, xh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(n2), "r"(x2));
    }

    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, Aux d, const uint64_t (&xp)[S][NP],
                                      const float (&xsum)[S], ThreadScale ts, float *part) {
        uint32_t n[NW][8];
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const uint32_t v = wd.w[w] >> 8;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                n[w][k] = wd.w[w] & (0x00030003u << (2 * k));
                n[w][4 + k] = v & (0x00030003u << (2 * k));
            }
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t x2 = xp[s][4 * w + q];
                    fma_mixed2(a0, a1, n[w][2 * q], (uint32_t)x2);
                    fma_mixed2(a0, a1, n[w][2 * q + 1], (uint32_t)(x2 >> 32));
                }
            part[s] = fmaf(d, fmaf((a0 + a1) * ts.p1, ts.p2, -xsum[s]), part[s]);
        }
    }
};

bool q2_tma_plan(int I, int O, TmaPlan *pl) {
    TmaGeom g;
    g.units = I / 32;
    g.granule = 16;                              // 8 blocks = 144 bytes = 9 lines of 16
    g.rowbytes = (uint32_t)((I / 64) * 18);
    g.granule_bytes = 144;
    g.arowbytes = 0;
    return tma_plan_rows(g, 1, O, 3, pl);
}

bool q2_tma_ok(const uint16_t *x, const uint8_t *blocks, int I, int S) {
    return S == 1 && I % 512 == 0 && (uintptr_t)x % 16 == 0 && (uintptr_t)blocks % 16 == 0;
}

template <int RB>
void launch_tma_q2(const FmtQ2::Params &p, float *out, const TmaPlan &pl, cudaStream_t st) {
    if (pl.U == 2) return launch_tma<FmtQ2T, 1, 2, 2, RB>(p, out, pl, st);
    if (pl.U == 3) return launch_tma<FmtQ2T, 1, 2, 3, RB>(p, out, pl, st);
    launch_tma<FmtQ2T, 1, 2, 1, RB>(p, out, pl, st);
}

constexpr int q2_rb(int S) { return S <= 2 ? 8 : 4; }

CsPlan q2_plan(int S, int I, int O, int *U_out) {
    const int units = I / 8;
    const int U = S == 1 ? (units > 2 * kCsMaxThreads ? 3 : units > kCsMaxThreads ? 2 : 1) : 1;
    *U_out = U;
    const int regs = 40 + 8 * S * U + q2_rb(S) * U * 2 + 2 * q2_rb(S) * S;
    return cs_plan(units, O, U, q2_rb(S), regs);
}

template <int S, int U>
void launch_q2(const FmtQ2::Params &p, float *out, const CsPlan &pl, int units, cudaStream_t st) {
    dim3 grid(pl.grid_x, pl.splits);
    gemv_cs_kernel<FmtQ2, S, 1, U, q2_rb(S)><<<grid, pl.threads, 0, st>>>(p, out, units, pl.units_per_split,
                                                                         pl.nrowb, device_error_word());
    count_launch();
}

template <int S>
void launch_q2_s(const FmtQ2::Params &p, float *out, const CsPlan &pl, int units, int U, cudaStream_t st) {
    if constexpr (S == 1) {
        if (U == 2) return launch_q2<S, 2>(p, out, pl, units, st);
        if (U == 3) return launch_q2<S, 3>(p, out, pl, units, st);
    }
    (void)U;
    launch_q2<S, 1>(p, out, pl, units, st);
}

int gemv_q2_chunk(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                  size_t ws_bytes, cudaStream_t st) {
    FmtQ2::Params p;
    p.x = x; p.blocks = blocks; p.I = I; p.O = O; p.rowbytes = (size_t)(I / 64) * 18;
    TmaPlan tp;
    if (q2_tma_ok(x, blocks, I, S) && q2_tma_plan(I, O, &tp)) {
        const size_t need = tp.splits > 1 ? (size_t)tp.splits * O * sizeof(float) : 0;
        if (need > 0 && (ws == nullptr || ws_bytes < need)) {
            set_error_detail("qgemv_q2_0: this shape splits the reduction and needs %zu bytes of workspace "
                             "(got %zu)", need, ws == nullptr ? (size_t)0 : ws_bytes);
            return kEWorkspace;
        }
        float *out = tp.splits > 1 ? static_cast<float *>(ws) : y;
        if (tp.rb == 8) launch_tma_q2<8>(p, out, tp, st);
        else if (tp.rb == 4) launch_tma_q2<4>(p, out, tp, st);
        else launch_tma<FmtQ2T, 1, 2, 1, 2>(p, out, tp, st);
        if (tp.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), tp.splits, 1, O, st);
        return check_launch("qgemv_q2_0");
    }
    int U = 1;
    const CsPlan pl = q2_plan(S, I, O, &U);
    const size_t need = cs_ws_bytes(pl, S, O);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) {
        set_error_detail("qgemv_q2_0: this shape splits the reduction and needs %zu bytes of workspace (got %zu)",
                         need, ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    float *out = pl.splits > 1 ? static_cast<float *>(ws) : y;
    const int units = I / 8;
    switch (S) {
#define QG_CASE(SS) case SS: launch_q2_s<SS>(p, out, pl, units, U, st); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    if (pl.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), pl.splits, S, O, st);
    return check_launch("qgemv_q2_0");
}

}  // namespace

size_t ws_q2_0(int S, int I, int O) {
    const int s = S < 8 ? S : 8;
    int U = 1;
    size_t need = cs_ws_bytes(q2_plan(s, I, O, &U), s, O);
    TmaPlan tp;   // the larger of the staged and the direct plan (the pointers decide the path)
    if (s == 1 && I % 512 == 0 && q2_tma_plan(I, O, &tp) && tp.splits > 1) {
        const size_t t = (size_t)tp.splits * O * sizeof(float);
        if (t > need) need = t;
    }
    return need;
}

int run_gemv_q2_0(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                  size_t ws_bytes, cudaStream_t st) {
    for (int s0 = 0; s0 < S; s0 += 8) {
        const int sc = S - s0 < 8 ? S - s0 : 8;
        const int rc = gemv_q2_chunk(y + (size_t)s0 * O, x + (size_t)s0 * I, blocks, sc, I, O, ws, ws_bytes, st);
        if (rc != kOk) return rc;
    }
    return kOk;
}

}  // namespace qg
