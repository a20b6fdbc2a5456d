// gemv_q2_0.cu -- decode GEMV for the Q2_0 codec (the ggml Q2_0 layout the
// strata review checks in "convert_k256_q2_0.cpp vs ref_quant.cpp", 2.5):
// 18 bytes per 64 weights, an fp16 d at bytes [0,2) and 2-bit codes at
// [2,18), weight e of the block in byte 2 + e/4 at bit 2*(e%4);
//     w_e = (code_e - 1) * d.
//
// Direct column-stationary kernel (gemv_cs.cuh): a unit is 8 weights, the two
// code bytes 2 + 2h, 3 + 2h of a block (h = 0..7) -- blocks of 18 bytes keep
// units 2-byte aligned only, so a unit is one 16-bit load.  Per unit and
// token: sum_k code_k x_k in f32 (codes exact), then d * (that - sum_k x_k).
#include "gemv_cs.cuh"
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
                                                                         pl.nrowb);
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
    return cs_ws_bytes(q2_plan(s, I, O, &U), s, O);
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
