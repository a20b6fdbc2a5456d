// gemv_cs.cuh -- "column-stationary" decode GEMV skeleton.
//
// One thread block owns a contiguous column range of the weight matrix (the
// whole row unless the row is split across blocks) and walks down the rows in
// batches of RB.  Each thread owns U "units" -- NW 32-bit words of packed
// weights at fixed column positions -- so its slice of the activations is
// loaded once, pre-processed, and kept in registers for every row it visits:
// the main loop reads nothing but weights (and their scales/headers).  Per
// batch every thread issues RB*U independent streaming loads, decodes them in
// registers and produces RB*S partial dot products, which are summed across
// the block with a reduce-scatter butterfly and one barrier.
//
// A format supplies (see FmtI4G / FmtFp8B128 / FmtMq4v2):
//   kElemsPerWord               elements per 32-bit word of packed weights
//   Params                      device pointers and shape
//   unit_ptr(p, o, u)           address of unit u of row o
//   unit_aux(p, o, u, tc)       per-(row, unit) side data (scale / header)
//   load_x(p, s, u, xs[], xsum) unit u's activations of token s, in the form
//                               accumulate() wants
//   accumulate(words, aux, xs, xsum, part)
//                               add the unit's contribution for all S tokens
//
// Output: out[(split * S + s) * O + o]; split 0 of an unsplit call is y.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace qg {

constexpr int kCsMaxThreads = 512;

inline int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

template <int X> struct NextPow2 {
    static constexpr int value = X <= 1 ? 1 : X <= 2 ? 2 : X <= 4 ? 4 : X <= 8 ? 8 : X <= 16 ? 16 : 32;
};

// A unit's words: NW 32-bit streaming loads, or the format's own load when it
// defines load_unit (units that are only 2-byte aligned).
template <class F, int NW, class = void>
struct CsLoad {
    static constexpr uint32_t kBytes = 4u * NW;     // bytes a unit load reads
    __device__ static Words<NW> load(const void *p) { return ld_stream<NW>(p); }
};
template <class F, int NW>
struct CsLoad<F, NW, std::void_t<decltype(&F::template load_unit<NW>)>> {
    static constexpr uint32_t kBytes = 2u * NW;     // 16-bit units
    __device__ static Words<NW> load(const void *p) { return F::template load_unit<NW>(p); }
};

// Guards of the bounds-checking build for a unit access of row o: the unit's
// bytes lie inside the row, its side data inside its array; activations of
// token s, unit u lie inside x.
template <class F, int NW>
__device__ __forceinline__ bool cs_unit_in_bounds(const typename F::Params &p, int o, int u, int XU,
                                                  const typename F::ThreadConst &tc) {
    const long off = (long)((const uint8_t *)F::unit_ptr(p, o, u, XU) - (const uint8_t *)F::w_src(p, o, 0u));
    return o >= 0 && o < p.O && u >= 0 && off >= 0 && off + (long)CsLoad<F, NW>::kBytes <= (long)F::row_bytes(p) &&
           F::aux_ok(p, o, tc);
}
template <class F>
__device__ __forceinline__ bool x_unit_in_bounds(const typename F::Params &p, int s, int S, int u, int XU) {
    return s >= 0 && s < S && (u < 0 || (long)(u + 1) * XU <= (long)p.I);
}

template <class F, int S, int NW, int U, int RB>
__global__ void __launch_bounds__(kCsMaxThreads)
gemv_cs_kernel(const typename F::Params p, float *__restrict__ out, int units, int units_per_split,
               int nrowb, int *err)
{
    constexpr int XU = NW * F::kElemsPerWord;           // elements per unit
    constexpr int NV = NextPow2<RB * S>::value;          // reduced values per batch
    static_assert(RB * S <= 32, "RB * S must be <= 32");

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int split = blockIdx.y;
    const int ubeg = split * units_per_split;
    const int uend = min(units, ubeg + units_per_split);

    __shared__ float red[2][kCsMaxThreads / 32][NV];

    // ---- per-thread activation slice, loaded once -------------------------
    int uidx[U];
    bool uok[U];
    typename F::ThreadConst tc[U];
    float xs[U][S][XU];
    float xsum[U][S];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        uidx[j] = ubeg + tid + j * blockDim.x;
        uok[j] = uidx[j] < uend;
        tc[j] = F::thread_const(p, uok[j] ? uidx[j] : 0, XU);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int ux = uok[j] ? uidx[j] : -1;
            F::template load_x<XU>(p, s, qg_guard(x_unit_in_bounds<F>(p, s, S, ux, XU), err) ? ux : -1, xs[j][s],
                                   xsum[j][s]);
        }
    }

    // ---- walk the row batches ---------------------------------------------
    int buf = 0;
    for (int rb = blockIdx.x; rb < nrowb; rb += gridDim.x, buf ^= 1) {
        const int o0 = rb * RB;
        Words<NW> raw[RB][U];
        typename F::Aux aux[RB][U];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int o = o0 + r;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                if (o < p.O && uok[j] && qg_guard(cs_unit_in_bounds<F, NW>(p, o, uidx[j], XU, tc[j]), err)) {
                    raw[r][j] = CsLoad<F, NW>::load(F::unit_ptr(p, o, uidx[j], XU));
                    aux[r][j] = F::unit_aux(p, o, uidx[j], tc[j]);
                } else {
#pragma unroll
                    for (int k = 0; k < NW; ++k) raw[r][j].w[k] = 0u;
                    aux[r][j] = F::zero_aux();
                }
            }
        }

        float part[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) part[v] = 0.f;
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int j = 0; j < U; ++j)
                F::template accumulate<S, NW, XU>(raw[r][j], aux[r][j], xs[j], xsum[j], &part[r * S]);

        const float tot = warp_reduce_scatter<NV>(part, lane);
        if ((lane & ((32 / NV) - 1)) == 0)
            red[buf][warp][reduce_scatter_index<NV>(lane)] = tot;
        __syncthreads();
        if (tid < RB * S) {
            const int r = tid / S, s = tid - (tid / S) * S;
            const int o = o0 + r;
            float acc = 0.f;
            for (int w = 0; w < nwarps; ++w) acc += red[buf][w][tid];
            if (o < p.O && qg_guard(split < (int)gridDim.y && s < S, err)) out[((size_t)split * S + s) * p.O + o] = acc;
        }
    }
}

// Host-side launch plan of a column-stationary call.
struct CsPlan {
    int threads;          // threads per block (multiple of 32)
    int splits;           // column splits (grid.y); > 1 needs workspace
    int units_per_split;  // units owned by one block
    int nrowb;            // row batches
    int grid_x;           // blocks along the rows (each walks nrowb / grid_x batches)
};

// units: row length in units; u: units per thread; rb: rows per batch;
// regs_per_thread: estimate used for the residency bound.
CsPlan cs_plan(int units, int O, int u, int rb, int regs_per_thread);

// Workspace bytes of a plan for S tokens and O rows.
inline size_t cs_ws_bytes(const CsPlan &pl, int S, int O) {
    return pl.splits > 1 ? (size_t)pl.splits * (size_t)S * (size_t)O * sizeof(float) : 0;
}

// Enqueue the split reduction y[s, o] = sum_k ws[k, s, o].
void launch_splitk_reduce(float *y, const float *ws, int splits, int S, int O, cudaStream_t st);

int num_sms();  // SM count of the current device (cached per device)

}  // namespace qg
