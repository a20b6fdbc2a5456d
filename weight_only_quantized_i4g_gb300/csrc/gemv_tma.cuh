// gemv_tma.cuh -- warp-specialized decode GEMV: bulk-copy (TMA) streaming of
// weight rows through a shared-memory ring, decode from shared memory.
//
// Block = 1 producer warp + nc consumer warps.  The block walks row batches
// rb = blockIdx.x, blockIdx.x + gridDim.x, ... of RB rows each.
//   producer  lane 0 fills up to nst ring slots ahead with 1-D bulk copies of
//             the batch's rows (one copy for whole rows, one per row for a
//             column split), completion counted on the slot's `full`
//             mbarrier; when the consumers release a slot (`empty` mbarrier)
//             the warp adds the consumers' per-warp partial sums of that
//             batch, writes the outputs and refills the slot.
//   consumers every thread owns U fixed column units (NW 32-bit words of
//             packed weights each) and holds the matching activations in
//             registers, loaded once with 16-byte vector loads and already in
//             the form the decode needs.  Per batch it reads its units from
//             shared memory, decodes, multiplies, reduces across the warp
//             with a reduce-scatter butterfly and leaves one partial per
//             (row, token) per warp in shared memory.
// Every wait is bounded; a wait that gives up raises the device error word
// and the warp leaves (the producer first lets its copies in flight land).
//
// A format F supplies:
//   kElemsPerWord, kPairsPerWord     elements / f32 pairs per 32-bit word
//   Params, TConst, StageConst
//   row_bytes(p), aux_row_bytes(p)   staged bytes per row (weights, side data)
//   w_src(p, o, col_byte), a_src(p, o)
//   seg_byte(p, u, XU)               byte offset in a row where unit u's segment starts
//   tconst(p, u, XU, seg_col)        per-unit offsets inside the staged segment
//   stage_const(p, o0, tc)           per-batch side data read from global
//   aux(sw_row, sa_row, tc, sc)      per-(row, unit) side data
//   load_x<XU, NP>(p, s, u, xp, xsum)  raw activations in decode order, their sum
//   prepare_x<U, S, NP>(xp, xsum)     per-thread scaling of the activations -> ThreadScale
//   zero_staged_aux()                 side data of an absent (row, unit): contributes 0
//   accumulate<S, NW, NP>(words, aux, xp, xsum, ts, part)
#pragma once

#include "common.cuh"
#include "gemv_cs.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qg {

// Consumer warps per block.  15 + the producer = 16 warps, four per SM
// sub-partition, leaves up to 128 registers per thread; the lighter
// one-unit, one-token variants (<= 96 registers) take 17 + 1.
constexpr int kTmaMaxConsumerWarps = 17;
__host__ __device__ constexpr int tma_max_consumer_warps(int S, int U) { return (U == 1 && S == 1) ? 17 : 15; }

template <int NW>
__device__ __forceinline__ Words<NW> lds_words(const uint8_t *p);
template <>
__device__ __forceinline__ Words<4> lds_words<4>(const uint8_t *p) {
    Words<4> r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "r"(smem_addr(p)));
    return r;
}
template <>
__device__ __forceinline__ Words<2> lds_words<2>(const uint8_t *p) {
    Words<2> r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "r"(smem_addr(p)));
    return r;
}
template <>
__device__ __forceinline__ Words<1> lds_words<1>(const uint8_t *p) {
    Words<1> r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r.w[0]) : "r"(smem_addr(p)));
    return r;
}

// Loads at 32-bit shared addresses (the stage ring is addressed that way).
template <int NW, bool kAlign16>
__device__ __forceinline__ Words<NW> lds_at(uint32_t a) {
    Words<NW> r;
    if constexpr (NW == 4 && kAlign16) {
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "r"(a));
    } else if constexpr (NW == 4) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%4];\n\tld.shared.v2.u32 {%2,%3}, [%4+8];"
                     : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "r"(a));
    } else if constexpr (NW == 2) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "r"(a));
    } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r.w[0]) : "r"(a));
    }
    return r;
}
__device__ __forceinline__ float lds_f32_at(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32_at(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// 2^k as a binary32, k in [-126, 127]
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

__device__ __forceinline__ float lds_f32(const uint8_t *p) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_addr(p)));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)));
    return v;
}

// ---------------------------------------------------------------------------
// Packed f32x2 helpers (sm_100 family)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
    return make_float2(a, b);
}
__device__ __forceinline__ void ffma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Scale every activation pair p of the thread by 2^(149 - 4*(p%4) - c), c
// chosen from the largest |x| it holds so the results are finite (see
// nibbles_as_denormals); returns 2^c as two representable factors.  Both
// multiplications are by powers of two, so they are exact.
struct Pow2Pair { float p1, p2; };
template <int U, int S, int NP>
__device__ __forceinline__ Pow2Pair prescale_for_denormals(uint64_t (&xp)[U][S][NP]) {
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < U; ++j)
#pragma unroll
        for (int s = 0; s < S; ++s)
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const float2 v = unpack2(xp[j][s][i]);
                m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
            }
    const int field = (int)((__float_as_uint(m) >> 23) & 0xFF);
    const int c = (field == 0 ? 1 : field) - 126 + 23;       // |x| < 2^(c - 23); c in [-102, 152]
    uint64_t f1[4], f2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int kq = 149 - 4 * q - c;                      // in [-15, 251]
        const float a = pow2i(kq >> 1), b = pow2i(kq - (kq >> 1));
        f1[q] = pack2(a, a);
        f2[q] = pack2(b, b);
    }
#pragma unroll
    for (int j = 0; j < U; ++j)
#pragma unroll
        for (int s = 0; s < S; ++s)
#pragma unroll
            for (int i = 0; i < NP; ++i) xp[j][s][i] = fmul2(fmul2(xp[j][s][i], f1[i % 4]), f2[i % 4]);
    return Pow2Pair{pow2i(c >> 1), pow2i(c - (c >> 1))};
}

// Eight nibbles of one word -> four f32 pairs d[q] = {n(q)*16^q, n(q+4)*16^q} - c_q
// where n(e) is the nibble of element e (bits 4e..4e+3).  OR-ing the masked
// nibble into the pattern of 2^23 gives 2^23 + n*16^q exactly; subtracting
// c_q = 2^23 + bias*16^q (bias 8 for signed nibbles, 0 for unsigned) is exact.
template <bool kSigned>
__device__ __forceinline__ void decode_nibbles(uint32_t w, uint64_t (&d)[4]) {
    // -(2^23 + bias*16^q) as f32 bit patterns, twice
    constexpr uint64_t c0 = kSigned ? 0xCB000008CB000008ull : 0xCB000000CB000000ull;
    constexpr uint64_t c1 = kSigned ? 0xCB000080CB000080ull : 0xCB000000CB000000ull;
    constexpr uint64_t c2 = kSigned ? 0xCB000800CB000800ull : 0xCB000000CB000000ull;
    constexpr uint64_t c3 = kSigned ? 0xCB008000CB008000ull : 0xCB000000CB000000ull;
    const uint32_t hi = w >> 16;
    uint64_t f0, f1, f2, f3;
    asm("{.reg .b32 a, b;\n\t"
        "lop3.b32 a, %1, 0x0000000F, 0x4B000000, 0xEA;\n\t"
        "lop3.b32 b, %2, 0x0000000F, 0x4B000000, 0xEA;\n\t"
        "mov.b64 %0, {a, b};}" : "=l"(f0) : "r"(w), "r"(hi));
    asm("{.reg .b32 a, b;\n\t"
        "lop3.b32 a, %1, 0x000000F0, 0x4B000000, 0xEA;\n\t"
        "lop3.b32 b, %2, 0x000000F0, 0x4B000000, 0xEA;\n\t"
        "mov.b64 %0, {a, b};}" : "=l"(f1) : "r"(w), "r"(hi));
    asm("{.reg .b32 a, b;\n\t"
        "lop3.b32 a, %1, 0x00000F00, 0x4B000000, 0xEA;\n\t"
        "lop3.b32 b, %2, 0x00000F00, 0x4B000000, 0xEA;\n\t"
        "mov.b64 %0, {a, b};}" : "=l"(f2) : "r"(w), "r"(hi));
    asm("{.reg .b32 a, b;\n\t"
        "lop3.b32 a, %1, 0x0000F000, 0x4B000000, 0xEA;\n\t"
        "lop3.b32 b, %2, 0x0000F000, 0x4B000000, 0xEA;\n\t"
        "mov.b64 %0, {a, b};}" : "=l"(f3) : "r"(w), "r"(hi));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d[0]) : "l"(f0), "l"(c0));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d[1]) : "l"(f1), "l"(c1));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d[2]) : "l"(f2), "l"(c2));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d[3]) : "l"(f3), "l"(c3));
}

// Nibbles read as denormal floats.  For a 32-bit pair {a, b} (two words of
// packed nibbles in one 64-bit register pair), AND-ing with a nibble mask
// leaves, in each half, the bit pattern n*16^q, which as a binary32 is the
// denormal n*16^q*2^-149 exactly.  d[q] holds nibble q of a and of b,
// d[4+q] nibble q+4 of a and of b (from the halves shifted down by 16).
// Multiplying by an activation pre-scaled by 2^(149-4q-c) gives n*x*2^-c in
// one fma with no subtraction; c is chosen per thread so every pre-scaled
// activation is finite and every product of a nonzero nibble is normal.
__device__ __forceinline__ void nibbles_as_denormals(uint64_t ab, uint64_t (&d)[8]) {
    uint64_t hab;
    asm("{.reg .b32 a, b, c, e;\n\t"
        "mov.b64 {a, b}, %1;\n\t"
        "shr.b32 c, a, 16;\n\t"
        "shr.b32 e, b, 16;\n\t"
        "mov.b64 %0, {c, e};}" : "=l"(hab) : "l"(ab));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint64_t m = (uint64_t)(0xFu << (4 * q)) * 0x0000000100000001ull;
        d[q] = ab & m;
        d[4 + q] = hab & m;
    }
}

// Two e4m3 codes (low 16 bits of `two`) -> f32 pair (exact; NaN codes -> NaN)
__device__ __forceinline__ uint64_t decode_e4m3x2(uint32_t two) {
    uint64_t r;
    asm("{.reg .b16 lo, hi;\n\t"
        ".reg .b32 h2;\n\t"
        ".reg .f16 fl, fh;\n\t"
        ".reg .f32 a, b;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, lo;\n\t"
        "mov.b32 {fl, fh}, h2;\n\t"
        "cvt.f32.f16 a, fl;\n\t"
        "cvt.f32.f16 b, fh;\n\t"
        "mov.b64 %0, {a, b};}" : "=l"(r) : "r"(two));
    return r;
}

struct TmaLayout {
    uint32_t stage_w;    // bytes per ring slot, weights
    uint32_t stage_a;    // bytes per ring slot, side data
    uint32_t red_off;    // offset of the partial-sum area
    uint32_t bar_off;    // offset of the mbarriers
    uint32_t total;      // dynamic shared memory bytes
};

// TG > 1 (token split): the consumer threads of a unit form TG groups (lanes
// with equal lane % TG), each holding the activations of ST = ceil(S / TG)
// tokens only; the groups' partial sums are reduced across the lanes of the
// same group.  Used where S tokens of activations per thread would not fit
// in registers.
template <class F, int S, int NW, int U, int RB, int TG = 1>
__device__ __forceinline__ void gemv_tma_body(const typename F::Params &p, float *__restrict__ out, int units,
                                              int units_per_split, int nrowb, int nst, const TmaLayout &L,
                                              int *err)
{
    constexpr int XU = NW * F::kElemsPerWord;
    constexpr int NP = NW * F::kPairsPerWord;
    constexpr int NV = NextPow2<RB * S>::value;
    constexpr int ST = (S + TG - 1) / TG;             // tokens per consumer thread
    constexpr int NT = TG == 1 ? NV : RB * ST;        // partial sums per consumer thread
    static_assert(RB * S <= 32, "RB * S must be <= 32");
    static_assert(TG == 1 || TG == 2 || TG == 4, "token groups must divide a warp evenly");

    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nc = (blockDim.x >> 5) - 1;
    uint8_t *stage_w = smem;
    uint8_t *stage_a = smem + (size_t)nst * L.stage_w;
    float *red = reinterpret_cast<float *>(smem + L.red_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *empty = full + nst;

    if (tid == 0) {
        qg_stamp_entry(err);
        griddep_launch_dependents();
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], (uint32_t)nc);
        }
        mbar_fence_init();
    }
    __syncthreads();

    const int G = gridDim.x, b = blockIdx.x;
    const int split = blockIdx.y, nsplit = gridDim.y;
    const int n_my = b < nrowb ? (nrowb - b + G - 1) / G : 0;
    const uint32_t rowbytes = F::row_bytes(p);
    const uint32_t arowbytes = F::aux_row_bytes(p);
    const int ubeg = split * units_per_split;
    const int uend = min(units, ubeg + units_per_split);
    // bytes of one row staged by this block (the whole row, or this split's segment)
    const uint32_t seg_col = nsplit == 1 ? 0u : F::seg_byte(p, ubeg, XU);
    const uint32_t seg_bytes = nsplit == 1 ? rowbytes : F::seg_byte(p, uend, XU) - seg_col;

    if (warp == 0) {
        // ------------------------------- producer -------------------------------
        auto issue = [&](int k) {
            const int slot = k % nst;
            const int o0 = (b + k * G) * RB;
            const int rows = min(RB, p.O - o0);
            const uint32_t wb = (uint32_t)rows * seg_bytes, ab = (uint32_t)rows * arowbytes;
            // the batch's rows lie inside the matrix and the segment inside a row
            // (bounds-checking build); a refused batch is armed with no bytes
            const bool in = qg_guard(o0 >= 0 && rows >= 1 && o0 + rows <= p.O && seg_col + seg_bytes <= rowbytes, err);
            mbar_arrive_expect_tx(&full[slot], in ? wb + ab : 0u);
            if (!in) return;
            uint8_t *dw = stage_w + (size_t)slot * L.stage_w;
            if (nsplit == 1) {
                bulk_copy_g2s(dw, F::w_src(p, o0, 0u), wb, &full[slot]);
            } else {
                for (int r = 0; r < rows; ++r)
                    bulk_copy_g2s(dw + (size_t)r * seg_bytes, F::w_src(p, o0 + r, seg_col), seg_bytes, &full[slot]);
            }
            if (ab) bulk_copy_g2s(stage_a + (size_t)slot * L.stage_a, F::a_src(p, o0), ab, &full[slot]);
        };
        // The weights do not depend on the previous kernel on the stream: the
        // first batches stream in before the wait that guards the outputs.
        if (lane == 0)
            for (int k = 0; k < min(nst, n_my); ++k) issue(k);
        __syncwarp();
        griddep_wait();
        for (int k = 0; k < n_my; ++k) {
            const int slot = k % nst;
            if (!mbar_wait(&empty[slot], (uint32_t)(k / nst) & 1u)) {
                if (lane == 0) {
                    raise_device_error(err, kErrTimeout);
                    for (int j = k; j < min(k + nst, n_my); ++j)
                        (void)mbar_wait(&full[j % nst], (uint32_t)(j / nst) & 1u);
                }
                return;
            }
            const int o0 = (b + k * G) * RB;
            if (lane < RB * S) {
                const int r = lane / S, s = lane - (lane / S) * S;
                const float *rs = red + (size_t)slot * nc * NV + lane;
                float acc = 0.f;
                for (int w = 0; w < nc; ++w) acc += rs[(size_t)w * NV];
                if (o0 + r < p.O && qg_guard(split < nsplit && s < S, err))
                    out[((size_t)split * S + s) * p.O + o0 + r] = acc;
            }
            __syncwarp();
            if (lane == 0 && k + nst < n_my) issue(k + nst);
        }
        if (lane == 0) {
            qg_stamp(err, kStStored);
            qg_stamp_put(err, kStBatches, (unsigned long long)n_my);
        }
        return;
    }

    // ------------------------------- consumers ----------------------------------
    griddep_wait();   // x may be the previous kernel's output
    if (tid == 32) qg_stamp(err, kStWaitDone);
    const int cw = warp - 1;
    const int ct = tid - 32;
    const int tg = TG == 1 ? 0 : ct % TG;             // token group (lane % TG)
    const int nuth = nc * 32 / TG;                    // unit slots per block
    int uidx[U];
    bool uok[U];
    typename F::TConst tc[U];   // a thread past the last unit takes unit ubeg (zero activations)
    uint64_t xp[U][ST][NP];
    float xsum[U][ST];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        uidx[j] = ubeg + (TG == 1 ? ct : ct / TG) + j * nuth;
        uok[j] = uidx[j] < uend;
        tc[j] = F::tconst(p, uok[j] ? uidx[j] : ubeg, XU, seg_col);
#pragma unroll
        for (int s = 0; s < ST; ++s) {
            const int tok = tg * ST + s;              // a padding token (tok >= S) reads zeros
            const int tx = tok < S ? tok : 0, ux = (uok[j] && tok < S) ? uidx[j] : -1;
            F::template load_x<XU, NP>(p, tx, qg_guard(x_unit_in_bounds<F>(p, tx, S, ux, XU), err) ? ux : -1,
                                       xp[j][s], xsum[j][s]);
        }
    }
    const typename F::ThreadScale ts = F::template prepare_x<U, ST, NP>(xp, xsum);
    if (tid == 32) qg_stamp(err, kStXReady);
    typename F::StageConst scur[U], snext[U];
#pragma unroll
    for (int j = 0; j < U; ++j) scur[j] = F::stage_const(p, b * RB, tc[j]);
    const uint32_t sw0 = smem_addr(stage_w), sa0 = smem_addr(stage_a);

    for (int k = 0; k < n_my; ++k) {
        const int slot = k % nst;
#pragma unroll
        for (int j = 0; j < U; ++j) snext[j] = F::stage_const(p, (b + (k + 1) * G) * RB, tc[j]);
        if (!mbar_wait(&full[slot], (uint32_t)(k / nst) & 1u)) {
            if (lane == 0) raise_device_error(err, kErrTimeout);
            return;
        }
        if (tid == 32 && k == 0) qg_stamp(err, kStFirstBatch);
        const uint32_t swb = sw0 + (uint32_t)slot * L.stage_w;
        const uint32_t sab = sa0 + (uint32_t)slot * L.stage_a;
        float part[NT];
#pragma unroll
        for (int v = 0; v < NT; ++v) part[v] = 0.f;
        // Rows in sub-batches of RS: the sub-batch's shared-memory reads first,
        // then its arithmetic.  No predicates: a thread without a unit of its
        // own reads unit ubeg of the same row with zero activations (adds 0),
        // and rows past the end of the matrix (last batch) read stale slot
        // bytes whose partial sums are never written out.
        constexpr int RS = (S <= 2 ? 4 : 2) / U >= 1 ? (S <= 2 ? 4 : 2) / U : 1;
#pragma unroll
        for (int r0 = 0; r0 < RB; r0 += RS) {
            Words<NW> wd[RS][U];
            typename F::Aux ax[RS][U];
#pragma unroll
            for (int rr = 0; rr < RS; ++rr) {
                const uint32_t rw = swb + (uint32_t)(r0 + rr) * seg_bytes;
                const uint32_t ra = sab + (uint32_t)(r0 + rr) * arowbytes;
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    wd[rr][j] = F::template lds_unit<NW>(rw + tc[j].uoff);
                    ax[rr][j] = F::aux(rw, ra, tc[j], scur[j]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < RS; ++rr)
#pragma unroll
                for (int j = 0; j < U; ++j)
                    F::template accumulate<ST, NW, NP>(wd[rr][j], ax[rr][j], xp[j], xsum[j], ts,
                                                       &part[(r0 + rr) * ST]);
        }
        if constexpr (TG == 1) {
            const float tot = warp_reduce_scatter<NV>(part, lane);
            if ((lane & ((32 / NV) - 1)) == 0)
                red[((size_t)slot * nc + cw) * NV + reduce_scatter_index<NV>(lane)] = tot;
        } else {
            // sum over the lanes of this token group; lanes 0 .. TG-1 write
            // (row r, token) at r * S + token, the layout the producer reads
#pragma unroll
            for (int off = TG; off < 32; off <<= 1)
#pragma unroll
                for (int v = 0; v < NT; ++v) part[v] += __shfl_xor_sync(0xFFFFFFFFu, part[v], off);
            if (lane < TG) {
#pragma unroll
                for (int r = 0; r < RB; ++r)
#pragma unroll
                    for (int t = 0; t < ST; ++t)
                        if (lane * ST + t < S)
                            red[((size_t)slot * nc + cw) * NV + r * S + lane * ST + t] = part[r * ST + t];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
#pragma unroll
        for (int j = 0; j < U; ++j) scur[j] = snext[j];
    }
    if (tid == 32) qg_stamp(err, kStConsumed);
}

// A token-split kernel is capped for two blocks per SM (64 registers): the
// occupancy is worth more than the few spilled bytes (measured at S = 8).
template <class F, int S, int NW, int U, int RB, int TG = 1>
__global__ void __launch_bounds__(32 * (tma_max_consumer_warps(S, U) + 1), TG > 1 ? 2 : 1)
gemv_tma_kernel(const typename F::Params p, float *__restrict__ out, int units, int units_per_split,
                int nrowb, int nst, TmaLayout L, int *err)
{
    gemv_tma_body<F, S, NW, U, RB, TG>(p, out, units, units_per_split, nrowb, nst, L, err);
}

// ---------------------------------------------------------------------------
// Routed experts: one launch for n_slots GEMVs of one format and shape.
// Slot r (blockIdx.z) multiplies the expert table[ids[r]] (device arrays,
// possibly written by the previous kernel on the stream, hence the wait
// before they are read) with x + r * x_stride into out + r * S * O.  An
// expert id outside [0, n_experts) or an expert whose pointers the staged
// copies cannot take (F::expert_ok) raises kErrExpert; that slot's outputs
// are then written as NaN.
// ---------------------------------------------------------------------------
struct ExpertW {            // same layout as qg_expert in qgemv.h
    const void *w;
    const float *scales;
};
struct MoeSlots {
    const ExpertW *table;
    const int *ids;
    int n_experts;
    size_t x_stride;         // activation elements between consecutive slots (0: shared x)
};
constexpr int kErrExpert = -8;

template <class F, int S, int NW, int U, int RB, int TG = 1>
__global__ void __launch_bounds__(32 * (tma_max_consumer_warps(S, U) + 1), TG > 1 ? 2 : 1)
gemv_tma_moe_kernel(const typename F::Params p0, float *__restrict__ out0, MoeSlots m, int units,
                    int units_per_split, int nrowb, int nst, TmaLayout L, int *err)
{
    griddep_wait();          // the routing (ids) may be the previous kernel's output
    const int r = blockIdx.z;
    float *out = out0 + (size_t)r * S * p0.O;
    const int id = m.ids[r];
    ExpertW e = {nullptr, nullptr};
    if (id >= 0 && id < m.n_experts) e = m.table[id];
    if (!F::expert_ok(p0, e.w, e.scales)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_device_error(err, kErrExpert);
        if (blockIdx.y == 0)
            for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < S * p0.O; i += gridDim.x * blockDim.x)
                out[i] = __int_as_float(0x7FC00000);
        return;
    }
    const typename F::Params p = F::with_expert(p0, e.w, e.scales, (size_t)r * m.x_stride);
    gemv_tma_body<F, S, NW, U, RB, TG>(p, out, units, units_per_split, nrowb, nst, L, err);
}

// ---------------------------------------------------------------------------
// Host side: plan and launch
// ---------------------------------------------------------------------------
struct TmaPlan {
    int rb;               // rows per batch
    int units;            // units per row
    int U;                // units per consumer thread
    int nc;               // consumer warps
    int splits;           // column splits (grid.y)
    int units_per_split;
    int nrowb;            // row batches
    int nst;              // ring slots
    int per_sm;           // blocks per SM the ring was sized for
    TmaLayout L;
};

// Row geometry handed to the planner by a format.
struct TmaGeom {
    int units;                // units per row
    int granule;              // a column split covers a multiple of this many units
    uint32_t rowbytes;        // staged bytes of a whole row
    uint32_t granule_bytes;   // staged bytes of one granule
    uint32_t arowbytes;       // staged side-data bytes per row
    int tg = 1;               // token groups (consumer threads per unit)
};

// Plan of RB-row batches; at most max_per_sm blocks per SM share its shared
// memory (the ring is sized for that many).  A plan of one block per SM keeps
// at most one_block_slots ring slots: the spare shared memory lets the next
// kernel's blocks start on the SM (and prefetch their weights) while this
// one finishes (measured: MQ4-V2 5120x17408 14.2 -> 13.0 us, fmt=7
// 24576x7168 28.0 -> 27.6 us with three slots instead of six).
bool tma_plan(const TmaGeom &g, int S, int O, int RB, int NV, int U_max, TmaPlan *pl, int max_per_sm = 8,
              int one_block_slots = 3);

// Plan for a matrix of a few MB at S <= 2: one block per SM, 8-row batches.
// Otherwise the largest batch (8, 4 or 2 rows; only 4 or 2 when S > 2, only
// 8 or 4 when a thread owns several units) that gives every resident block at
// least three batches to overlap with an even last wave (mean batches per
// block >= 92% of the maximum), else the most even of those; short matrices
// get 2-row batches.
bool tma_plan_rows(const TmaGeom &g, int S, int O, int U_max, TmaPlan *pl);

// Device address of this device's error word (cached per device).
int *device_error_word();

// Launch gemv_tma_kernel<F, S, NW, U, RB> with plan `pl`.
// With `moe`, the routed-expert kernel over moe->n_slots slots (grid.z; the
// plan must not split the reduction); each slot gets an equal share of the
// resident blocks (at least one).
// Rows a routed-expert launch is planned for: all slots' rows together (one
// launch streams them all), capped to an int.
inline int moe_plan_rows(int O, int n_slots) {
    const long long r = (long long)O * n_slots;
    return r > 0x7FFFFFFF ? 0x7FFFFFFF : (int)r;
}

struct MoeLaunch {
    MoeSlots slots;
    int n_slots;
};

template <class F, int S, int NW, int U, int RB, int TG = 1>
void launch_tma(const typename F::Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                const MoeLaunch *moe = nullptr) {
    auto kern = gemv_tma_kernel<F, S, NW, U, RB, TG>;
    auto kern_moe = gemv_tma_moe_kernel<F, S, NW, U, RB, TG>;
    const void *kfn = moe ? reinterpret_cast<const void *>(kern_moe) : reinterpret_cast<const void *>(kern);
    // The shared-memory limit is an attribute of the kernel in the current
    // context: set once per context and kernel.
    set_max_dynamic_smem(kfn, 232448);
    const int threads = 32 * (pl.nc + 1);
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, threads, pl.L.total) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    long resident = (long)num_sms() * per_sm / pl.splits;
    if (moe) resident /= moe->n_slots;
    if (resident < 1) resident = 1;
    const int grid_x = pl.nrowb < resident ? pl.nrowb : (int)resident;
    // Programmatic dependent launch: the kernel may start while the previous
    // kernel on the stream finishes (see griddep_wait).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, pl.splits, moe ? moe->n_slots : 1);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = pl.L.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (moe)
        cudaLaunchKernelEx(&cfg, kern_moe, p, out, moe->slots, pl.units, pl.units_per_split, pl.nrowb, pl.nst,
                           pl.L, device_error_word());
    else
        cudaLaunchKernelEx(&cfg, kern, p, out, pl.units, pl.units_per_split, pl.nrowb, pl.nst, pl.L,
                           device_error_word());
    count_launch();
}

}  // namespace qg
