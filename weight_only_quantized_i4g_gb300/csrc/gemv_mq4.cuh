// gemv_mq4.cuh -- decode GEMV for the 136-byte MQ4 block formats, templated
// on the header kind HK (instantiated by gemv_mq4v2.cu, gemv_mq4v1.cu,
// gemv_mq4c.cu).
//
// Formats (hipfire "MQ4 V2", sections 1b, 1e, 2 and 4): 136 bytes per 256
// weights, 128 payload bytes at [8,136), weight j in payload byte j/2 (low
// nibble for even j), w_j = q_j * scale + zero with
//   HK = 44  MQ4-V2 (qt=44): dword [0,4) = fp16 scale (low half) | fp16 zero
//            (high half) of weights 0..127, dword [4,8) the same for weights
//            128..255 (h = payload byte offset >= 64)
//   HK = 45  MQ4C pad (qt=45): one fp16 scale | fp16 zero dword at [0,4) for
//            all 256 weights, zero bytes at [4,8)
//   HK = 13  MQ4 v1 (qt=13): f32 scale at [0,4), f32 zero at [4,8), for all
//            256 weights
//
// Fast path (column-stationary): a unit is 4*NW payload bytes (8*NW weights)
// inside one half, so one header serves the unit; the half is derived from
// the unit's payload byte offset, never from a lane id.  The sum is
// folded as scale * sum(q*x) + zero * sum(x); the activations' sum over the
// unit is computed once per thread.  Nibble decode as for fmt=4 (the float
// 2^23 + q*16^p minus 2^23).
//
// Paths: staged (gemv_tma.cuh) when the rows are a whole number of 16-byte
// lines (I/256 even) and blocks and x are 16-byte aligned; direct otherwise.
// The staged path at one token (FmtMq4v2H) multiplies in the mixed-precision
// form fp16 x fp16 -> f32: one AND leaves two nibbles as fp16 subnormals
// (exact), which halves the integer-pipe work per weight, the bottleneck of
// the f32 pair form at batch 1; products stay exact and the accumulation f32.
#pragma once
#include "gemv_cs.cuh"
#include "gemv_mma.cuh"
#include "gemv_tma.cuh"
#include "launch.h"

namespace qg {

// Header of a block by kind: where a unit's header sits (from the unit's
// payload byte offset), how it is loaded and how it decodes.
template <int HK>
struct Mq4Header;
template <>
struct Mq4Header<44> {
    typedef uint32_t Raw;
    __device__ static int offset(int poff) { return poff >= 64 ? 4 : 0; }
    __device__ static Raw load_global(const uint8_t *p) { return ld_nc_u32(p); }
    __device__ static Raw load_shared(uint32_t a) { return lds_u32_at(a); }
    __device__ static Raw zero_raw() { return 0u; }
    __device__ static float scale(Raw h) { return f16_bits_to_f32((uint16_t)(h & 0xFFFFu)); }
    __device__ static float zero(Raw h) { return f16_bits_to_f32((uint16_t)(h >> 16)); }
};
template <>
struct Mq4Header<45> : Mq4Header<44> {
    __device__ static int offset(int) { return 0; }
};
template <>
struct Mq4Header<13> {
    typedef uint2 Raw;
    __device__ static int offset(int) { return 0; }
    __device__ static Raw load_global(const uint8_t *p) {
        uint2 v;
        asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
        return v;
    }
    __device__ static Raw load_shared(uint32_t a) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
        return v;
    }
    __device__ static Raw zero_raw() { return make_uint2(0u, 0u); }
    __device__ static float scale(Raw h) { return __uint_as_float(h.x); }
    __device__ static float zero(Raw h) { return __uint_as_float(h.y); }
};

struct Mq4Params {
    const uint16_t *x;
    const uint8_t *blocks;
    int I, O;
    size_t rowbytes;
};

template <int HK>
struct FmtMq4 {
    typedef Mq4Header<HK> Hdr;
    static constexpr int kElemsPerWord = 8;
    static constexpr int kPairsPerWord = 4;
    typedef Mq4Params Params;
    struct ThreadConst { int uoff; int hoff; };   // byte offsets of the unit and its header in a row
    typedef typename Hdr::Raw Aux;                 // the header of the unit

    __device__ static ThreadConst thread_const(const Params &, int u, int XU) {
        const int ub = XU / 2;                     // payload bytes per unit
        const int upb = 128 / ub;                  // units per block
        const int b = u / upb, k = u - (u / upb) * upb;
        const int poff = ub * k;                   // payload byte offset of the unit
        return ThreadConst{136 * b + 8 + poff, 136 * b + Hdr::offset(poff)};
    }
    __device__ static const void *unit_ptr(const Params &p, int o, int u, int XU) {
        return p.blocks + (size_t)o * p.rowbytes + thread_const(p, u, XU).uoff;
    }
    __device__ static Aux unit_aux(const Params &p, int o, int, ThreadConst tc) {
        return Hdr::load_global(p.blocks + (size_t)o * p.rowbytes + tc.hoff);
    }
    __device__ static Aux zero_aux() { return Hdr::zero_raw(); }
    // the unit's header lies inside the row (bounds-checking build)
    __device__ static bool aux_ok(const Params &p, int, ThreadConst tc) {
        return tc.hoff >= 0 && (size_t)tc.hoff + sizeof(Aux) <= p.rowbytes;
    }

    template <int XU>
    __device__ static void load_x(const Params &p, int s, int u, float (&xs)[XU], float &xsum) {
        float sum = 0.f;
#pragma unroll
        for (int wq = 0; wq < XU / 8; ++wq) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float sc = q == 0 ? 1.f : q == 1 ? 0.0625f : q == 2 ? 0.00390625f : 0.000244140625f;
                float a = 0.f, b = 0.f;
                if (u >= 0) {
                    const uint16_t *xp = p.x + (size_t)s * p.I + (size_t)u * XU + 8 * wq;
                    a = bf16_bits_to_f32(xp[q]);
                    b = bf16_bits_to_f32(xp[q + 4]);
                }
                sum += a + b;
                xs[2 * (4 * wq + q)] = a * sc;
                xs[2 * (4 * wq + q) + 1] = b * sc;
            }
        }
        xsum = sum;
    }

    template <int S, int NW, int XU>
    __device__ static void accumulate(const Words<NW> &wd, Aux hd, const float (&xs)[S][XU],
                                      const float (&xsum)[S], float *part) {
        constexpr uint32_t kMagic = 0x4B000000u;
        float2 d[NW * 4];
#pragma unroll
        for (int wq = 0; wq < NW; ++wq) {
            const uint32_t lo = wd.w[wq];
            const uint32_t hi = lo >> 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t m = 0xFu << (4 * q);
                float2 f = make_float2(__uint_as_float((lo & m) | kMagic), __uint_as_float((hi & m) | kMagic));
                d[4 * wq + q] = __fadd2_rn(f, make_float2(-8388608.f, -8388608.f));
            }
        }
        const float scale = Hdr::scale(hd);
        const float zero = Hdr::zero(hd);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NW * 4; ++i)
                acc = __ffma2_rn(d[i], make_float2(xs[s][2 * i], xs[s][2 * i + 1]), acc);
            part[s] = fmaf(scale, acc.x + acc.y, fmaf(zero, xsum[s], part[s]));
        }
    }

    // ---- staged (TMA) kernel -------------------------------------------------
    struct TConst { uint32_t uoff; uint32_t hoff; };   // unit and header byte offsets in the segment
    struct StageConst {};
    // routed experts: 16-byte aligned blocks for the staged copies (no side array)
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
    // a segment starts at a block boundary (splits cover whole blocks)
    __device__ static uint32_t seg_byte(const Params &, int u, int XU) {
        return 136u * (uint32_t)(u / (128 / (XU / 2)));
    }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.blocks + (size_t)o * p.rowbytes + col;
    }
    __device__ static const void *a_src(const Params &, int) { return nullptr; }
    __device__ static TConst tconst(const Params &p, int u, int XU, uint32_t seg_col) {
        const ThreadConst t = thread_const(p, u, XU);
        return TConst{(uint32_t)t.uoff - seg_col, (uint32_t)t.hoff - seg_col};
    }
    __device__ static StageConst stage_const(const Params &, int, TConst) { return StageConst{}; }
    template <int NW>
    __device__ static Words<NW> lds_unit(uint32_t a) { return lds_at<NW, false>(a); }  // 8-byte aligned units
    __device__ static Aux aux(uint32_t row_w, uint32_t, TConst tc, StageConst) {
        return Hdr::load_shared(row_w + tc.hoff);
    }


    // Activation pairs in the order nibbles_as_denormals produces weights
    // (see FmtI4G::load_x), raw; xsum = the unit's activation sum.
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        float e[XU];
#pragma unroll
        for (int v = 0; v < XU / 8; ++v) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (u >= 0) q = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + v);
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                e[8 * v + 2 * i] = __uint_as_float(wv[i] << 16);
                e[8 * v + 2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
            }
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

    // sum (q*scale + zero) * x = scale * 2^c * sum(q * x * 2^-c) + zero * xsum
    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, Aux hd, const uint64_t (&xp)[S][NP],
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
        const float scale = Hdr::scale(hd) * ts.p1;
        const float zero = Hdr::zero(hd);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            uint64_t acc = fmul2(d[0], xp[s][0]);
#pragma unroll
            for (int i = 1; i < NP; ++i) ffma2(acc, d[i], xp[s][i]);
            const float2 u = unpack2(acc);
            part[s] = fmaf(scale, (u.x + u.y) * ts.p2, fmaf(zero, xsum[s], part[s]));
        }
    }
};

// Batch-1 staged variant: fp16 activations, mixed-precision products.
//
// Per 32-bit word of nibbles n0..n7 (bits 4k), four ANDs leave f16x2 pairs
//   (n0, n4) * 2^-24   (n1, n5) * 2^-20   (n2, n6) * 2^-24   (n3, n7) * 2^-20
// (fp16 subnormals: the bit pattern n * 16^p with p <= 1 read as fp16 is
// exactly n * 16^p * 2^-24); the second pair of each comes from the word
// shifted down by 8.  Each multiplies, in fma.rn.f32.f16, the matching
// activations held as fp16 pairs, pre-scaled by 2^(141 - F) for the 2^-24
// positions and 2^(137 - F) for the 2^-20 ones, F being the exponent field
// of the thread's largest finite |x|: the scaled activations stay below
// 2^15, bf16 -> fp16 is exact for every x within 2^29 of that maximum (2^25
// for the 2^-20 positions), and every product is n * x * 2^(117 - F)
// exactly, accumulated in f32.
template <int HK>
struct FmtMq4H : FmtMq4<HK> {
    typedef FmtMq4<HK> Base;
    typedef typename Base::Params Params;
    typedef typename Base::Aux Aux;
    typedef typename Base::Hdr Hdr;
    static constexpr int kPairsPerWord = 2;   // two 64-bit registers = four fp16 pairs per word

    // Raw bf16 activations in slot order: word w of the unit holds slots
    // (x[8w], x[8w+4]), (x[8w+1], x[8w+5]) in xp[2w] and (x[8w+2], x[8w+6]),
    // (x[8w+3], x[8w+7]) in xp[2w+1]; prepare_x converts them to scaled fp16.
    template <int XU, int NP>
    __device__ static void load_x(const Params &p, int s, int u, uint64_t (&xp)[NP], float &xsum) {
        static_assert(NP == XU / 4, "four activations per 64-bit register");
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < XU / 8; ++w) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (u >= 0) q = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)s * p.I + (size_t)u * XU) + w);
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) sum += __uint_as_float(wv[i] << 16) + __uint_as_float(wv[i] & 0xFFFF0000u);
            uint32_t s0, s1, s2, s3;
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(s0) : "r"(q.x), "r"(q.z));
            asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(s1) : "r"(q.x), "r"(q.z));
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(s2) : "r"(q.y), "r"(q.w));
            asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(s3) : "r"(q.y), "r"(q.w));
            xp[2 * w] = (uint64_t)s0 | ((uint64_t)s1 << 32);
            xp[2 * w + 1] = (uint64_t)s2 | ((uint64_t)s3 << 32);
        }
        xsum = sum;
    }

    typedef Pow2Pair ThreadScale;   // 2^(F - 117) as two factors

    // bf16 pair -> fp16 pair of x * k1 * k2 (both factors powers of two).
    __device__ static uint32_t bf16x2_to_scaled_f16x2(uint32_t b, float k1, float k2) {
        const float lo = __uint_as_float(b << 16) * k1 * k2, hi = __uint_as_float(b & 0xFFFF0000u) * k1 * k2;
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }

    template <int U, int S, int NP>
    __device__ static ThreadScale prepare_x(uint64_t (&xp)[U][S][NP], float (&)[U][S]) {
        // largest finite |x| as a bf16 magnitude pattern (patterns >= 0x7F80 are inf / NaN)
        uint32_t m = 0;
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
        int F = (int)(m >> 7);                       // exponent field
        if (F < 1) F = 1;
        const int k24 = 141 - F, k20 = 137 - F;      // in [-117, 140]
        const float a24 = pow2i(k24 >> 1), b24 = pow2i(k24 - (k24 >> 1));
        const float a20 = pow2i(k20 >> 1), b20 = pow2i(k20 - (k20 >> 1));
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int s = 0; s < S; ++s)
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    // xp[2w] = slots (0, 1): 2^-24 then 2^-20 positions; xp[2w+1] likewise
                    const uint32_t lo = (uint32_t)xp[j][s][i], hi = (uint32_t)(xp[j][s][i] >> 32);
                    xp[j][s][i] = (uint64_t)bf16x2_to_scaled_f16x2(lo, a24, b24) |
                                  ((uint64_t)bf16x2_to_scaled_f16x2(hi, a20, b20) << 32);
                }
        const int c = F - 117;                       // in [-116, 137]
        return Pow2Pair{pow2i(c >> 1), pow2i(c - (c >> 1))};
    }

    // a0 += n(lo) * x(lo), a1 += n(hi) * x(hi), fp16 inputs, f32 result
    __device__ static void fma_mixed2(float &a0, float &a1, uint32_t n2, uint32_t x2) {
        asm("{.reg .f16 nl, nh, xl, xh;\n\t"
            "mov.b32 {nl, nh}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.f16 %0, nl, xl, %0;\n\t"
            "fma.rn.f32.f16 %1, nh, xh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(n2), "r"(x2));
    }

    // sum (q*scale + zero) * x = scale * 2^(F-117) * sum(q * x * 2^(117-F)) + zero * xsum
    template <int S, int NW, int NP>
    __device__ static void accumulate(const Words<NW> &wd, Aux hd, const uint64_t (&xp)[S][NP],
                                      const float (&xsum)[S], ThreadScale ts, float *part) {
        uint32_t n[NW][4];
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const uint32_t v = wd.w[w] >> 8;
            n[w][0] = wd.w[w] & 0x000F000Fu;
            n[w][1] = wd.w[w] & 0x00F000F0u;
            n[w][2] = v & 0x000F000Fu;
            n[w][3] = v & 0x00F000F0u;
        }
        const float scale = Hdr::scale(hd) * ts.p1;
        const float zero = Hdr::zero(hd);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const uint64_t x01 = xp[s][2 * w], x23 = xp[s][2 * w + 1];
                fma_mixed2(a0, a1, n[w][0], (uint32_t)x01);
                fma_mixed2(a0, a1, n[w][1], (uint32_t)(x01 >> 32));
                fma_mixed2(a0, a1, n[w][2], (uint32_t)x23);
                fma_mixed2(a0, a1, n[w][3], (uint32_t)(x23 >> 32));
            }
            part[s] = fmaf(scale, (a0 + a1) * ts.p2, fmaf(zero, xsum[s], part[s]));
        }
    }
};

// Warp-MMA decode (gemv_mma.cuh): a scale unit is a 128-weight half block
// (two 64-weight spans) with one header; A = q as fp16 subnormals, so
// acc += scale * sum(q x) + zero * sum(x) per half.
template <int HK>
struct MmaMq4 {
    static constexpr bool kHiLo = false;
    static constexpr bool kNeg8 = false;
    static constexpr int kSpansPerUnit = 2;
    static constexpr bool kFenceUnits = false;
    static constexpr int kMaxConsumerWarps = 15;   // 128 registers a thread
    static constexpr int kRedStride = 8;           // eight tokens per launch
    typedef Mq4Params Params;
    struct Side { float s, z; };
    __device__ static uint32_t row_bytes(const Params &p) { return (uint32_t)p.rowbytes; }
    __device__ static uint32_t aux_row_bytes(const Params &) { return 0u; }
    __device__ static const void *w_src(const Params &p, int o, uint32_t col) {
        return p.blocks + (size_t)o * p.rowbytes + col;
    }
    __device__ static const void *a_src(const Params &, int) { return nullptr; }
    // four spans per 136-byte block, at payload bytes 0, 32, 64, 96
    __host__ __device__ static uint32_t span_byte(int sp) { return 136u * (uint32_t)(sp >> 2); }
    __device__ static uint32_t span_off(int sp_local) {
        return 136u * (uint32_t)(sp_local >> 2) + 8u + 32u * (uint32_t)(sp_local & 3);
    }
    static constexpr int kXWords = 4;   // eight bf16 activations
    __device__ static const void *x_src(const Params &p, int tok, int col) { return p.x + (size_t)tok * p.I + col; }
    // largest |x| of eight bf16: packed 16-bit maximum of the magnitudes
    __device__ static float abs_max8(const uint32_t (&w)[4]) {
        const uint32_t m = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                    __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
        return __uint_as_float(max(m << 16, m & 0xFFFF0000u));
    }
    __device__ static uint64_t pair(const uint32_t (&w)[4], int i) {
        return (uint64_t)(w[i] << 16) | ((uint64_t)(w[i] & 0xFFFF0000u) << 32);
    }
    // The header of the half a unit covers: MQ4-V2 keeps the second half's
    // in the second dword (the unit's payload offset is >= 64), the one-header
    // formats one header for both halves.
    __device__ static uint32_t side_off(int, int sp_local0, int u) {
        return 136u * (uint32_t)(sp_local0 >> 2) + 136u * (uint32_t)(u >> 1) + (HK == 44 ? 4u * (uint32_t)(u & 1) : 0u);
    }
    __device__ static Side side(uint32_t row_w, uint32_t, uint32_t off) {
        if constexpr (HK == 13) {
            const uint2 h = lds_u32x2(row_w + off);
            return Side{__uint_as_float(h.x), __uint_as_float(h.y)};
        } else {
            const float2 f = f16x2_to_f32(lds_u32_at(row_w + off));
            return Side{f.x, f.y};
        }
    }
    __device__ static void apply(float (&acc)[4], const float (&d)[4], Side s0, Side s1, const float (&X)[2]) {
        acc[0] = fmaf(s0.s, d[0], fmaf(s0.z, X[0], acc[0]));
        acc[1] = fmaf(s0.s, d[1], fmaf(s0.z, X[1], acc[1]));
        acc[2] = fmaf(s1.s, d[2], fmaf(s1.z, X[0], acc[2]));
        acc[3] = fmaf(s1.s, d[3], fmaf(s1.z, X[1], acc[3]));
    }
};

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
namespace mq4 {

// Warp-MMA path: blocks and x 16-byte aligned (the staged copies, the
// activation vectors); any I % 256 == 0.
inline bool mq4_mma_ok(const uint16_t *x, const uint8_t *blocks) {
    return ((uintptr_t)blocks % 16 == 0) && ((uintptr_t)x % 16 == 0);
}

inline bool mq4_mma_plan(int S, int I, int O, MmaPlan *pl) {
    // column splits on 16-byte boundaries: whole pairs of blocks (272 bytes)
    return mma_plan(I / 64, 8, (uint32_t)((I / 256) * 136), 0u, 2u, S, O, 16, MmaMq4<44>::kMaxConsumerWarps,
                    MmaMq4<44>::kRedStride,
                    [](int sp) { return 136u * (uint32_t)(sp >> 2); }, pl);
}

inline int mq4_nw(int S) { return S <= 4 ? 2 : 1; }      // activation registers 8*NW*S <= 64
inline int mq4_rb(int S, int U) { return S <= 2 ? (U == 1 ? 8 : 4) : 4; }


inline bool mq4_tma_ok(const uint16_t *x, const uint8_t *blocks, int I) {
    return ((I / 256) % 2 == 0) && ((uintptr_t)blocks % 16 == 0) && ((uintptr_t)x % 16 == 0);
}

// staged path: 32-weight units (two 8-byte shared loads) at S <= 2, 16-weight
// units at S = 3, 4; from five tokens on, the four threads of a 32-weight
// unit split the tokens (two each), so each thread keeps the activations of
// two tokens as fp16 pairs (the batch-1 mixed-precision form) instead of all
// S tokens in f32 (measured at S = 8: 69.4 -> 59.3 us for 5120x17408, 71.8 ->
// 59.7 us for 17408x5120; at S = 4 it was not faster)
inline int mq4_nw_tma(int S) { return S <= 2 ? 4 : S <= 4 ? 2 : 4; }
inline int mq4_token_groups(int S) { return S <= 4 ? 1 : 4; }
constexpr int mq4_tg(int S) { return S <= 4 ? 1 : 4; }

inline bool mq4_tma_plan(int S, int I, int O, TmaPlan *pl) {
    const int nw = mq4_nw_tma(S);
    const int upb = 128 / (4 * nw);              // units per 256-weight block
    TmaGeom g;
    g.units = I / (8 * nw);
    g.granule = 2 * upb;                         // two blocks = 272 bytes = 17 lines of 16
    g.rowbytes = (uint32_t)((I / 256) * 136);
    g.granule_bytes = 272;
    g.arowbytes = 0;
    g.tg = mq4_token_groups(S);
    return tma_plan_rows(g, S, O, S == 1 ? 3 : 1, pl);
}

inline CsPlan mq4_plan(int S, int I, int O, int *U_out) {
    const int nw = mq4_nw(S);
    const int units = I / (8 * nw);
    // up to three units per thread at S = 1 (at S > 1 more than one spills
    // registers); longer rows split across blocks
    const int U = S == 1 ? (units > 2 * kCsMaxThreads ? 3 : units > kCsMaxThreads ? 2 : 1) : 1;
    *U_out = U;
    const int regs = 40 + 8 * nw * S * U + S * U + mq4_rb(S, U) * U * (nw + 1) + 2 * mq4_rb(S, U) * S;
    return cs_plan(units, O, U, mq4_rb(S, U), regs);
}

template <int HK, int S, int NW, int U>
void launch_cs_mq4(const Mq4Params &p, float *out, const CsPlan &pl, int units, cudaStream_t st) {
    constexpr int RB = S <= 2 ? (U == 1 ? 8 : 4) : 4;
    dim3 grid(pl.grid_x, pl.splits);
    gemv_cs_kernel<FmtMq4<HK>, S, NW, U, RB><<<grid, pl.threads, 0, st>>>(p, out, units, pl.units_per_split,
                                                                       pl.nrowb, device_error_word());
    count_launch();
}

template <int HK, int S>
void launch_cs_mq4_s(const Mq4Params &p, float *out, const CsPlan &pl, int units, int U,
                     cudaStream_t st) {
    constexpr int NW = S <= 4 ? 2 : 1;
    if constexpr (S == 1) {
        if (U == 2) {
            launch_cs_mq4<HK, S, NW, 2>(p, out, pl, units, st);
            return;
        }
        if (U == 3) {
            launch_cs_mq4<HK, S, NW, 3>(p, out, pl, units, st);
            return;
        }
    }
    (void)U;
    launch_cs_mq4<HK, S, NW, 1>(p, out, pl, units, st);
}

template <int HK, int S, int RB>
void launch_tma_mq4_u(const Mq4Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    constexpr int NW = S <= 2 ? 4 : S <= 4 ? 2 : 4;
    if constexpr (mq4_tg(S) > 1) {
        launch_tma<FmtMq4H<HK>, S, NW, 1, RB, mq4_tg(S)>(p, out, pl, st, moe);
    } else if constexpr (S == 1) {
        if (pl.U == 2) {
            launch_tma<FmtMq4H<HK>, S, NW, 2, RB>(p, out, pl, st, moe);
            return;
        }
        if (pl.U == 3) {
            launch_tma<FmtMq4H<HK>, S, NW, 3, RB>(p, out, pl, st, moe);
            return;
        }
        launch_tma<FmtMq4H<HK>, S, NW, 1, RB>(p, out, pl, st, moe);
    } else {
        launch_tma<FmtMq4<HK>, S, NW, 1, RB>(p, out, pl, st, moe);
    }
}

template <int HK, int S>
void launch_tma_mq4_s(const Mq4Params &p, float *out, const TmaPlan &pl, cudaStream_t st,
                      const MoeLaunch *moe = nullptr) {
    if constexpr (S <= 2) {
        if (pl.rb == 8) {
            launch_tma_mq4_u<HK, S, 8>(p, out, pl, st, moe);
            return;
        }
    }
    if (pl.rb == 2) {
        if constexpr (mq4_tg(S) > 1)
            launch_tma<FmtMq4H<HK>, S, 4, 1, 2, mq4_tg(S)>(p, out, pl, st, moe);
        else
            launch_tma<FmtMq4<HK>, S, (S <= 2 ? 4 : 2), 1, 2>(p, out, pl, st, moe);
        return;
    }
    launch_tma_mq4_u<HK, S, 4>(p, out, pl, st, moe);
}

template <int HK>
int gemv_mq4_chunk(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st, const char *name) {
    Mq4Params p;
    p.x = x; p.blocks = blocks; p.I = I; p.O = O; p.rowbytes = (size_t)(I / 256) * 136;

    // The warp-MMA kernel from two tokens on, and at one token when the rows
    // fit one block; the staged kernel at one token with a column split
    // (measured on GB300: 17408x5120 11.2 us against 11.9, 5120x17408 14.9
    // against 13.1; at eight tokens 14.4 and 19.1 us against 59.6 and 59.3).
    MmaPlan mp;
    if (mq4_mma_ok(x, blocks) && mq4_mma_plan(S, I, O, &mp) && (S > 1 || mp.splits == 1)) {
        const size_t need = mp.splits > 1 ? (size_t)mp.splits * S * O * sizeof(float) : 0;
        if (need > 0 && (ws == nullptr || ws_bytes < need)) {
            set_error_detail("%s: this shape splits the reduction and needs %zu bytes of workspace "
                             "(got %zu)", name, need, ws == nullptr ? (size_t)0 : ws_bytes);
            return kEWorkspace;
        }
        float *out = mp.splits > 1 ? static_cast<float *>(ws) : y;
        launch_mma<MmaMq4<HK>, kMmaSpansPerWarp, 16>(p, out, mp, st);
        if (mp.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), mp.splits, S, O, st);
        return check_launch(name);
    }

    TmaPlan tp;
    if (mq4_tma_ok(x, blocks, I) && mq4_tma_plan(S, I, O, &tp)) {
        const size_t need = tp.splits > 1 ? (size_t)tp.splits * S * O * sizeof(float) : 0;
        if (need > 0 && (ws == nullptr || ws_bytes < need)) {
            set_error_detail("%s: this shape splits the reduction and needs %zu bytes of workspace "
                             "(got %zu)", name, need, ws == nullptr ? (size_t)0 : ws_bytes);
            return kEWorkspace;
        }
        float *out = tp.splits > 1 ? static_cast<float *>(ws) : y;
        switch (S) {
#define QG_CASE(SS) case SS: launch_tma_mq4_s<HK, SS>(p, out, tp, st); break;
            QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
        }
        if (tp.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), tp.splits, S, O, st);
        return check_launch(name);
    }

    // the ABI guarantees 8-byte aligned blocks and 2-byte aligned x, which is
    // all the direct path needs, so the MQ4 formats have no general kernel
    int U = 1;
    const CsPlan pl = mq4_plan(S, I, O, &U);
    const int units = I / (8 * mq4_nw(S));
    const size_t need = cs_ws_bytes(pl, S, O);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) {
        set_error_detail("%s: this shape splits the reduction and needs %zu bytes of workspace "
                         "(got %zu)", name, need, ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    float *out = pl.splits > 1 ? static_cast<float *>(ws) : y;
    switch (S) {
#define QG_CASE(SS) case SS: launch_cs_mq4_s<HK, SS>(p, out, pl, units, U, st); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    if (pl.splits > 1) launch_splitk_reduce(y, static_cast<float *>(ws), pl.splits, S, O, st);
    return check_launch(name);
}

}  // namespace mq4

// Workspace bytes of the GEMV: the larger of the staged and the direct plan
// (the pointers decide the path).
inline size_t ws_mq4(int S, int I, int O) {
    const int s = S < 8 ? S : 8;
    size_t need = 0;
    TmaPlan tp;
    if ((I / 256) % 2 == 0 && mq4::mq4_tma_plan(s, I, O, &tp) && tp.splits > 1)
        need = (size_t)tp.splits * s * O * sizeof(float);
    MmaPlan mp;
    if (mq4::mq4_mma_plan(s, I, O, &mp) && mp.splits > 1)
        need = std::max(need, (size_t)mp.splits * s * O * sizeof(float));
    int U = 1;
    const size_t cs = cs_ws_bytes(mq4::mq4_plan(s, I, O, &U), s, O);
    return need > cs ? need : cs;
}

// GEMV of any S, in chunks of up to eight tokens.
template <int HK>
int run_gemv_mq4(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                 size_t ws_bytes, cudaStream_t st, const char *name) {
    for (int s0 = 0; s0 < S; s0 += 8) {
        const int sc = S - s0 < 8 ? S - s0 : 8;
        const int rc = mq4::gemv_mq4_chunk<HK>(y + (size_t)s0 * O, x + (size_t)s0 * I, blocks, sc, I, O, ws,
                                               ws_bytes, st, name);
        if (rc != kOk) return rc;
    }
    return kOk;
}


// Routed experts (the MQ4 formats): every slot on the staged kernel, one launch.
template <int HK>
int run_gemv_moe_mq4(float *y, const uint16_t *x, size_t x_stride, const void *table, int n_experts,
                     const int *ids, int n_slots, int S, int I, int O, cudaStream_t st) {
    const uint8_t *probe = reinterpret_cast<const uint8_t *>(uintptr_t(256));   // stands for any 16-byte aligned expert
    TmaPlan tp;
    if (!mq4::mq4_tma_ok(x, probe, I) || !mq4::mq4_tma_plan(S, I, moe_plan_rows(O, n_slots), &tp) ||
        tp.splits != 1) {
        set_error_detail("qgemv_moe: MQ4 routed experts need an even number of 256-weight blocks per row, a "
                         "16-byte aligned x and rows short enough for one block (I = %d)", I);
        return kEShape;
    }
    Mq4Params p;
    p.x = x; p.blocks = nullptr; p.I = I; p.O = O; p.rowbytes = (size_t)(I / 256) * 136;
    tp.nrowb = (O + tp.rb - 1) / tp.rb;            // the plan sized the launch for all slots' rows
    const MoeLaunch m{MoeSlots{static_cast<const ExpertW *>(table), ids, n_experts, x_stride}, n_slots};
    switch (S) {
#define QG_CASE(SS) case SS: mq4::launch_tma_mq4_s<HK, SS>(p, y, tp, st, &m); break;
        QG_CASE(1) QG_CASE(2) QG_CASE(3) QG_CASE(4) QG_CASE(5) QG_CASE(6) QG_CASE(7) QG_CASE(8)
#undef QG_CASE
    }
    return check_launch("qgemv_moe");
}

}  // namespace qg
