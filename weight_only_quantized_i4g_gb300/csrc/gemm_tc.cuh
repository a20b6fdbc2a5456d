// gemm_tc.cuh -- batched-prefill dequant-GEMM on the 5th-generation tensor
// cores (tcgen05 MMA, accumulators in tensor memory), generic over the
// weight format.
//
//   Y[m, o] = sum_i X[m, i] * w(o, i)       X bf16 [M, I], Y f32 [M, O]
//
// where w(o, i) is the format's dequantized weight.  A format supplies a
// policy F (see gemm_i4g_tc.cu, gemm_fp8b128_tc.cu, gemm_mq4v2_tc.cu): a
// bound on |w| over (part of) a row, how one thread loads the bytes of 32
// consecutive weights of one row for a 128-wide K step, and how it turns
// them into 16 f16x2 words.
//
// Operand precision.  Both MMA operands are fp16 (11 significant bits), so
// every product carries a relative error of at most 2^-11 + 2^-24 < 1e-3 and
// the bound 1e-3 * sum_i |w_i x_i| holds for every output, whatever the
// spread of the terms (bf16 operands, 8 bits, can exceed it when a few
// large terms dominate a sum).  fp16's range is kept by powers of two: a
// preparation kernel converts each token row of X to fp16 as x * 2^-F[m],
// with F[m] placing the row's largest finite |x| in [2^14, 2^15) (exact for
// every element within 2^29 of that maximum); each weight row gets a scale
// 2^E[o] that places the format's bound on its |w| in [2^14, 2^15] (the
// same kernel, one warp per row).  The weight is formed in f32 (one
// rounding), scaled by 2^E[o] (exact) and rounded to fp16.  The store multiplies the f32 accumulator by
// 2^(F[m] - E[o]) (exact).  The MMA runs at the same rate as with bf16.
//
// One persistent thread block per SM, warp-specialized.  Output tile: 128
// outputs (the weight rows, MMA M) by BT tokens (MMA N), K in steps of 128.
//   warp 0      TMA producer: per K step the BT x 128 fp16 tile of X (two
//               128-byte-swizzled boxes of 64) into a shared-memory ring
//               (operand B);
//   warp 1      allocates tensor memory and issues the MMAs from one thread:
//               per K step 8 instructions of M=128, N=BT, K=16 with operand
//               A read from tensor memory;
//   warps 2-5   epilogue: accumulator -> registers -> Y (or a partial slot);
//   warps 6-21  load the weights of the tile straight from global memory
//               (three K steps ahead in registers), dequantize them and
//               store the fp16 rows into a ring of A tiles in tensor memory
//               (tcgen05.st): warp w covers the 32 lanes (weight rows) its
//               position allows and one 32-wide quarter of the K step (four
//               dequantizing warps per sub-partition hide each other's
//               latency).
// One barrier per stage counts both the X bytes and the sixteen dequantizing
// warps, and one commit per step frees the stage: the MMA thread's waits and
// commits cost ~200 cycles each, so they are kept to one of each per 1024
// cycles of tensor-core work.
// Keeping the dequantized weights as operand A in tensor memory means each
// of them serves BT = 256 tokens, and shared memory carries only X: the
// dequantization work per MAC is half that of a 128-token tile, and no
// shared-memory bandwidth goes to writing and re-reading fp16 weights.
// The (tile, K step) units are split evenly over the blocks ("stream-K",
// streamk.h); a tile shared by several blocks is summed in contributor order
// by the block that arrives last at the tile's counter.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"
#include "streamk.h"

namespace qg {
int num_sms();
int *device_error_word();

namespace tc {

constexpr int kMmaM = 128;        // rows of one MMA (weight rows = outputs)
constexpr int kBK = 128;          // K per stage: two 128-byte rows of fp16
constexpr int kBKBox = 64;        // K of one 128-byte-swizzled box
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpEpi = 2, kNumEpiWarps = 4, kWarpDeq = 6, kNumDeqWarps = 16;
constexpr int kThreads = 32 * (kWarpDeq + kNumDeqWarps);
constexpr uint32_t kSmemBudget = 227 * 1024;
constexpr int kPrefetch = 3;      // K steps of packed weights in flight per dequantizing thread

// Instruction descriptor of tcgen05.mma kind::f16: f32 accumulator, fp16 A
// and B (format code 0), both K-major, M = 128, N = n.
constexpr uint32_t idesc_f16(int n) {
    return (1u << 4)                          // D format f32
           | ((uint32_t)(n >> 3) << 17)       // N / 8
           | ((uint32_t)(kMmaM >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row groups of 128-byte rows, 1024 bytes apart).  Advancing K by
// 16 fp16 inside the 128-byte row moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                      // leading offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;            // stride offset between 8-row groups
    d |= (uint64_t)1 << 46;                      // descriptor version
    d |= (uint64_t)2 << 61;                      // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) (+)= A (tensor memory, 128 rows x 16 fp16 in 8
// columns) x B (shared memory, descriptor)^T.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(accumulate), "r"(idesc));
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// 32 consecutive f32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive f32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Helpers of the 4-bit formats.  A nibble n moved to bit 4p (p <= 4, inside
// the 23-bit mantissa) and ORed under the exponent of 2^23 is the f32 value
// 2^23 + n*16^p, so one f32 add with -(2^23 + c*16^p) leaves (n - c)*16^p
// exactly; a scale multiplied by 16^-p (exact: a power of two) then undoes
// the position.  Pairs run on the f32x2 pipe.
constexpr uint32_t kNibExp = 0x4B000000u;   // 2^23

__device__ __forceinline__ uint64_t f32_pair(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// (lo + bias.lo) * scale.lo and the same for hi, each rounded once to f32,
// then both rounded to one f16x2 word (nearest even), lo in the low half.
__device__ __forceinline__ uint32_t nib_add_mul(uint32_t lo, uint32_t hi, uint64_t bias2, uint64_t scale2) {
    uint32_t r;
    asm("{\n\t.reg .b64 t;\n\t.reg .f32 a, b;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "add.rn.f32x2 t, t, %3;\n\t"
        "mul.rn.f32x2 t, t, %4;\n\t"
        "mov.b64 {a, b}, t;\n\t"
        "cvt.rn.f16x2.f32 %0, b, a;\n\t}"
        : "=r"(r)
        : "r"(lo), "r"(hi), "l"(bias2), "l"(scale2));
    return r;
}

// (lo + bias.lo) * scale.lo + zero.lo with one rounding (fused), the same
// for hi, then to one f16x2 word.
__device__ __forceinline__ uint32_t nib_add_fma(uint32_t lo, uint32_t hi, uint64_t bias2, uint64_t scale2,
                                                uint64_t zero2) {
    uint32_t r;
    asm("{\n\t.reg .b64 t;\n\t.reg .f32 a, b;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "add.rn.f32x2 t, t, %3;\n\t"
        "fma.rn.f32x2 t, t, %4, %5;\n\t"
        "mov.b64 {a, b}, t;\n\t"
        "cvt.rn.f16x2.f32 %0, b, a;\n\t}"
        : "=r"(r)
        : "r"(lo), "r"(hi), "l"(bias2), "l"(scale2), "l"(zero2));
    return r;
}

// Scale pairs for the nibble positions nib_positions uses, lane 0 = the even
// weight: (p0, p1), (p2, p3), (p4, p2), (p3, p4), each scale * 16^-p.
struct NibPairs {
    uint64_t v[4];
};
__device__ __forceinline__ NibPairs nib_scale_pairs(float s) {
    const float s1 = s * 0.0625f, s2 = s * 0.00390625f, s3 = s * 0.000244140625f, s4 = s * 0.0000152587890625f;
    NibPairs p;
    p.v[0] = f32_pair(s, s1);
    p.v[1] = f32_pair(s2, s3);
    p.v[2] = f32_pair(s4, s2);
    p.v[3] = f32_pair(s3, s4);
    return p;
}

// The eight nibbles of `w` (nibble j = weight j) as four pairs of f32 bit
// patterns 2^23 + n*16^p: nibbles 0-4 masked in place, 5-7 after one shift
// by 12 (positions 2-4).  Pair i holds weights 2i and 2i+1.
__device__ __forceinline__ void nib_positions(uint32_t w, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    const uint32_t v = w >> 12;
    lo[0] = (w & 0xFu) | kNibExp;
    hi[0] = (w & 0xF0u) | kNibExp;
    lo[1] = (w & 0xF00u) | kNibExp;
    hi[1] = (w & 0xF000u) | kNibExp;
    lo[2] = (w & 0xF0000u) | kNibExp;
    hi[2] = (v & 0xF00u) | kNibExp;
    lo[3] = (v & 0xF000u) | kNibExp;
    hi[3] = (v & 0xF0000u) | kNibExp;
}

__device__ __forceinline__ uint4 ldg_w16(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldcg_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void stcg_f4(float *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.cg.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Tile of 128 weight rows (outputs) by BT tokens, and the shared / tensor
// memory that follows from it.
template <int BT>
struct Cfg {
    static_assert(BT % 32 == 0 && BT >= 32 && BT <= 256, "N of one MMA, whole 32-token chunks");
    static constexpr uint32_t kBoxBytes = BT * kBKBox * 2;  // one 64-wide box of X
    static constexpr uint32_t kXBytes = 2 * kBoxBytes;      // operand B stage: BT tokens x 128 fp16
    static constexpr uint32_t kACols = kBK / 2;             // 128 fp16 per row = 64 columns
    static constexpr uint32_t kACol0 = 256;                 // A ring after the accumulator
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kAStagesMax = (int)((kTmemCols - kACol0) / kACols);   // 4
    static constexpr int kNumBarsFor(int st) { return 2 * st + 3; }
    // After the X stages: the barriers, four words (tensor-memory address,
    // flags), then, 16-byte aligned, the tile's 256 token scales.
    static constexpr uint32_t kXsOffFor(int st) { return (8u * kNumBarsFor(st) + 16u + 15u) & ~15u; }
    static constexpr uint32_t kTailFor(int st) { return kXsOffFor(st) + 256u * 4u; }
    static constexpr int kStagesFit = (int)((kSmemBudget - 1024 - kTailFor(kAStagesMax)) / kXBytes);
    static constexpr int kStages = kStagesFit > kAStagesMax ? kAStagesMax : kStagesFit;
    static constexpr int kNumBars = kNumBarsFor(kStages);
    static constexpr uint32_t kXsOff = kXsOffFor(kStages);
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kXBytes + kTailFor(kStages);   // + alignment slack
    static constexpr int kSlotFloats = kMmaM * BT;          // one partial slot
    static constexpr uint32_t kIdesc = idesc_f16(BT);
    static_assert(kStages >= 3, "at least three stages");
    static_assert(kBoxBytes % 1024 == 0, "swizzled tiles must stay 1024-byte aligned");
    static_assert(kACol0 >= (uint32_t)BT && kACol0 + kStages * kACols <= kTmemCols, "tensor memory map");
};

// Routed experts in one launch: group g multiplies token rows [row0[g],
// row0[g] + rows[g]) of X (tokens sorted by expert) by its own weights and
// owns tiles [tile0[g], tile0[g+1]) (ceil(rows[g] / BT) token blocks times
// the output tiles, token block fastest); its row exponents are
// wexp[g * O + o].  n = 0: one matrix (Args::w, Args::scales, rows [0, M)).
constexpr int kMaxGroups = 64;
static_assert(kMaxGroups == kMoeGroupsPerLaunch, "one group table per launch");
struct Groups {
    int n;
    int tile0[kMaxGroups + 1];
    int row0[kMaxGroups];
    int rows[kMaxGroups];
    const uint8_t *w[kMaxGroups];
    const float *scales[kMaxGroups];
};

struct Args {
    float *Y;
    const uint8_t *w;     // packed weights (format-specific layout)
    const float *scales;  // fmt=4: [O, ng] group scales; fmt=7: [ceil(O/128), nbi] block scales
    unsigned *counters;   // one per output tile, zero at launch
    float *partials;      // 2 slots per block
    int M, O, gs, ng, nbi, MB, Kt;
    int tail_half;        // the last K step of every tile is 64 wide (I % 128 == 64)
    long long rowbytes;   // bytes of one weight row (fmt=4 and fmt=7; MQ4-V2: I/256 * 136)
    long long U;          // (tile, K step) units
    // Written by the preparation kernel:
    uint16_t *xh;         // fp16 copy of X [M, I]: x * 2^-F[m]
    float *xscale;        // 2^F[m] per token row (padded to whole 256-token blocks)
    int *wexp;            // E[o] per weight row (per group and row when grouped)
    int *err;
};

// The grouped kernel's arguments: the table travels only with it, so the
// single-matrix kernels keep their small argument block.
struct GroupedArgs : Args {
    Groups grp;
};
template <bool GR>
using KArgs = typename std::conditional<GR, GroupedArgs, Args>::type;

// 2^k as an f32, |k| <= 126.
__device__ __forceinline__ float exp2_int(int k) { return __int_as_float((k + 127) << 23); }

// The exponents F and E are clamped to [-kExpClamp, kExpClamp], so 2^(F-E)
// is a normal f32 and the store's scaling is one exact product.
constexpr int kExpClamp = 60;

// Largest value over the warp (fmaxf ignores NaN).
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
}

// Exponent k with 2^k * v in [2^14, 2^15) for a finite v > 0, clamped;
// 0 for v = 0 or a non-finite v.
__device__ __forceinline__ int range_exponent(float v) {
    if (!(v > 0.f && v <= 3.402823466e38f)) return 0;
    int e;
    frexpf(v, &e);   // v = f * 2^e, f in [0.5, 1)
    return max(-kExpClamp, min(kExpClamp, 15 - e));
}


// Token block and output tile of tile index t = nb * MB + mb.
__device__ __forceinline__ void tile_coords(long long t, int MB, int &mb, int &nb) {
    mb = (int)(t % MB);
    nb = (int)(t / MB);
}

// Where tile t sits: its first token row m0, the end of its token rows (the
// matrix's, or its group's), its output tile nb and its group g.
struct TileLoc {
    int m0, mend, nb, g;
};
// GR: the kernel is compiled for grouped calls (the single-matrix kernel
// keeps the matrix's bounds in the kernel arguments, no group lookup).
template <int BT, bool GR>
__device__ __forceinline__ TileLoc tile_loc(const KArgs<GR> &a, long long t) {
    TileLoc L;
    if constexpr (!GR) {
        int mb, nb;
        tile_coords(t, a.MB, mb, nb);
        L.m0 = mb * BT;
        L.mend = a.M;
        L.nb = nb;
        L.g = 0;
        return L;
    } else {
    int g = 0;
    while (g + 1 < a.grp.n && t >= a.grp.tile0[g + 1]) ++g;   // groups hold at least one tile
    const int local = (int)(t - a.grp.tile0[g]);
    const int mbg = (a.grp.rows[g] + BT - 1) / BT;
    L.m0 = a.grp.row0[g] + (local % mbg) * BT;
    L.mend = a.grp.row0[g] + a.grp.rows[g];
    L.nb = local / mbg;
    L.g = g;
    return L;
    }
}
template <bool GR>
__device__ __forceinline__ const uint8_t *group_w(const KArgs<GR> &a, int g) {
    if constexpr (GR) return a.grp.w[g];
    else return a.w;
}
template <bool GR>
__device__ __forceinline__ const float *group_scales(const KArgs<GR> &a, int g) {
    if constexpr (GR) return a.grp.scales[g];
    else return a.scales;
}

// Segment of a block's range that starts at unit u: tile t, K steps [ks, ke).
struct Seg {
    long long t;
    int ks, ke;
};
__device__ __forceinline__ Seg segment_at(long long u, long long ue, int Kt) {
    Seg g;
    g.t = u / Kt;
    g.ks = (int)(u - g.t * Kt);
    g.ke = (int)min(ue - g.t * Kt, (long long)Kt);
    return g;
}

// 16 token scales 2^F[m] from shared memory (16-byte aligned).
__device__ __forceinline__ void load_xscale16(const float *p, float (&xs)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 v = reinterpret_cast<const float4 *>(p)[j];
        xs[4 * j] = v.x;
        xs[4 * j + 1] = v.y;
        xs[4 * j + 2] = v.z;
        xs[4 * j + 3] = v.w;
    }
}

// Epilogue of one segment (tile t, K steps [ks, ke)) of this block's range,
// run by the four epilogue warps (one per tensor-memory lane quarter): wait
// for the accumulator, then either store it to Y (the whole K range is this
// block's) or go through the partial slots.  `et` numbers the 128
// participating threads.
template <int BT, bool GR>
__device__ __forceinline__ void epilogue_segment(const KArgs<GR> &a, const Seg g, const uint32_t seg, const uint32_t tmem,
                                              const int q, const int lane, const int et, const long long cta,
                                              const long long U, const long long P, const int Kt,
                                              uint64_t *acc_full, uint64_t *acc_empty, volatile uint32_t *flag,
                                              volatile uint32_t *abort, const int nslots, float *sxs,
                                              uint64_t *xs_ready) {
    using C = Cfg<BT>;
    const int row = q * 32 + lane;          // accumulator row = weight row within the tile
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const TileLoc L = tile_loc<BT, GR>(a, g.t);
    const int m0 = L.m0, o = L.nb * kMmaM + row;
    const float pe = o < a.O ? exp2_int(-a.wexp[(size_t)L.g * a.O + o]) : 0.f;   // 2^-E of this row
    // The tile's token scales into shared memory, once every epilogue warp is
    // done with the previous segment's.  With a whole tile (nslots > 1) the
    // dequantizing warps read them too, after xs_ready.
    named_sync(1, 32 * kNumEpiWarps);
    for (int i = et; i < BT; i += 32 * kNumEpiWarps) sxs[i] = a.xscale[m0 + i];
    named_sync(1, 32 * kNumEpiWarps);
    if (nslots > 1 && lane == 0) mbar_arrive(xs_ready);
    {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_backoff(acc_full, seg & 1, abort);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && lane == 0) raise_device_error(a.err, kErrTimeout);
    }
    tc_fence_after();
    auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
    };
    // Column j of the accumulator is token m0 + j; lanes hold 32
    // consecutive outputs, so each store of a warp is 128 bytes.
    auto store_chunk = [&](int c, const float (&v)[16]) {
        if (o < a.O) {
            float xs[16];
            load_xscale16(sxs + c * 16, xs);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + c * 16 + j;
                if (m < L.mend) a.Y[(size_t)m * a.O + o] = v[j] * (xs[j] * pe);
            }
        }
    };
    if (g.ks == 0 && g.ke == Kt) {
        // The whole K range is ours: straight to Y.  With nslots > 1 the
        // dequantizing warps of this lane quarter take chunks 1, 2, ... of
        // every nslots (store_tile_slice).
#pragma unroll 1
        for (int c = 0; c < BT / 16; c += nslots) {
            uint32_t r[16];
            tmem_ld16(tq + c * 16, r);
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            store_chunk(c, v);
        }
        release();
    } else {
        const long long cf = sk::first_contributor(g.t, Kt, U, P);
        const long long cl = sk::last_contributor(g.t, Kt, U, P);
        const unsigned nc = (unsigned)(cl - cf + 1);
        // Are all other contributors done already?  Then this block
        // finishes the tile from its own accumulator and their slots.
        if (et == 0) *flag = (ld_acquire_u32(&a.counters[g.t]) + 1 == nc) ? 1u : 0u;
        named_sync(1, 32 * kNumEpiWarps);
        const bool last_now = *flag != 0;
        named_sync(1, 32 * kNumEpiWarps);
        bool finish = last_now;
        if (!last_now) {
            // Park the partial sums ([token / 4][row] float4s), then count in.
            float *mine = a.partials + (size_t)sk::partial_slot(cta, g.t, Kt, U, P) * C::kSlotFloats;
#pragma unroll 1
            for (int c = 0; c < BT / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(tq + c * 16, r);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    stcg_f4(mine + ((size_t)(c * 4 + j) * kMmaM + row) * 4, r[4 * j], r[4 * j + 1],
                            r[4 * j + 2], r[4 * j + 3]);
            }
            release();
            __threadfence();
            named_sync(1, 32 * kNumEpiWarps);
            if (et == 0) *flag = (atomicAdd(&a.counters[g.t], 1u) + 1 == nc) ? 1u : 0u;
            named_sync(1, 32 * kNumEpiWarps);
            finish = *flag != 0;
            if (finish) __threadfence();
        }
        if (finish) {
            // Sum the contributors in order (the same order whichever
            // block finishes), 16 tokens at a time, then store.
            const long long slot_cf = sk::partial_slot(cf, g.t, Kt, U, P);
#pragma unroll 1
            for (int c = 0; c < BT / 16; ++c) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
                for (long long cc = cf; cc <= cl; ++cc) {
                    if (last_now && cc == cta) {   // warp-uniform
                        uint32_t own[16];
                        tmem_ld16(tq + c * 16, own);
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] += __uint_as_float(own[j]);
                        continue;
                    }
                    // Every contributor after the first starts its range
                    // inside this tile, so its slot is 2 * cc.
                    const long long slot = cc == cf ? slot_cf : 2 * cc;
                    const float *src = a.partials + (size_t)slot * C::kSlotFloats +
                                       ((size_t)(c * 4) * kMmaM + row) * 4;
                    float4 p[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) p[j] = ldcg_f4(src + (size_t)j * kMmaM * 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[4 * j] += p[j].x;
                        v[4 * j + 1] += p[j].y;
                        v[4 * j + 2] += p[j].z;
                        v[4 * j + 3] += p[j].w;
                    }
                }
                store_chunk(c, v);
            }
        }
        if (last_now) release();
    }
}

// The part of a whole tile's store that a dequantizing warp takes once its
// block has no K steps left: chunks slot, slot + nslots, ... of its lane
// quarter, after the accumulator is complete.
template <int BT, bool GR>
__device__ __forceinline__ void store_tile_slice(const KArgs<GR> &a, const Seg g, const uint32_t tmem, const int q,
                                                 const int lane, const int slot, const int nslots,
                                                 uint64_t *acc_full, volatile uint32_t *abort, const float *sxs,
                                                 uint64_t *xs_ready, const float pe) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_backoff(acc_full, 0u, abort) && mbar_wait_backoff(xs_ready, 0u, abort);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && lane == 0) raise_device_error(a.err, kErrTimeout);
    tc_fence_after();
    const TileLoc L = tile_loc<BT, GR>(a, g.t);
    const int o = L.nb * kMmaM + q * 32 + lane, m0 = L.m0;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
    for (int c = slot; c < BT / 16; c += nslots) {
        uint32_t r[16];
        tmem_ld16(tq + c * 16, r);
        if (o < a.O) {
            float xs[16];
            load_xscale16(sxs + c * 16, xs);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + c * 16 + j;
                if (m < L.mend) a.Y[(size_t)m * a.O + o] = __uint_as_float(r[j]) * (xs[j] * pe);
            }
        }
    }
    tc_fence_before();
}

template <class F, int BT, bool GR>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, KArgs<GR> a) {
    using C = Cfg<BT>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kXBytes);
    uint64_t *full = bars, *empty = bars + C::kStages;   // per stage: X bytes + dequantized A / MMA done
    uint64_t *acc_full = empty + C::kStages, *acc_empty = acc_full + 1, *xs_ready = acc_full + 2;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bars + C::kNumBars);
    volatile uint32_t *flag = tmem_slot + 1;    // epilogue broadcast: this block finishes the tile
    volatile uint32_t *abort = tmem_slot + 2;   // set by the first wait that times out
    float *sxs = reinterpret_cast<float *>(smem + C::kStages * C::kXBytes + C::kXsOff);   // the tile's token scales

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1 + kNumDeqWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kNumEpiWarps);
        mbar_init(xs_ready, kNumEpiWarps);
        *abort = 0u;
        mbar_fence_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    }
    if (warp == kWarpMma) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr((const void *)tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long P = gridDim.x, cta = blockIdx.x, U = a.U;
    const long long ub = sk::range_begin(cta, U, P), ue = sk::range_begin(cta + 1, U, P);
    const int Kt = a.Kt;
    // A range that is exactly one whole tile: the dequantizing warps, idle
    // after its last K step, help store it (5 warps per lane quarter).
    const bool whole_only = ub % Kt == 0 && ue - ub == Kt;
    constexpr int kEpiSlots = 1 + kNumDeqWarps / 4;

    if (warp == kWarpTma) {
        // The fp16 copy of X is the preparation kernel's output
        // (programmatic dependent launch): wait for it.
        griddep_wait();
        if (lane == 0) {
            uint32_t it = 0;
            for (long long u = ub; u < ue;) {
                const Seg g = segment_at(u, ue, Kt);
                const int m0 = tile_loc<BT, GR>(a, g.t).m0;
                for (int k = g.ks; k < g.ke; ++k, ++it) {
                    const uint32_t s = it % C::kStages, r = it / C::kStages;
                    const bool half = a.tail_half && k == Kt - 1;
                    if (r > 0 && !mbar_wait_or_abort(&empty[s], (r & 1) ^ 1, abort))
                        raise_device_error(a.err, kErrTimeout);
                    mbar_arrive_expect_tx(&full[s], half ? C::kBoxBytes : C::kXBytes);
                    const uint32_t st = sbase + s * C::kXBytes;
                    tma_load_2d(st, &tmX, k * kBK, m0, &full[s]);
                    if (!half) tma_load_2d(st + C::kBoxBytes, &tmX, k * kBK + kBKBox, m0, &full[s]);
                }
                u = g.t * Kt + g.ke;
            }
            // Every copy issued must have landed before the block exits.
            for (uint32_t j = it > (uint32_t)C::kStages ? it - C::kStages : 0; j < it; ++j)
                if (!mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1)) raise_device_error(a.err, kErrTimeout);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            uint32_t it = 0, seg = 0;
            for (long long u = ub; u < ue; ++seg) {
                const Seg g = segment_at(u, ue, Kt);
                if (seg > 0 && !mbar_wait_or_abort(acc_empty, (seg - 1) & 1, abort))
                    raise_device_error(a.err, kErrTimeout);
                tc_fence_after();
                for (int k = g.ks; k < g.ke; ++k, ++it) {
                    const uint32_t s = it % C::kStages, r = it / C::kStages;
                    const int nk = (a.tail_half && k == Kt - 1) ? kBKBox / 16 : kBK / 16;
                    if (!mbar_wait_or_abort(&full[s], r & 1, abort)) raise_device_error(a.err, kErrTimeout);
                    tc_fence_after();
                    const uint32_t xa = sbase + s * C::kXBytes;
                    const uint32_t at = tmem + C::kACol0 + s * C::kACols;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        if (kk < nk)
                            mma_f16_ts(tmem, at + kk * 8, sw128_desc(xa + (kk >> 2) * C::kBoxBytes + (kk & 3) * 32),
                                        C::kIdesc, (k > g.ks || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                mma_commit(acc_full);
                u = g.t * Kt + g.ke;
            }
        }
    } else if (warp < kWarpEpi + kNumEpiWarps) {
        // Epilogue of every segment of the range, in order (Y, the
        // counters and the partial slots only after the previous kernel).
        griddep_wait();
        uint32_t seg = 0;
        for (long long u = ub; u < ue; ++seg) {
            const Seg g = segment_at(u, ue, Kt);
            epilogue_segment<BT, GR>(a, g, seg, tmem, warp & 3, lane, threadIdx.x - 32 * kWarpEpi, cta, U, P, Kt,
                                    acc_full, acc_empty, flag, abort, whole_only ? kEpiSlots : 1, sxs, xs_ready);
            u = g.t * Kt + g.ke;
        }
    } else {
        // Dequantize.  Warp w may write tensor-memory lanes 32*(w % 4) ..
        // +31 (weight rows of the tile); the four warps of a lane quarter
        // split each K step into quarters kq = 0..3 of 32 weights, so every
        // sub-partition holds four dequantizing warps.
        const int q = warp & 3, kq = (warp - kWarpDeq) >> 2;
        const int R = q * 32 + lane;
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + C::kACol0 + kq * (C::kACols / 4);
        using Fetch = typename F::Fetch;
        // Fetch state: the next unit to load and the format's state of this
        // thread's row (set again when the tile changes).
        typename F::Row row;
        long long pu = ub, pt = ub / Kt;
        int pk = (int)(ub - pt * Kt);
        auto set_tile = [&]() {
            const TileLoc L = tile_loc<BT, GR>(a, pt);
            F::row_begin(a, group_w<GR>(a, L.g), group_scales<GR>(a, L.g), L.nb * kMmaM + R, kq, pk, row);
        };
        if (pu < ue) set_tile();
        auto fetch = [&](Fetch &f) {
            F::clear(f);
            if (pu < ue) {
                // The 64-wide last step of a row with I % 128 == 64 has no upper half.
                F::fetch(a, row, pk, kq, kq >= 2 && a.tail_half && pk == Kt - 1, f);
                ++pu;
                if (++pk == Kt) {
                    pk = 0;
                    ++pt;
                    if (pu < ue) set_tile();
                }
            }
        };
        // Step state: the tile of the unit being dequantized and this row's
        // 2^E there (E from the preparation kernel, read after its grid is
        // done; once per tile).
        long long st_t = ub / Kt;
        int st_k = (int)(ub - st_t * Kt), e = 0;
        float p2 = 0.f;
        auto load_exp = [&]() {
            const TileLoc L = tile_loc<BT, GR>(a, st_t);
            const int o = L.nb * kMmaM + R;
            e = o < a.O ? a.wexp[(size_t)L.g * a.O + o] : 0;
            p2 = exp2_int(e);
        };
        uint32_t it = 0;
        auto step = [&](const Fetch &cur) {
            const uint32_t s = it % C::kStages, r = it / C::kStages;
            if (r > 0 && !mbar_wait_or_abort(&empty[s], (r & 1) ^ 1, abort)) raise_device_error(a.err, kErrTimeout);
            tc_fence_after();
            uint32_t col[16];
            F::dequant(cur, p2, col);
            tmem_st16(ta + s * C::kACols, col);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
            ++it;
            if (++st_k == Kt) {   // the next unit, if any, starts a tile
                st_k = 0;
                ++st_t;
                if (ub + it < ue) load_exp();
            }
        };
        // Three register buffers used in rotation with fixed names, so a
        // buffer is read only when its loads were issued three K steps ago.
        static_assert(kPrefetch == 3, "the loop below is unrolled for three buffers");
        Fetch f0, f1, f2;
        fetch(f0);
        fetch(f1);
        fetch(f2);
        // The weights' loads are in flight; the row exponents come from the
        // preparation kernel.
        griddep_wait();
        load_exp();
        for (long long u = ub; u < ue;) {
            step(f0);
            fetch(f0);
            if (++u >= ue) break;
            step(f1);
            fetch(f1);
            if (++u >= ue) break;
            step(f2);
            fetch(f2);
            ++u;
        }
        if (whole_only)
            store_tile_slice<BT, GR>(a, segment_at(ub, ue, Kt), tmem, q, lane, 1 + kq, kEpiSlots, acc_full, abort, sxs,
                                 xs_ready, exp2_int(-e));
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

// Operand preparation.  Blocks 0 .. M-1 take one token row of X each: F[m]
// from the row's largest finite |x|, then Xh = fp16(x * 2^-F[m]) and
// xscale[m] = 2^F[m].  A row of up to kPrepRegChunks * 2048 elements is held
// in registers (all its loads in flight at once); a longer one is read twice
// (the second pass hits the cache).  The remaining blocks take eight weight
// rows each, one warp per row: E[o] from the format's bound on |w(o, .)|.
constexpr int kPrepThreads = 256;
constexpr int kPrepRegChunks = 4;   // 16-byte chunks per thread kept in registers

__device__ __forceinline__ float bf16x2_absmax(uint32_t w, float mx) {
    const float lo = fabsf(__uint_as_float(w << 16)), hi = fabsf(__uint_as_float(w & 0xFFFF0000u));
    if (lo <= 3.402823466e38f) mx = fmaxf(mx, lo);   // skips inf and NaN
    if (hi <= 3.402823466e38f) mx = fmaxf(mx, hi);
    return mx;
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v, float sc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16) * sc, hi = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(hi), "f"(lo));
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

template <class F, bool GR>
__global__ void __launch_bounds__(kPrepThreads, 8) gemm_tc_prep_kernel(KArgs<GR> a, const uint16_t *__restrict__ X,
                                                                         int I) {
    // The main kernel may launch once every block of this one runs (its
    // blocks take an SM as this kernel's leave it); it waits for this grid's
    // completion before it reads what this one writes.
    griddep_launch_dependents();
    // X may be the previous kernel's output, and that kernel may still read
    // this workspace.
    griddep_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (blockIdx.x >= (unsigned)a.M) {
        // weight row o of group g (one group when the call is not grouped)
        const int go = (blockIdx.x - a.M) * (kPrepThreads / 32) + wid;
        const int g = go / a.O, o = go - g * a.O;
        int ngroups = 1;
        if constexpr (GR) ngroups = a.grp.n;
        if (g < ngroups) {
            const int e = range_exponent(F::row_bound(a, group_w<GR>(a, g), group_scales<GR>(a, g), o, lane));
            if (lane == 0) a.wexp[go] = e;
        }
        return;
    }
    __shared__ float red[kPrepThreads / 32];
    const int m = blockIdx.x;
    uint16_t *xh = a.xh;
    float *xscale = a.xscale;
    const uint4 *src = reinterpret_cast<const uint4 *>(X + (size_t)m * I);
    uint4 *dst = reinterpret_cast<uint4 *>(xh + (size_t)m * I);
    const int n8 = I / 8;
    const bool in_regs = n8 <= kPrepRegChunks * kPrepThreads;
    uint4 v[kPrepRegChunks];
    float mx = 0.f;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kPrepRegChunks; ++j) {
            const int c = threadIdx.x + j * kPrepThreads;
            v[j] = c < n8 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kPrepRegChunks; ++j)
            mx = bf16x2_absmax(v[j].w, bf16x2_absmax(v[j].z, bf16x2_absmax(v[j].y, bf16x2_absmax(v[j].x, mx))));
    } else {
#pragma unroll 4
        for (int c = threadIdx.x; c < n8; c += kPrepThreads) {
            const uint4 u = __ldg(src + c);
            mx = bf16x2_absmax(u.w, bf16x2_absmax(u.z, bf16x2_absmax(u.y, bf16x2_absmax(u.x, mx))));
        }
    }
    mx = warp_max(mx);
    if (lane == 0) red[wid] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int k = 1; k < kPrepThreads / 32; ++k) mx = fmaxf(mx, red[k]);
    const int fm = -range_exponent(mx);
    const float sc = exp2_int(-fm);
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kPrepRegChunks; ++j) {
            const int c = threadIdx.x + j * kPrepThreads;
            if (c < n8) dst[c] = bf16x8_to_f16x8(v[j], sc);
        }
    } else {
#pragma unroll 4
        for (int c = threadIdx.x; c < n8; c += kPrepThreads) dst[c] = bf16x8_to_f16x8(__ldg(src + c), sc);
    }
    if (threadIdx.x == 0) xscale[m] = exp2_int(fm);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// The token widths compiled (MMA N).
enum TileId { kT256 = 0, kT128, kT64, kNumTiles };
constexpr int kTileBT[kNumTiles] = {256, 128, 64};

struct Plan {
    int tile, bt, MB, NB, Kt, P;
    long long T, U;
    // Workspace: tile counters, partial slots (split plans only), 2^F per
    // token (padded to whole 256-token blocks; the tail is never stored),
    // E per weight row, the fp16 copy of X; every part 256-byte aligned.
    size_t counter_bytes, xscale_off, wexp_off, xh_off, ws_bytes;
};

inline size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

inline bool plan_splits(const Plan &p) { return !(p.U % p.P == 0 && (p.U / p.P) % p.Kt == 0); }

// `groups` > 0: a grouped call (one E per group and weight row; a group's last
// token block may start anywhere, so 2^F is padded by one more block).
inline void plan_layout(Plan &p, int M, int I, int O, int groups = 0) {
    p.counter_bytes = align256((size_t)p.T * sizeof(unsigned));
    const size_t partial_bytes = plan_splits(p) ? (size_t)2 * p.P * kMmaM * p.bt * sizeof(float) : 0;
    p.xscale_off = p.counter_bytes + partial_bytes;
    p.wexp_off = p.xscale_off + align256((((size_t)M + 255) / 256 + (groups ? 1 : 0)) * 256 * sizeof(float));
    p.xh_off = p.wexp_off + align256((size_t)(groups ? groups : 1) * O * sizeof(int));
    p.ws_bytes = p.xh_off + align256((size_t)M * I * sizeof(uint16_t));
}

inline Plan make_plan(int tile, int M, int I, int O, int nsm) {
    Plan p;
    p.tile = tile;
    p.bt = kTileBT[tile];
    p.MB = (M + p.bt - 1) / p.bt;
    p.NB = (O + kMmaM - 1) / kMmaM;
    p.Kt = (I + kBK - 1) / kBK;
    p.T = (long long)p.MB * p.NB;
    p.U = p.T * p.Kt;
    // One tile per block when the tiles fit in one wave; otherwise an even
    // split of the units over all SMs.
    p.P = (int)std::min<long long>(p.T <= nsm ? p.T : nsm, p.U);
    plan_layout(p, M, I, O);
    return p;
}

// Estimated cycles of the busiest block, from measurements on GB300: a
// 128-wide K step costs ~2300 cycles with 256 tokens per tile and ~2150 with
// fewer (the dequantization of 128 x 128 weights bounds it), and a tile whose
// K range is split over blocks costs ~14000 cycles per contributor for the
// partial sums (written, then read back by the block that finishes it).
inline double plan_cost(const Plan &p) {
    const double step = p.bt == 256 ? 2300.0 : 2150.0;
    const double steps = (double)((p.U + p.P - 1) / p.P);
    const bool split = (p.U / p.P) % p.Kt != 0 || p.U % p.P != 0;
    const double contributors = (double)p.Kt / std::max(1.0, (double)(p.U / p.P)) + 1.0;
    return steps * step + (split ? 14000.0 * contributors : 0.0);
}

// Both launch shapes for every token width: one whole tile per block when
// the tiles fit in one wave, and the stream-K split over all SMs.
inline Plan choose_plan(int M, int I, int O) {
    const int nsm = num_sms();
    Plan best = make_plan(0, M, I, O, nsm);
    double best_cost = plan_cost(best);
    for (int t = 0; t < kNumTiles; ++t) {
        for (int mode = 0; mode < 2; ++mode) {
            Plan p = make_plan(t, M, I, O, nsm);
            if (mode == 1) {
                if (p.T >= nsm) continue;   // already the split over all SMs
                p.P = (int)std::min<long long>(nsm, p.U);
                plan_layout(p, M, I, O);
            }
            const double c = plan_cost(p);
            if (c < best_cost) {
                best = p;
                best_cost = c;
            }
        }
    }
    return best;
}

template <class F, int BT, bool GR>
int launch_tile(const Plan &p, const CUtensorMap &tmX, const KArgs<GR> &args, cudaStream_t st) {
    using C = Cfg<BT>;
    // The shared-memory limit is an attribute of the kernel in the current
    // context: set once per context.
    set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc_kernel<F, BT, GR>), (int)C::kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, gemm_tc_kernel<F, BT, GR>, tmX, args);
    count_launch();
    return check_launch(F::kName);
}

// Launch plan `p` for X [M, I] bf16 and Y [M, O] f32; `args` carries the
// format's fields (w, scales, gs, ng, nbi) and is completed here.
template <class F, bool GR = false>
int launch_plan(const Plan &p, float *Y, const uint16_t *X, KArgs<GR> args, int M, int I, int O, void *ws,
                cudaStream_t st) {
    auto encode = encode_fn();
    if (!encode) {
        set_error_detail("%s: cuTensorMapEncodeTiled is not available from the driver", F::kName);
        return kECuda;
    }
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    args.xscale = reinterpret_cast<float *>(wsb + p.xscale_off);
    args.wexp = reinterpret_cast<int *>(wsb + p.wexp_off);
    args.xh = reinterpret_cast<uint16_t *>(wsb + p.xh_off);
    CUtensorMap tmX;
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)I * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBKBox, (cuuint32_t)p.bt};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, args.xh, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error_detail("%s: tensor map of X refused (CUresult %d)", F::kName, (int)r);
        return kECuda;
    }
    args.Y = Y;
    args.counters = static_cast<unsigned *>(ws);
    args.partials = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) + p.counter_bytes);
    args.M = M;
    args.O = O;
    args.MB = p.MB;
    args.Kt = p.Kt;
    args.tail_half = (I % kBK) != 0 ? 1 : 0;
    args.U = p.U;
    args.err = device_error_word();
    // Tile counters are only read when a tile's K range is split over blocks.
    if (plan_splits(p) && cudaMemsetAsync(ws, 0, (size_t)p.T * sizeof(unsigned), st) != cudaSuccess)
        return check_launch(F::kName);
    {
        cudaLaunchConfig_t cfg = {};
        long long wrows = O;
        if constexpr (GR) wrows *= args.grp.n;
        cfg.gridDim = dim3((unsigned)(M + (wrows + kPrepThreads / 32 - 1) / (kPrepThreads / 32)));
        cfg.blockDim = dim3(kPrepThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, gemm_tc_prep_kernel<F, GR>, args, X, I);
        count_launch();
        const int rc = check_launch(F::kName);
        if (rc != kOk) return rc;
    }
    switch (p.tile) {
        case kT256: return launch_tile<F, 256, GR>(p, tmX, args, st);
        case kT128: return launch_tile<F, 128, GR>(p, tmX, args, st);
        default: return launch_tile<F, 64, GR>(p, tmX, args, st);
    }
}

// Plan of a grouped call: n groups of rows[g] > 0 token rows, M rows in all.
// Every token block of a group dequantizes the group's whole weight tile, so
// the tile width minimises the token blocks times the cost of a K step
// (plan_cost's per-step figures); the tiles of all groups are one range,
// whole tiles per block when they fit in one wave, else split evenly over
// the SMs (stream-K).
inline Plan group_plan(const int *rows, int n, int M, int I, int O) {
    const int nsm = num_sms();
    int best_tile = kT256;
    double best = 0.0;
    for (int t = 0; t < kNumTiles; ++t) {
        const int bt = kTileBT[t];
        long long blocks = 0;
        for (int g = 0; g < n; ++g) blocks += (rows[g] + bt - 1) / bt;
        const double c = (double)blocks * (bt == 256 ? 2300.0 : 2150.0);
        if (t == 0 || c < best) {
            best = c;
            best_tile = t;
        }
    }
    Plan p;
    p.tile = best_tile;
    p.bt = kTileBT[p.tile];
    p.NB = (O + kMmaM - 1) / kMmaM;
    p.Kt = (I + kBK - 1) / kBK;
    p.MB = 0;
    p.T = 0;
    for (int g = 0; g < n; ++g) p.T += (long long)((rows[g] + p.bt - 1) / p.bt) * p.NB;
    p.U = p.T * p.Kt;
    p.P = (int)std::min<long long>(p.T <= nsm ? p.T : nsm, p.U);
    plan_layout(p, M, I, O, n);
    return p;
}

// A grouped call on the tensor cores: `args` carries the format's fields
// except the weights; group g is rows [row0[g], row0[g] + rows[g]) of X and
// Y with weights w[g] / scales[g] (rows[g] > 0, n <= kMaxGroups).
template <class F>
int launch_grouped(float *Y, const uint16_t *X, const Args &base, const int *row0, const int *rows,
                   const uint8_t *const *w, const float *const *scales, int n, int M, int I, int O, void *ws,
                   size_t ws_bytes, cudaStream_t st) {
    const Plan p = group_plan(rows, n, M, I, O);
    if (ws == nullptr || ws_bytes < p.ws_bytes) {
        set_error_detail("%s: this grouped call needs a workspace of %zu bytes (got %zu)", F::kName, p.ws_bytes,
                         ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    GroupedArgs args{};
    static_cast<Args &>(args) = base;
    args.grp.n = n;
    int t = 0;
    for (int g = 0; g < n; ++g) {
        args.grp.tile0[g] = t;
        args.grp.row0[g] = row0[g];
        args.grp.rows[g] = rows[g];
        args.grp.w[g] = w[g];
        args.grp.scales[g] = scales[g];
        t += ((rows[g] + p.bt - 1) / p.bt) * p.NB;
    }
    args.grp.tile0[n] = t;
    return launch_plan<F, true>(p, Y, X, args, M, I, O, ws, st);
}

}  // namespace tc
}  // namespace qg

