// common.cuh -- device helpers shared by the GEMV / GEMM kernels of libqgemv.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Streaming loads: weights are read exactly once per call, so they bypass L1
// (no_allocate) and ask L2 for whole 256-byte lines.
// ---------------------------------------------------------------------------
template <int NW> struct Words { uint32_t w[NW]; };

template <int NW>
__device__ __forceinline__ Words<NW> ld_stream(const void *p);

template <>
__device__ __forceinline__ Words<4> ld_stream<4>(const void *p) {
    Words<4> r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "l"(p));
    return r;
}
template <>
__device__ __forceinline__ Words<2> ld_stream<2>(const void *p) {
    Words<2> r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];"
        : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
    return r;
}
template <>
__device__ __forceinline__ Words<1> ld_stream<1>(const void *p) {
    Words<1> r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
    return r;
}

__device__ __forceinline__ float ld_nc_f32(const float *p) {
    float v;
    asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// UE8M0 (OCP MX E8M0): the byte e means 2^(e - 127), e = 0xFF is NaN.  Every
// value is an f32 value: e in 1..254 is the normal 2^(e-127) (the bits e << 23),
// e = 0 the subnormal 2^-127 (mantissa bit 22).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
    return __uint_as_float(e == 0u ? 0x00400000u : e == 255u ? 0x7FC00000u : e << 23);
}

// fmt=7 block-scale encodings: the stored type, its value and the entry
// points' names.  f32 is the encoding colibri PR #528 implements; UE8M0 (one
// byte per block, a power-of-two exponent) the DeepSeek-V4 encoding the same
// page names as the follow-up.
struct ScaleF32 {
    typedef float T;
    static constexpr const char *kGemv = "qgemv_fp8b128";
    static constexpr const char *kGemm = "qgemm_fp8b128";
    static constexpr const char *kGemmTc = "qgemm_fp8b128 (tensor-core kernel)";
    static constexpr const char *kGemmGeneral = "qgemm_fp8b128 (general kernel)";
    __device__ static float get(const float *p, size_t i) { return ld_nc_f32(p + i); }
};
struct ScaleE8M0 {
    typedef uint8_t T;
    static constexpr const char *kGemv = "qgemv_fp8ue8m0";
    static constexpr const char *kGemm = "qgemm_fp8ue8m0";
    static constexpr const char *kGemmTc = "qgemm_fp8ue8m0 (tensor-core kernel)";
    static constexpr const char *kGemmGeneral = "qgemm_fp8ue8m0 (general kernel)";
    __device__ static float get(const uint8_t *p, size_t i) { return e8m0_to_f32(__ldg(p + i)); }
};
__device__ __forceinline__ uint32_t ld_nc_u32(const void *p) {
    uint32_t v;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// bf16 bit pattern -> f32 (exact: bf16 is the top half of a binary32)
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// IEEE binary16 bit pattern -> f32 (exact; hardware conversion)
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    float f;
    asm("{.reg .f16 t; mov.b16 t, %1; cvt.f32.f16 %0, t;}" : "=f"(f) : "h"(h));
    return f;
}

// ---------------------------------------------------------------------------
// Block-wide reduction of N per-thread partial sums (N a power of two <= 32).
// Warp stage: a reduce-scatter butterfly -- at each xor distance a lane keeps
// half of its values and sends the other half, so N values cost N-1 shuffles
// instead of 5N.  Afterwards lane l holds the warp total of value
// (l >> (5 - log2 N)) & (N-1).  Block stage: one representative lane per
// value writes to shared memory; after one barrier, thread v < N adds the
// per-warp totals of value v.  `red` is double-buffered by the caller's
// batch parity, so one barrier per batch suffices.
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
#pragma unroll
    for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            float send = upper ? v[i] : v[i + n / 2];
            float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
    // remaining distances: plain butterfly on the single surviving value
    constexpr int kLog = (N == 1) ? 0 : (N == 2) ? 1 : (N == 4) ? 2 : (N == 8) ? 3 : (N == 16) ? 4 : 5;
#pragma unroll
    for (int off = 16 >> kLog; off >= 1; off >>= 1)
        r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

template <int N>
__device__ __forceinline__ int reduce_scatter_index(int lane) {
    constexpr int kLog = (N == 1) ? 0 : (N == 2) ? 1 : (N == 4) ? 2 : (N == 8) ? 3 : (N == 16) ? 4 : 5;
    return (lane >> (5 - kLog)) & (N - 1);
}

// Index guards of the bounds-checking build (compiled with -DQG_BOUNDS_CHECK,
// the stand-in for a memory checker): a guard whose condition is false records
// QG_EBOUNDS in the device error word `err` and the access it protects is
// skipped.  In the normal build every guard is the constant true and costs
// nothing.
constexpr int kErrBounds = -9;
#ifdef QG_BOUNDS_CHECK
__device__ __forceinline__ bool qg_guard(bool ok, int *err) {
    if (!ok && err != nullptr) atomicExch(err, kErrBounds);
    return ok;
}
#else
__device__ __forceinline__ constexpr bool qg_guard(bool, int *) { return true; }
#endif

// Timeline stamps of the stamps build (compiled with -DQG_STAMPS, for
// profiling): block b = blockIdx.x + gridDim.x * blockIdx.y (b <
// kStampBlocks) of a staged or warp-MMA decode GEMV writes kStampSlots 64-bit
// words at stamp area + b * kStampSlots: clock64 when the block starts
// (kStEntry), when its wait for the previous kernel returned (kStWaitDone),
// when its activations were ready (kStXReady), when its first row batch had
// landed (kStFirstBatch; on the warp-MMA kernel after the activation setup),
// when its consumers finished the last batch (kStConsumed) and when its last
// output was stored (kStStored); the number of row batches it ran
// (kStBatches) and the global timer in ns at its start (kStGlobalEntry).  The
// stamp area follows the device error word `err` (in that build its symbol is
// an array).  Routed-expert launches (grid z) are not told apart.  In other
// builds the calls compile to nothing.
constexpr int kStampSlots = 8, kStampBlocks = 2048, kStampOffsetInts = 4;
enum StampSlot {
    kStEntry = 0, kStWaitDone = 1, kStXReady = 2, kStFirstBatch = 3, kStConsumed = 4, kStStored = 5,
    kStBatches = 6, kStGlobalEntry = 7
};
#ifdef QG_STAMPS
__device__ __forceinline__ void qg_stamp_put(int *err, int slot, unsigned long long v) {
    const unsigned b = blockIdx.x + gridDim.x * blockIdx.y;
    if (err != nullptr && b < (unsigned)kStampBlocks)
        reinterpret_cast<unsigned long long *>(err + kStampOffsetInts)[(size_t)b * kStampSlots + slot] = v;
}
__device__ __forceinline__ void qg_stamp(int *err, int slot) { qg_stamp_put(err, slot, (unsigned long long)clock64()); }
__device__ __forceinline__ void qg_stamp_entry(int *err) {
    unsigned long long g;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g));
    qg_stamp_put(err, kStEntry, (unsigned long long)clock64());
    qg_stamp_put(err, kStGlobalEntry, g);
}
#else
__device__ __forceinline__ void qg_stamp_put(int *, int, unsigned long long) {}
__device__ __forceinline__ void qg_stamp(int *, int) {}
__device__ __forceinline__ void qg_stamp_entry(int *) {}
#endif

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

}  // namespace qg
