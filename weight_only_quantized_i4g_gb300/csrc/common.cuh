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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

}  // namespace qg
