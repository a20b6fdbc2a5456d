// gemm_mq4_tc.cuh -- batched-prefill dequant-GEMM on the tensor cores for
// the 136-byte MQ4 block formats: the format policy of the kernel in
// gemm_tc.cuh, templated on the header kind HK (instantiated by
// gemm_mq4v2_tc.cu, gemm_mq4v1_tc.cu, gemm_mq4c_tc.cu).
//
// hipfire "MQ4 V2", sections 1b, 1e, 2 and 4: 136 bytes per 256 weights, 128
// bytes of nibbles at [8,136), w_j = q_j * scale + zero, the header by kind:
//   HK = 44  MQ4-V2: fp16 scale | fp16 zero dword per 128-weight half
//   HK = 45  MQ4C pad: one fp16 scale | fp16 zero dword at [0,4)
//   HK = 13  MQ4 v1: f32 scale at [0,4), f32 zero at [4,8)
// Here each weight is formed in f32 with one rounding (a fused multiply-add
// of the exact q_j, scale and zero), scaled by the row's power of two and
// rounded to fp16 for the MMA.
//
// A 128-wide K step is exactly one half of a block, so one dequantizing
// thread takes one header and 16 payload bytes (32 weights) per step.
// Blocks are 136 bytes, so payload addresses are only 8-byte aligned: two
// 8-byte loads.
#pragma once
#include "gemm_tc.cuh"

namespace qg {
namespace tc {

static __device__ __forceinline__ uint2 ldg_w8(const uint8_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

static __device__ __forceinline__ float f16_to_f32(uint32_t h) {
    float f;
    asm("{.reg .b16 t, u; mov.b32 {t, u}, %1; cvt.f32.f16 %0, t;}" : "=f"(f) : "r"(h));
    return f;
}

// Header of a block by kind: its bytes (the first 8 of the block, read as
// two words), the header of K step pk's half, and its scale and zero.
template <int HK>
struct MqHead;
template <>
struct MqHead<44> {   // fp16 pair per 128-weight half
    typedef uint32_t Raw;
    static __device__ __forceinline__ Raw of_step(const uint8_t *blk, int pk) {
        return __ldg(reinterpret_cast<const unsigned *>(blk) + (pk & 1));
    }
    static __device__ __forceinline__ float scale(Raw h) { return f16_to_f32(h); }
    static __device__ __forceinline__ float zero(Raw h) { return f16_to_f32(h >> 16); }
    static __device__ __forceinline__ float block_bound(uint2 w) {
        return fmaxf(fabsf(f16_to_f32(w.x >> 16)) + 15.f * fabsf(f16_to_f32(w.x)),
                     fabsf(f16_to_f32(w.y >> 16)) + 15.f * fabsf(f16_to_f32(w.y)));
    }
};
template <>
struct MqHead<45> : MqHead<44> {   // one fp16 pair for the block, zero pad
    static __device__ __forceinline__ Raw of_step(const uint8_t *blk, int) {
        return __ldg(reinterpret_cast<const unsigned *>(blk));
    }
    static __device__ __forceinline__ float block_bound(uint2 w) {
        return fabsf(f16_to_f32(w.x >> 16)) + 15.f * fabsf(f16_to_f32(w.x));
    }
};
template <>
struct MqHead<13> {   // f32 scale, f32 zero for the block
    typedef uint2 Raw;
    static __device__ __forceinline__ Raw of_step(const uint8_t *blk, int) {
        return __ldg(reinterpret_cast<const uint2 *>(blk));
    }
    static __device__ __forceinline__ float scale(Raw h) { return __uint_as_float(h.x); }
    static __device__ __forceinline__ float zero(Raw h) { return __uint_as_float(h.y); }
    static __device__ __forceinline__ float block_bound(uint2 w) {
        return fabsf(__uint_as_float(w.y)) + 15.f * fabsf(__uint_as_float(w.x));
    }
};

template <int HK>
struct PolicyMq4 {
    typedef MqHead<HK> Hdr;
    static constexpr const char *kName = HK == 44 ? "qgemm_mq4v2 (tensor-core kernel)"
                                         : HK == 45 ? "qgemm_mq4c (tensor-core kernel)"
                                                    : "qgemm_mq4v1 (tensor-core kernel)";
    static constexpr int kBlockBytes = 136;
    // Bound on |w| over row o, q in 0..15: max over the row's headers of
    // |zero| + 15 |scale|.  Called by a whole warp.
    static __device__ __forceinline__ float row_bound(const Args &a, const uint8_t *w, const float *, int o,
                                                      int lane) {
        const uint8_t *row = w + (size_t)o * (size_t)a.rowbytes;
        const int nb = a.Kt >> 1;
        float b = 0.f;
#pragma unroll 4
        for (int k = lane; k < nb; k += 32)
            b = fmaxf(b, Hdr::block_bound(__ldg(reinterpret_cast<const uint2 *>(row + (size_t)k * kBlockBytes))));
        return warp_max(b);
    }
    struct Fetch {
        uint4 q;
        typename Hdr::Raw h;   // header of the step's weights
    };
    struct Row {
        const uint8_t *b;   // this row's blocks; the payload quarter kq added
    };
    static __device__ __forceinline__ void row_begin(const Args &a, const uint8_t *w, const float *, int o, int kq,
                                                     int, Row &r) {
        r.b = o < a.O ? w + (size_t)o * (size_t)a.rowbytes + 16 * kq : nullptr;
    }
    static __device__ __forceinline__ void clear(Fetch &f) {
        f.q = make_uint4(0u, 0u, 0u, 0u);
        f.h = typename Hdr::Raw{};   // scale 0, zero 0
    }
    static __device__ __forceinline__ void fetch(const Args &, Row &r, int pk, int kq, bool, Fetch &f) {
        if (r.b) {
            const int h = pk & 1;
            const uint8_t *blk = r.b + (size_t)(pk >> 1) * kBlockBytes;   // kq * 16 bytes past the block
            const uint2 lo = ldg_w8(blk + 8 + 64 * h);
            const uint2 hi = ldg_w8(blk + 16 + 64 * h);
            f.q = make_uint4(lo.x, lo.y, hi.x, hi.y);
            f.h = Hdr::of_step(blk - 16 * kq, pk);
        }
    }
    // q -> (q * scale + zero) * 2^E: bias -2^23 at every position, then one
    // fused multiply-add with (scale * 2^E * 16^-p, zero * 2^E).
    static __device__ __forceinline__ void dequant(const Fetch &f, float p2, uint32_t (&col)[16]) {
        constexpr uint64_t kBias = 0xCB000000CB000000ull;
        const float z = Hdr::zero(f.h) * p2;
        const NibPairs sp = nib_scale_pairs(Hdr::scale(f.h) * p2);
        const uint64_t z2 = f32_pair(z, z);
        const uint32_t wv[4] = {f.q.x, f.q.y, f.q.z, f.q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t lo[4], hi[4];
            nib_positions(wv[j], lo, hi);
#pragma unroll
            for (int p = 0; p < 4; ++p) col[4 * j + p] = nib_add_fma(lo[p], hi[p], kBias, sp.v[p], z2);
        }
    }
};

}  // namespace tc

// The format fixes I % 256 == 0 and 8-byte aligned blocks (checked by the
// entry point); the tensor-core kernel also wants a TMA-aligned X.
inline size_t ws_gemm_mq4(int M, int I, int O) {
    if (I % 256 != 0) return 0;
    return tc::choose_plan(M, I, O).ws_bytes;
}

template <int HK>
int run_gemm_mq4_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                    size_t ws_bytes, cudaStream_t st, bool *taken, const char *name) {
    *taken = false;
    if ((uintptr_t)X % 16 != 0 || I % 256 != 0) return kOk;
    *taken = true;
    const tc::Plan p = tc::choose_plan(M, I, O);
    if (ws == nullptr || ws_bytes < p.ws_bytes) {
        set_error_detail("%s: this shape needs a workspace of %zu bytes (got %zu)", name, p.ws_bytes,
                         ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    tc::Args args{};
    args.w = blocks;
    args.rowbytes = (long long)(I / 256) * tc::PolicyMq4<HK>::kBlockBytes;
    return tc::launch_plan<tc::PolicyMq4<HK>>(p, Y, X, args, M, I, O, ws, st);
}

inline size_t ws_gemm_moe_mq4_impl(const int *rows, int n, int M, int I, int O) {
    if (I % 256 != 0) return 0;
    return tc::group_plan(rows, n, M, I, O).ws_bytes;
}

template <int HK>
int run_gemm_moe_mq4_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                        int n, int M, int I, int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    *taken = false;
    if ((uintptr_t)X % 16 != 0 || I % 256 != 0) return kOk;
    for (int g = 0; g < n; ++g)
        if ((uintptr_t)w[g] % 8 != 0) return kOk;
    *taken = true;
    const float *none[tc::kMaxGroups] = {};
    tc::Args args{};
    args.rowbytes = (long long)(I / 256) * tc::PolicyMq4<HK>::kBlockBytes;
    return tc::launch_grouped<tc::PolicyMq4<HK>>(Y, X, args, row0, rows, w, none, n, M, I, O, ws, ws_bytes, st);
}

}  // namespace qg
