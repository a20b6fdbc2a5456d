// gemm_mq4v2_tc.cu -- MQ4-V2 (hipfire qt=44) batched-prefill dequant-GEMM on
// the tensor cores: the format policy of the kernel in gemm_tc.cuh.
//
// hipfire "MQ4 V2", sections 2 and 4: 136 bytes per 256 weights, a header
// dword per 128-weight half (fp16 scale low, fp16 zero high) and 128 bytes
// of nibbles; w_j = q_j * scale[h] + zero[h].  Here each weight is formed in
// f32 with one rounding (a fused multiply-add of the exact q_j, scale and
// zero), scaled by the row's power of two and rounded to fp16 for the MMA.
//
// A 128-wide K step is exactly one half of a block, so one dequantizing
// thread takes one header dword and 16 payload bytes (32 weights) per step.
// Blocks are 136 bytes, so payload addresses are only 8-byte aligned: two
// 8-byte loads.
#include "gemm_tc.cuh"

namespace qg {
namespace tc {
namespace {

__device__ __forceinline__ uint2 ldg_w8(const uint8_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ float f16_to_f32(uint32_t h) {
    float f;
    asm("{.reg .b16 t, u; mov.b32 {t, u}, %1; cvt.f32.f16 %0, t;}" : "=f"(f) : "r"(h));
    return f;
}

struct PolicyMq4v2 {
    static constexpr const char *kName = "qgemm_mq4v2 (tensor-core kernel)";
    static constexpr int kBlockBytes = 136;
    // Bound on |w| over row o, q in 0..15: max over the halves of
    // |zero| + 15 |scale|.  Called by a whole warp.
    static __device__ __forceinline__ float row_bound(const Args &a, int o, int lane) {
        const uint8_t *row = a.w + (size_t)o * (size_t)a.rowbytes;
        const int nb = a.Kt >> 1;
        float b = 0.f;
#pragma unroll 4
        for (int k = lane; k < nb; k += 32) {
            const uint2 h = __ldg(reinterpret_cast<const uint2 *>(row + (size_t)k * kBlockBytes));
            b = fmaxf(b, fabsf(f16_to_f32(h.x >> 16)) + 15.f * fabsf(f16_to_f32(h.x)));
            b = fmaxf(b, fabsf(f16_to_f32(h.y >> 16)) + 15.f * fabsf(f16_to_f32(h.y)));
        }
        return warp_max(b);
    }
    struct Fetch {
        uint4 q;
        uint32_t h;   // header of the half: fp16 scale (low), fp16 zero (high)
    };
    struct Row {
        const uint8_t *b;   // this row's blocks; the payload quarter kq added
    };
    static __device__ __forceinline__ void row_begin(const Args &a, int o, int kq, int, Row &r) {
        r.b = o < a.O ? a.w + (size_t)o * (size_t)a.rowbytes + 16 * kq : nullptr;
    }
    static __device__ __forceinline__ void clear(Fetch &f) {
        f.q = make_uint4(0u, 0u, 0u, 0u);
        f.h = 0u;   // scale 0, zero 0
    }
    static __device__ __forceinline__ void fetch(const Args &, Row &r, int pk, int kq, bool, Fetch &f) {
        if (r.b) {
            const int h = pk & 1;
            const uint8_t *blk = r.b + (size_t)(pk >> 1) * kBlockBytes;   // kq * 16 bytes past the block
            const uint2 lo = ldg_w8(blk + 8 + 64 * h);
            const uint2 hi = ldg_w8(blk + 16 + 64 * h);
            f.q = make_uint4(lo.x, lo.y, hi.x, hi.y);
            f.h = __ldg(reinterpret_cast<const unsigned *>(blk - 16 * kq + 4 * h));
        }
    }
    // q -> (q * scale + zero) * 2^E: bias -2^23 at every position, then one
    // fused multiply-add with (scale * 2^E * 16^-p, zero * 2^E).
    static __device__ __forceinline__ void dequant(const Fetch &f, float p2, uint32_t (&col)[16]) {
        constexpr uint64_t kBias = 0xCB000000CB000000ull;
        const float z = f16_to_f32(f.h >> 16) * p2;
        const NibPairs sp = nib_scale_pairs(f16_to_f32(f.h) * p2);
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

}  // namespace
}  // namespace tc

// The format fixes I % 256 == 0 and 8-byte aligned blocks (checked by the
// entry point); the tensor-core kernel also wants a TMA-aligned X.
size_t ws_gemm_mq4v2(int M, int I, int O) {
    if (I % 256 != 0) return 0;
    return tc::choose_plan(M, I, O).ws_bytes;
}

int run_gemm_mq4v2_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                      size_t ws_bytes, cudaStream_t st, bool *taken) {
    *taken = false;
    if ((uintptr_t)X % 16 != 0 || I % 256 != 0) return kOk;
    *taken = true;
    const tc::Plan p = tc::choose_plan(M, I, O);
    if (ws == nullptr || ws_bytes < p.ws_bytes) {
        set_error_detail("qgemm_mq4v2: this shape needs a workspace of %zu bytes (got %zu)", p.ws_bytes,
                         ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    tc::Args args{};
    args.w = blocks;
    args.rowbytes = (long long)(I / 256) * tc::PolicyMq4v2::kBlockBytes;
    return tc::launch_plan<tc::PolicyMq4v2>(p, Y, X, args, M, I, O, ws, st);
}

}  // namespace qg
