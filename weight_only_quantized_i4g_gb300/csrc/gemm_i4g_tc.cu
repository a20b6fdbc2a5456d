// gemm_i4g_tc.cu -- fmt=4 (grouped int4) batched-prefill dequant-GEMM on the
// tensor cores: the format policy of the kernel in gemm_tc.cuh.
//
// colibri PR #457 "metal: grouped-int4 (fmt=4) GEMV support + two latent
// fmt=4 fixes", section 4: the large-batch path computes the same grouped
// product as the GEMV, Y[m, o] = sum_i (n(o,i) - 8) * scale[o, i/gs] * X[m, i];
// here each weight (n - 8) * scale is rounded once to f32 and, scaled by the
// row's power of two, to fp16 for the MMA.
//
// Layout (section 11): row o holds (I+1)/2 bytes, weight i in byte i/2 (low
// nibble for even i); scales f32 [O, ceil(I/gs)].  One dequantizing thread
// takes 32 weights of its row per K step: one 16-byte load and one scale
// (gs % 32 == 0 keeps the 32 weights inside one group).
#include "gemm_tc.cuh"

namespace qg {
namespace tc {
namespace {

struct PolicyI4G {
    static constexpr const char *kName = "qgemm_i4g (tensor-core kernel)";
    // Bound on |w| over row o, |n - 8| <= 8: 8 max_g |scale[o, g]|.  Called by
    // a whole warp; every lane gets the result.
    static __device__ __forceinline__ float row_bound(const Args &a, const uint8_t *, const float *scales, int o,
                                                      int lane) {
        const float *src = scales + (size_t)o * a.ng;
        float b = 0.f;
#pragma unroll 4
        for (int g = lane; g < a.ng; g += 32) b = fmaxf(b, fabsf(__ldg(src + g)));
        return 8.f * warp_max(b);
    }
    struct Fetch {
        uint4 q;
        float s;
    };
    // Row pointers and the scale group of this thread's 32-weight quarter,
    // advanced without divisions (one division per tile change).
    struct Row {
        const uint8_t *w;
        const float *s;
        int gi, gr;
    };
    static __device__ __forceinline__ void row_begin(const Args &a, const uint8_t *w, const float *scales, int o,
                                                     int kq, int pk, Row &r) {
        const bool in = o < a.O;
        r.w = in ? w + (size_t)o * (size_t)(a.rowbytes) + kq * 16 : nullptr;
        r.s = in ? scales + (size_t)o * a.ng : nullptr;
        const int gq = a.gs / 32, u0 = 4 * pk + kq;
        r.gi = u0 / gq;
        r.gr = u0 - r.gi * gq;
    }
    static __device__ __forceinline__ void clear(Fetch &f) {
        f.q = make_uint4(0u, 0u, 0u, 0u);
        f.s = 0.f;
    }
    static __device__ __forceinline__ void fetch(const Args &a, Row &r, int pk, int, bool skip, Fetch &f) {
        if (r.w && !skip) {
            f.q = ldg_w16(r.w + pk * 64);
            f.s = __ldg(r.s + r.gi);
        }
        const int gq = a.gs >> 5;
        r.gr += 4;
        while (r.gr >= gq) {
            r.gr -= gq;
            ++r.gi;
        }
    }
    // Weight n -> (n - 8) * scale * 2^E: bias -(2^23 + 8*16^p) per position.
    static __device__ __forceinline__ void dequant(const Fetch &f, float p2, uint32_t (&col)[16]) {
        constexpr uint64_t kB01 = 0xCB000080CB000008ull, kB23 = 0xCB008000CB000800ull;
        constexpr uint64_t kB42 = 0xCB000800CB080000ull, kB34 = 0xCB080000CB008000ull;
        const NibPairs sp = nib_scale_pairs(f.s * p2);
        const uint32_t wv[4] = {f.q.x, f.q.y, f.q.z, f.q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t lo[4], hi[4];
            nib_positions(wv[j], lo, hi);
            col[4 * j + 0] = nib_add_mul(lo[0], hi[0], kB01, sp.v[0]);
            col[4 * j + 1] = nib_add_mul(lo[1], hi[1], kB23, sp.v[1]);
            col[4 * j + 2] = nib_add_mul(lo[2], hi[2], kB42, sp.v[2]);
            col[4 * j + 3] = nib_add_mul(lo[3], hi[3], kB34, sp.v[3]);
        }
    }
};

}  // namespace
}  // namespace tc

// Shapes the tensor-core kernel takes: K in whole 64-steps (a last step of 64),
// every 32-weight quarter step inside one scale group, a 16-byte aligned w
// (its rows then start on 16-byte boundaries too) and a TMA-aligned X.
static bool gemm_i4g_tc_ok(const uint16_t *X, const uint8_t *w, int I, int gs) {
    return I % tc::kBKBox == 0 && gs % 32 == 0 && (uintptr_t)X % 16 == 0 && (uintptr_t)w % 16 == 0;
}

size_t ws_gemm_i4g(int M, int I, int O, int gs) {
    if (I % tc::kBKBox != 0 || gs % 32 != 0) return 0;
    return tc::choose_plan(M, I, O).ws_bytes;
}

int run_gemm_i4g_tc(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I, int O,
                    int gs, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken) {
    *taken = false;
    if (!gemm_i4g_tc_ok(X, w, I, gs)) return kOk;
    *taken = true;
    const tc::Plan p = tc::choose_plan(M, I, O);
    if (ws == nullptr || ws_bytes < p.ws_bytes) {
        set_error_detail("qgemm_i4g: this shape needs a workspace of %zu bytes (got %zu)", p.ws_bytes,
                         ws == nullptr ? (size_t)0 : ws_bytes);
        return kEWorkspace;
    }
    tc::Args args{};
    args.w = w;
    args.scales = scales;
    args.gs = gs;
    args.ng = (I + gs - 1) / gs;
    args.rowbytes = I / 2;
    return tc::launch_plan<tc::PolicyI4G>(p, Y, X, args, M, I, O, ws, st);
}

size_t ws_gemm_moe_i4g(const int *rows, int n, int M, int I, int O, int gs) {
    if (I % tc::kBKBox != 0 || gs % 32 != 0) return 0;
    return tc::group_plan(rows, n, M, I, O).ws_bytes;
}

int run_gemm_moe_i4g_tc(float *Y, const uint16_t *X, const int *row0, const int *rows, const uint8_t *const *w,
                        const float *const *scales, int n, int M, int I, int O, int gs, void *ws, size_t ws_bytes,
                        cudaStream_t st, bool *taken) {
    *taken = false;
    for (int g = 0; g < n; ++g)
        if (!gemm_i4g_tc_ok(X, w[g], I, gs)) return kOk;
    *taken = true;
    tc::Args args{};
    args.gs = gs;
    args.ng = (I + gs - 1) / gs;
    args.rowbytes = I / 2;
    return tc::launch_grouped<tc::PolicyI4G>(Y, X, args, row0, rows, w, scales, n, M, I, O, ws, ws_bytes, st);
}

}  // namespace qg
