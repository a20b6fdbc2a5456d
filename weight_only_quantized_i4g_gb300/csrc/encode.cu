// encode.cu -- weight preparation on the device: the fmt=4 symmetric group
// quantizer, the MQ4-V2 encoder and the signed FWHT-256 rotation.  These run
// once per weight tensor (or once per token for the activation rotation of
// the MQ line), not inside the GEMV.
//
// Every rounding step is a single IEEE binary32 operation in round-to-
// nearest-even (__fdiv_rn, __fsub_rn, rintf, cvt.rn.f16.f32), so the bytes
// produced depend only on the binary32 inputs.
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace qg {

// ---------------------------------------------------------------------------
// fmt=4 quantizer: one thread per (row, group).
//   scale = max|w| / 7;  q = clamp(rint(w / scale), -8, 7);  nibble = q + 8
// ---------------------------------------------------------------------------
__global__ void quantize_i4g_kernel(uint8_t *__restrict__ wq, float *__restrict__ scales,
                                    const float *__restrict__ w, int O, int I, int gs) {
    const int ng = (I + gs - 1) / gs;
    const size_t rb = ((size_t)I + 1) / 2;
    const size_t total = (size_t)O * ng;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const int o = (int)(t / ng);
        const int g = (int)(t - (size_t)o * ng);
        const int i0 = g * gs;
        const int i1 = i0 + gs < I ? i0 + gs : I;
        const float *src = w + (size_t)o * I;
        float amax = 0.f;
        for (int i = i0; i < i1; ++i) {
            const float a = fabsf(src[i]);
            if (a > amax) amax = a;
        }
        const float sc = __fdiv_rn(amax, 7.0f);
        scales[(size_t)o * ng + g] = sc;
        uint8_t *dst = wq + (size_t)o * rb;
        for (int i = i0; i < i1; i += 2) {
            uint32_t nib[2] = {8u, 8u};
            for (int k = 0; k < 2 && i + k < i1; ++k) {
                int q = 0;
                if (sc != 0.f) {
                    float r = rintf(__fdiv_rn(src[i + k], sc));
                    r = r < -8.f ? -8.f : (r > 7.f ? 7.f : r);
                    q = (int)r;
                }
                nib[k] = (uint32_t)(q + 8);
            }
            dst[i >> 1] = (uint8_t)(nib[0] | (nib[1] << 4));
        }
    }
}

int run_quantize_i4g(uint8_t *wq, float *scales, const float *w, int O, int I, int gs, cudaStream_t st) {
    const size_t total = (size_t)O * ((I + gs - 1) / gs);
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    quantize_i4g_kernel<<<(unsigned)blocks, 256, 0, st>>>(wq, scales, w, O, I, gs);
    count_launch();
    return check_launch("qg_quantize_i4g");
}

// ---------------------------------------------------------------------------
// MQ4-V2 encoder: one thread per 128-weight half (hipfire "MQ4 V2", section 3)
// ---------------------------------------------------------------------------
__global__ void encode_mq4v2_kernel(uint8_t *__restrict__ blocks, const float *__restrict__ w, int O, int I) {
    const size_t nb = (size_t)I / 256;
    const size_t total = (size_t)O * nb * 2;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const int h = (int)(t & 1);
        const size_t ob = t >> 1;                   // o * nb + b
        const size_t o = ob / nb, b = ob - o * nb;
        const float *hw = w + o * (size_t)I + b * 256 + 128 * h;
        uint8_t *blk = blocks + ob * 136;
        float lo = hw[0], hi = hw[0];
        for (int j = 1; j < 128; ++j) {
            const float v = hw[j];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        const float step = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        const __half sc16 = hi == lo ? __ushort_as_half((unsigned short)0) : __float2half_rn(step);
        const __half z16 = __float2half_rn(lo);
        const float stf = __half2float(sc16);
        const float zf = __half2float(z16);
        const uint32_t hd = (uint32_t)__half_as_ushort(sc16) | ((uint32_t)__half_as_ushort(z16) << 16);
        // Header and payload go out as aligned 32-bit words (the block base is
        // 8-byte aligned).  An 8-bit store of the low byte of an fp16
        // conversion result stores 0 on this toolchain (the .b16 result
        // register straight into st.global.b8; reproduced by
        // tests/f16_byte_store_repro.cu), so the header bytes are never stored
        // one by one.
        reinterpret_cast<uint32_t *>(blk)[h] = hd;
        uint32_t *pay = reinterpret_cast<uint32_t *>(blk + 8 + 64 * h);
        for (int k = 0; k < 16; ++k) {            // word k holds weights 8k..8k+7 of the half
            uint32_t word = 0u;
            for (int m = 0; m < 8; ++m) {
                int q = 0;
                if (stf != 0.f) {
                    float r = rintf(__fdiv_rn(__fsub_rn(hw[8 * k + m], zf), stf));
                    r = r < 0.f ? 0.f : (r > 15.f ? 15.f : r);
                    q = (int)r;
                }
                word |= (uint32_t)q << (4 * m);
            }
            pay[k] = word;
        }
    }
}

int run_encode_mq4v2(uint8_t *blocks, const float *w, int O, int I, cudaStream_t st) {
    const size_t total = (size_t)O * (I / 256) * 2;
    size_t nblk = (total + 255) / 256;
    if (nblk > 65535) nblk = 65535;
    encode_mq4v2_kernel<<<(unsigned)nblk, 256, 0, st>>>(blocks, w, O, I);
    count_launch();
    return check_launch("qg_encode_mq4v2");
}

// ---------------------------------------------------------------------------
// MQ4 v1 (f32 header) and MQ4C pad (fp16 header, four zero bytes) encoders:
// one thread per 256-weight block, the MQ4 rule over the whole block
// (hipfire "MQ4 V2", sections 1b and 1c).
// ---------------------------------------------------------------------------
template <bool kFp16>
__global__ void encode_mq4_one_header_kernel(uint8_t *__restrict__ blocks, const float *__restrict__ w, int O,
                                             int I) {
    const size_t nb = (size_t)I / 256;
    const size_t total = (size_t)O * nb;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const size_t o = t / nb, b = t - o * nb;
        const float *v = w + o * (size_t)I + b * 256;
        uint32_t *blk = reinterpret_cast<uint32_t *>(blocks + t * 136);
        float lo = v[0], hi = v[0];
        for (int j = 1; j < 256; ++j) {
            const float x = v[j];
            if (x < lo) lo = x;
            if (x > hi) hi = x;
        }
        const float step = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        float scale, zero;
        if (kFp16) {
            const __half s16 = hi == lo ? __ushort_as_half((unsigned short)0) : __float2half_rn(step);
            const __half z16 = __float2half_rn(lo);
            scale = __half2float(s16);
            zero = __half2float(z16);
            blk[0] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
            blk[1] = 0u;
        } else {
            scale = hi == lo ? 0.f : step;
            zero = lo;
            blk[0] = __float_as_uint(scale);
            blk[1] = __float_as_uint(zero);
        }
        for (int k = 0; k < 32; ++k) {               // word k holds weights 8k..8k+7
            uint32_t word = 0u;
            for (int m = 0; m < 8; ++m) {
                int q = 0;
                if (scale != 0.f) {
                    float r = rintf(__fdiv_rn(__fsub_rn(v[8 * k + m], zero), scale));
                    r = r < 0.f ? 0.f : (r > 15.f ? 15.f : r);
                    q = (int)r;
                }
                word |= (uint32_t)q << (4 * m);
            }
            blk[2 + k] = word;
        }
    }
}

int run_encode_mq4_one_header(uint8_t *blocks, const float *w, int O, int I, bool fp16_header, cudaStream_t st) {
    const size_t total = (size_t)O * (I / 256);
    size_t nblk = (total + 127) / 128;
    if (nblk > 65535) nblk = 65535;
    if (fp16_header) {
        encode_mq4_one_header_kernel<true><<<(unsigned)nblk, 128, 0, st>>>(blocks, w, O, I);
        count_launch();
        return check_launch("qg_encode_mq4c");
    }
    encode_mq4_one_header_kernel<false><<<(unsigned)nblk, 128, 0, st>>>(blocks, w, O, I);
    count_launch();
    return check_launch("qg_encode_mq4v1");
}

// ---------------------------------------------------------------------------
// signed FWHT-256: one warp per block; lane l holds elements 8l..8l+7.
// Butterfly distances 1, 2, 4 inside a lane, 8..128 across lanes (xor 1..16).
// ---------------------------------------------------------------------------
__global__ void fwht256_kernel(float *out, const float *in, const int8_t *__restrict__ signs, size_t nblocks) {
    const int lane = threadIdx.x & 31;
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t b = blockIdx.x * (size_t)(blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += warps) {
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = (float)signs[8 * lane + t] * in[b * 256 + 8 * lane + t];
#pragma unroll
        for (int len = 1; len < 8; len <<= 1) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if ((t & len) == 0) {
                    const float a = v[t], c = v[t + len];
                    v[t] = a + c;
                    v[t + len] = a - c;
                }
            }
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float other = __shfl_xor_sync(0xffffffffu, v[t], m);
                v[t] = upper ? (other - v[t]) : (v[t] + other);
            }
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 8; ++t) out[b * 256 + 8 * lane + t] = v[t] * 0.0625f;
    }
}

int run_fwht256(float *out, const float *in, const int8_t *signs, size_t nblocks, cudaStream_t st) {
    size_t blocks = (nblocks + 7) / 8;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    fwht256_kernel<<<(unsigned)blocks, 256, 0, st>>>(out, in, signs, nblocks);
    count_launch();
    return check_launch("qg_fwht256");
}

}  // namespace qg
