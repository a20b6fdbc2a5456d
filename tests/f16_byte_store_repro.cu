// Minimal reproduction: the low byte of an fp16 conversion result, stored with
// an 8-bit store.  Each form converts x[i] with cvt.rn.f16.f32 and stores the
// low byte of the fp16 bits at out[i]; the reference stores all 16 bits with a
// 16-bit store and the host takes the low byte.  Prints, per form, how many
// bytes differ from the reference and how many of those are 0.
//   form 0  the .b16 result register straight into st.global.b8
//   form 1  widened with cvt.u32.u16 first
//   form 2  moved to a .u16 integer register and masked first
//   form 3  C++: (uint8_t)(__half_as_ushort(__float2half_rn(v)) & 0xFF)
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o repro f16_byte_store_repro.cu
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

__global__ void store_low_byte(uint8_t *out, const float *x, int n, int form) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint8_t *p = out + i;
    const float v = x[i];
    if (form == 0)
        asm volatile("{.reg .b16 h; cvt.rn.f16.f32 h, %1; st.global.b8 [%0], h;}" ::"l"(p), "f"(v) : "memory");
    else if (form == 1)
        asm volatile("{.reg .b16 h; .reg .b32 r; cvt.rn.f16.f32 h, %1; cvt.u32.u16 r, h; st.global.b8 [%0], r;}" ::"l"(p),
                     "f"(v)
                     : "memory");
    else if (form == 2)
        asm volatile("{.reg .b16 h; .reg .u16 u; cvt.rn.f16.f32 h, %1; mov.b16 u, h; and.b16 u, u, 255; st.global.u8 [%0], u;}" ::"l"(
                         p),
                     "f"(v)
                     : "memory");
    else if (form == 3)
        *p = (uint8_t)(__half_as_ushort(__float2half_rn(v)) & 0xFF);
    else
        asm volatile("{.reg .b16 h; cvt.rn.f16.f32 h, %1; st.global.b16 [%0], h;}" ::"l"(out + 2 * i), "f"(v) : "memory");
}

int main() {
    const int n = 4096;
    static float hx[n];
    for (int i = 0; i < n; ++i) hx[i] = -0.05f + 0.1f * (float)i / n + 1e-4f * (float)(i % 7);
    float *x = nullptr;
    uint8_t *o = nullptr;
    if (cudaMalloc(&x, n * sizeof(float)) != cudaSuccess || cudaMalloc(&o, 2 * n) != cudaSuccess) return 2;
    cudaMemcpy(x, hx, n * sizeof(float), cudaMemcpyHostToDevice);
    static uint8_t ref[2 * n], got[2 * n];
    cudaMemset(o, 0xAA, 2 * n);
    store_low_byte<<<(n + 255) / 256, 256>>>(o, x, n, 4);
    cudaMemcpy(ref, o, 2 * n, cudaMemcpyDeviceToHost);
    int nonzero = 0;
    for (int i = 0; i < n; ++i) nonzero += ref[2 * i] != 0;
    printf("bytes %d, reference low bytes nonzero %d\n", n, nonzero);
    for (int f = 0; f < 4; ++f) {
        cudaMemset(o, 0xAA, 2 * n);
        store_low_byte<<<(n + 255) / 256, 256>>>(o, x, n, f);
        const cudaError_t e = cudaDeviceSynchronize();
        cudaMemcpy(got, o, n, cudaMemcpyDeviceToHost);
        int bad = 0, zero = 0;
        for (int i = 0; i < n; ++i)
            if (got[i] != ref[2 * i]) {
                ++bad;
                zero += got[i] == 0;
            }
        printf("form %d: %s wrong %d zero %d\n", f, cudaGetErrorString(e), bad, zero);
    }
    return 0;
}
