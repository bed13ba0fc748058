// srwm_probe.cu -- FP32 FMA throughput probe used to calibrate the roofline of
// the SRWM kernels (their bound is the FP32 FMA pipe, not memory).
#include <cuda_runtime.h>

#include "srwm.h"

namespace {

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// 8 independent dependency chains per thread; each iteration is 8 FMAs
// (scalar) or 8 two-wide FMAs (packed).
template <bool PACKED>
__global__ void fma_probe_kernel(float* out, int iters)
{
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    const float mul = 0.9999999f, add = 1.0e-7f;
    float r = 0.f;
    if constexpr (PACKED) {
        float2 a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = make_float2(tid * 1e-9f + k, tid * 1e-9f - k);
        const float2 m2 = make_float2(mul, mul), c2 = make_float2(add, add);
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = ffma2(a[k], m2, c2);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) r += a[k].x + a[k].y;
    } else {
        float a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = tid * 1e-9f + k;
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = fmaf(a[k], mul, add);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) r += a[k];
    }
    out[tid] = r;
}

}  // namespace

extern "C" int srwm_probe_fma(int blocks, int threads, int iters, int packed, float* out, void* stream)
{
    if (!out) return SRWM_ERR_NULL;
    if (blocks <= 0 || threads <= 0 || threads > 1024 || iters < 0) return SRWM_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (packed) fma_probe_kernel<true><<<blocks, threads, 0, s>>>(out, iters);
    else fma_probe_kernel<false><<<blocks, threads, 0, s>>>(out, iters);
    if (cudaGetLastError() != cudaSuccess) return SRWM_ERR_CUDA;
    return SRWM_OK;
}
