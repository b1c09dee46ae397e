// fp8.cu — per-tensor FP8: the static quantisation kernel.
//
// Source: the sglang PR #28333 page, "关键源码片段" (fp8_kernel.py,
// _static_quant_fp8): with y and the scale y_s read as fp32, the kernel forms
// y_s_inv = 1 / y_s and stores clamp(y * y_s_inv, fp8_min, fp8_max) converted
// to e4m3.  Here: the same steps in binary32 (IEEE division for the
// reciprocal, one rounded product), then the hardware conversion
// cvt.rn.satfinite.e4m3x2.f32 (round to nearest even; the clamp has already
// put the value in range).  Eight bf16 values per thread (16 bytes in, 8 out),
// a scalar tail; PDL hooks as in the GEMM kernels (the scale and x are read
// after the grid-dependency wait).
//
// The FP8 linear itself is the router MMA split-K kernel (dotmma.cu) with e4m3
// operands.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

// Two fp32 values -> two e4m3 codes, lo in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float quant_one(uint16_t xb, float inv) {
    float y = bf16_to_f32(xb) * inv;
    y = fminf(fmaxf(y, -448.0f), 448.0f);
    return y;
}

__global__ void __launch_bounds__(256) quant_fp8_kernel(const uint16_t *__restrict__ x, const float *__restrict__ scale,
                                                        uint8_t *__restrict__ q, long long n, int vec) {
    pdl_launch_dependents();
    pdl_wait();  // x and the scale may be written by the previous kernel
    const float inv = 1.0f / __ldg(scale);
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (vec) {
        const long long nv = n / 8;
        for (long long v = i; v < nv; v += stride) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(x) + v);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            uint16_t c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = e4m3x2(quant_one((uint16_t)(u[j] & 0xFFFFu), inv), quant_one((uint16_t)(u[j] >> 16), inv));
            uint2 o;
            o.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
            o.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
            reinterpret_cast<uint2 *>(q)[v] = o;
        }
        // the tail (n % 8 values), one element per thread
        for (long long k = (n / 8) * 8 + ((long long)blockIdx.x * blockDim.x + threadIdx.x); k < n; k += stride)
            q[k] = (uint8_t)(e4m3x2(quant_one(x[k], inv), 0.0f) & 0xFFu);
    } else {
        for (; i < n; i += stride) q[i] = (uint8_t)(e4m3x2(quant_one(x[i], inv), 0.0f) & 0xFFu);
    }
}

}  // namespace

int launch_quant_fp8(const void *x, const float *scale, void *q, long long n, int num_sms, uint32_t flags,
                     void *stream) {
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(q)) & 15u) == 0;
    const long long work = vec ? (n + 7) / 8 : n;
    long long blocks = (work + 255) / 256;
    const long long cap = 4LL * num_sms;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, quant_fp8_kernel, static_cast<const uint16_t *>(x), scale,
                                   static_cast<uint8_t *>(q), n, vec ? 1 : 0);
}

}  // namespace bf16l
