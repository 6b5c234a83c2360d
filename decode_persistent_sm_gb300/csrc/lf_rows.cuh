// Row kernels shared by the batched prefill and the batched decode: one CTA
// per row of a [rows][D] fp32 residual (each translation unit that includes
// this header gets its own copy).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// Delayed residual adds fused with the RMSNorm that reads their result, one
// block per row i: x[i] += P_u[i] for u = u0 .. u0 + n_u - 1 in that order
// (P_u is slot u % R of `ring`, slot_elems floats per slot, rows of D), then
// h[i] = FP16(g * x[i] / sqrt(mean(x[i]^2) + eps)).  The row stays in
// registers (D / 4 float4 over the block, at most kNormV per thread).
constexpr int kNormThreads = 256, kNormV = 8;

__global__ void __launch_bounds__(kNormThreads) pf_addnorm(float *__restrict__ x, const float *__restrict__ ring,
                                                           size_t slot_elems, int u0, int n_u, int R,
                                                           const __half *__restrict__ g, __half *__restrict__ h,
                                                           int D, float eps) {
    __shared__ float red[32];
    const int n4 = D >> 2;
    float4 *xr = reinterpret_cast<float4 *>(x + (size_t)blockIdx.x * D);
    float4 v[kNormV];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kNormV; ++k) {
        const int c = threadIdx.x + k * kNormThreads;
        if (c < n4) {
            v[k] = xr[c];
            for (int u = u0; u < u0 + n_u; ++u) {
                const float4 a =
                    reinterpret_cast<const float4 *>(ring + (size_t)(u % R) * slot_elems + (size_t)blockIdx.x * D)[c];
                v[k].x += a.x;
                v[k].y += a.y;
                v[k].z += a.z;
                v[k].w += a.w;
            }
            if (n_u > 0) xr[c] = v[k];
            ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        }
    }
    const float inv = rsqrtf(block_sum(ss, red) / D + eps);
    const uint2 *gr = reinterpret_cast<const uint2 *>(g);
    uint2 *hr = reinterpret_cast<uint2 *>(h + (size_t)blockIdx.x * D);
#pragma unroll
    for (int k = 0; k < kNormV; ++k) {
        const int c = threadIdx.x + k * kNormThreads;
        if (c < n4) {
            const uint2 gw = gr[c];
            const float2 g01 = __half22float2(*reinterpret_cast<const __half2 *>(&gw.x));
            const float2 g23 = __half22float2(*reinterpret_cast<const __half2 *>(&gw.y));
            const __half2 o01 = __floats2half2_rn(g01.x * v[k].x * inv, g01.y * v[k].y * inv);
            const __half2 o23 = __floats2half2_rn(g23.x * v[k].z * inv, g23.y * v[k].w * inv);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t *>(&o01);
            o.y = *reinterpret_cast<const uint32_t *>(&o23);
            hr[c] = o;
        }
    }
}

}  // namespace
