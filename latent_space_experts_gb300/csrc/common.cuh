// Shared device helpers of the slmoe library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace slmoe {

// ---------------------------------------------------------------- element conversions
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- activations
// SiTU gate (beta1 * tanh(g / beta1) * sigmoid(g)) and the soft cap of the up branch
// (beta2 * tanh(u / beta2)); K3 architecture write-up, SiTU激活优化.  Accurate variants use
// the CUDA math library; the fast variants use the PTX tanh.approx.f32 instruction
// (sigmoid(g) = 0.5 + 0.5 tanh(g / 2)).
__device__ __forceinline__ float situ_glu_accurate(float g, float u, float b1, float b2) {
    float sig = 1.0f / (1.0f + expf(-g));
    return (b1 * tanhf(g / b1) * sig) * (b2 * tanhf(u / b2));
}

__device__ __forceinline__ float tanh_fast(float v) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float situ_glu_fast(float g, float u, float inv_b1, float b1,
                                               float inv_b2, float b2) {
    float sig = fmaf(0.5f, tanh_fast(0.5f * g), 0.5f);
    return (b1 * tanh_fast(g * inv_b1) * sig) * (b2 * tanh_fast(u * inv_b2));
}

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// status word indices (see slmoe.h)
enum { ST_NAN = 0, ST_OVERFLOW = 1, ST_TIMEOUT = 2 };

}  // namespace slmoe
