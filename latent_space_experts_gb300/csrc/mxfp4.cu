// MXFP4 weights and MXFP8 activations: the OCP Microscaling block format (blocks of 32 values
// along K sharing one E8M0 power-of-two scale; FP4 E2M1 weight codes, FP8 E4M3 activation
// codes), for the routed experts ("Stable Latent MoE" concept note, 训练基础设施: MXFP4 weights,
// MXFP8 activations).  The layer's tensor cores read both directly (block-scaled MMA,
// tc_gemm.cu); this file converts bf16 weights to MXFP4, and fp32 values to MXFP8 with the
// same block conversion the layer's epilogues use (mx.cuh).
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "mx.cuh"

namespace slmoe {
namespace {

// One thread per block of 32 values: e = floor(log2 max|v|) - 2 clamped to [-127, 127] (from
// the fp32 exponent field; an all-zero or subnormal maximum gives -127), then each v * 2^-e
// (exact: a power-of-two scaling) goes to the nearest E2M1 magnitude with ties to the even
// mantissa, by counting the midpoints it passes (a tie stays below when the lower magnitude
// has an even code, goes above otherwise), saturating at 6.
__global__ void __launch_bounds__(256) mxfp4_quantize_kernel(const __nv_bfloat16 *__restrict__ W, long long nblocks,
                                                             uint8_t *__restrict__ packed,
                                                             uint8_t *__restrict__ scales) {
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
         b += (long long)gridDim.x * blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(W + b * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = src[q];
            const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[8 * q + j] = __bfloat162float(h[j]);
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
        const int be = (__float_as_int(amax) >> 23) & 0xFF;
        int e = (be == 0 ? -127 : be - 127) - 2;
        e = max(-127, min(127, e));
        uint32_t words[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float s = ldexpf(v[j], -e);
            const float m = fabsf(s);
            const uint32_t idx = (m > 0.25f) + (m >= 0.75f) + (m > 1.25f) + (m >= 1.75f) + (m > 2.5f) +
                                 (m >= 3.5f) + (m > 5.0f);
            const uint32_t code = idx | (s < 0.f ? 8u : 0u);
            words[j >> 3] |= code << (4 * (j & 7));
        }
        reinterpret_cast<uint4 *>(packed)[b] = make_uint4(words[0], words[1], words[2], words[3]);
        scales[b] = (uint8_t)(e + 127);
    }
}

// One thread per block of 32 fp32 values (rows of K values, K a multiple of 32): 32 code bytes
// and one scale byte through mx8_quant32.
__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const float *__restrict__ X, long long nblocks,
                                                             uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ scales) {
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
         b += (long long)gridDim.x * blockDim.x) {
        const float4 *src = reinterpret_cast<const float4 *>(X + b * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 u = src[q];
            v[4 * q] = u.x; v[4 * q + 1] = u.y; v[4 * q + 2] = u.z; v[4 * q + 3] = u.w;
        }
        uint32_t w[8];
        scales[b] = (uint8_t)mx8_quant32(v, w);
        uint4 *dst = reinterpret_cast<uint4 *>(codes + b * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

}  // namespace

int launch_mxfp8_quantize(const float *X, long long rows, int K, uint8_t *codes, uint8_t *scales, cudaStream_t st) {
    const long long nblocks = rows * (K / 32);
    if (nblocks == 0) return SLMOE_OK;
    const long long want = (nblocks + 255) / 256;
    const int grid = (int)(want < 16LL * sm_count() ? want : 16LL * sm_count());
    mxfp8_quantize_kernel<<<grid, 256, 0, st>>>(X, nblocks, codes, scales);
    return check_launch("mxfp8_quantize");
}

int launch_mxfp4_quantize(const void *W, long long rows, int K, uint8_t *packed, uint8_t *scales, cudaStream_t st) {
    const long long nblocks = rows * (K / 32);
    if (nblocks == 0) return SLMOE_OK;
    const long long want = (nblocks + 255) / 256;
    const int grid = (int)(want < 16LL * sm_count() ? want : 16LL * sm_count());
    mxfp4_quantize_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(W), nblocks, packed, scales);
    return check_launch("mxfp4_quantize");
}

}  // namespace slmoe
