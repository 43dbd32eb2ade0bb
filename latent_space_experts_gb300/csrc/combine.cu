// Gate-weighted combine of the k expert outputs and the RMSNorm that follows it.
//
// 苏神复盘 Kimi K3 §02 and K3 architecture write-up 归一化策略调整: the only norm of the
// Stable LatentMoE block sits after the combine and before the up-projection.
//   c_t = sum_j topk_w[t,j] * y_e[slot_pos[t,j]]       (fp32, slots in order j = 0..k-1)
//   z_t = gamma * c_t / sqrt(mean(c_t^2) + eps)
// Resident blocks (as many as fit on the SMs) take the tokens in turn, one token at a time;
// 16-byte vector loads of the k expert rows, eight rows in flight per thread; c_t is staged
// in shared memory between the two passes.  HBM-bound: it reads k rows of d_latent per token.
#include "common.cuh"
#include "internal.h"

namespace slmoe {
namespace {

constexpr int CB_THREADS = 256;
constexpr int CB_GROUP = 8;        // expert rows loaded before they are added

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; using U = float4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; using U = uint4; };

template <typename T>
__device__ __forceinline__ void unpack(const typename Vec<T>::U &u, float *f);
template <>
__device__ __forceinline__ void unpack<float>(const float4 &u, float *f) {
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <typename T>
__device__ __forceinline__ typename Vec<T>::U pack(const float *f);
template <>
__device__ __forceinline__ float4 pack<float>(const float *f) { return make_float4(f[0], f[1], f[2], f[3]); }
template <>
__device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(CB_THREADS)
combine_rmsnorm_kernel(const T *__restrict__ y_e, const float *__restrict__ topk_w,
                       const int32_t *__restrict__ slot_pos, const float *__restrict__ gamma,
                       int n_tok, int d_l, int k, float eps, T *__restrict__ z) {
    using U = typename Vec<T>::U;
    constexpr int V = Vec<T>::N;
    extern __shared__ float c_s[];
    __shared__ int64_t rows[32];
    __shared__ float wts[32];
    __shared__ float red[CB_THREADS / 32];
    const int tid = threadIdx.x;
    for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
        if (tid < k) {
            rows[tid] = (int64_t)slot_pos[(int64_t)t * k + tid] * d_l;
            wts[tid] = topk_w[(int64_t)t * k + tid];
        }
        __syncthreads();
        const int nv = d_l / V;
        float ss = 0.f;
        for (int q = tid; q < nv; q += CB_THREADS) {
            float acc[V];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = 0.f;
            // the slots' rows are loaded CB_GROUP at a time before any is added, so that a thread
            // keeps that many loads in flight; the adds stay in slot order j = 0..k-1
            for (int j0 = 0; j0 < k; j0 += CB_GROUP) {
                U u[CB_GROUP];
#pragma unroll
                for (int g = 0; g < CB_GROUP; ++g)
                    if (j0 + g < k) u[g] = *reinterpret_cast<const U *>(y_e + rows[j0 + g] + (int64_t)q * V);
#pragma unroll
                for (int g = 0; g < CB_GROUP; ++g) {
                    if (j0 + g < k) {
                        float f[V];
                        unpack<T>(u[g], f);
                        const float wj = wts[j0 + g];
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < V; ++i) {
                c_s[q * V + i] = acc[i];
                ss = fmaf(acc[i], acc[i], ss);
            }
        }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < CB_THREADS / 32; ++i) tot += red[i];
        const float scale = 1.0f / sqrtf(tot / (float)d_l + eps);
        for (int q = tid; q < nv; q += CB_THREADS) {
            float f[V];
#pragma unroll
            for (int i = 0; i < V; ++i) f[i] = gamma[q * V + i] * (c_s[q * V + i] * scale);
            *reinterpret_cast<U *>(z + (int64_t)t * d_l + (int64_t)q * V) = pack<T>(f);
        }
        __syncthreads();    // c_s, red and the row offsets are read before the next token writes them
    }
}

// Blocks of the combine that fit on the SMs at once (a host-side occupancy query), at most T.
template <typename K>
int combine_grid(K kern, size_t smem, int T) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, CB_THREADS, smem) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const long long n = (long long)per_sm * sm_count();
    return (int)(n < T ? n : T);
}

}  // namespace

int launch_combine_rmsnorm(int dtype, const void *y_e, const float *topk_w,
                           const int32_t *slot_pos, const float *gamma, int T, int d_latent,
                           int k, float eps, void *z, cudaStream_t st) {
    if (T <= 0) return SLMOE_OK;
    const size_t smem = (size_t)d_latent * sizeof(float);
    if (dtype == DT_BF16) {
        auto kern = combine_rmsnorm_kernel<__nv_bfloat16>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<combine_grid(kern, smem, T), CB_THREADS, smem, st>>>(static_cast<const __nv_bfloat16 *>(y_e), topk_w,
                                                                  slot_pos, gamma, T, d_latent, k, eps,
                                                                  static_cast<__nv_bfloat16 *>(z));
    } else {
        auto kern = combine_rmsnorm_kernel<float>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<combine_grid(kern, smem, T), CB_THREADS, smem, st>>>(static_cast<const float *>(y_e), topk_w, slot_pos,
                                                                  gamma, T, d_latent, k, eps, static_cast<float *>(z));
    }
    return check_launch("combine_rmsnorm");
}

}  // namespace slmoe
