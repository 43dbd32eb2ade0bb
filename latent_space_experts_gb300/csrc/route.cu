// Biased top-k selection and the expert-sorted permutation.
//
// Selection (苏神复盘 Kimi K3 §02; K3 architecture write-up, 负载均衡优化): the k experts with
// the largest s + b, ties to the lower expert index, slots in that order; the gate weights
// are the chosen raw scores renormalised to sum 1.
// Permutation (single-GPU stand-in for the dispatch of §01): counts per expert, their
// exclusive scan, and a stable scatter that lists tokens by expert, then token id.  All
// three kernels are deterministic: positions come from counts and scans, never from the
// order in which atomics land.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace slmoe {
namespace {

constexpr int TOPK_WARPS = 8;
constexpr int MAX_E = 4096;          // E per lane <= 128 -> 4 words of "taken" bits

__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}

// One block per chunk of ROUTE_CHUNK tokens, one warp per token at a time.
__global__ void __launch_bounds__(TOPK_WARPS * 32)
topk_kernel(const float *__restrict__ scores, const float *__restrict__ bias, int T, int E,
            int k, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
            int32_t *__restrict__ chunk_counts, int32_t *status) {
    extern __shared__ float sm[];
    float *bias_s = sm;
    int *cnt = reinterpret_cast<int *>(sm + E);
    float *rows = sm + 2 * E;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < E; i += blockDim.x) {
        bias_s[i] = bias[i];
        cnt[i] = 0;
    }
    __syncthreads();

    float *row = rows + (size_t)warp * E;
    const int t_begin = blockIdx.x * ROUTE_CHUNK;
    int nan_count = 0;
    for (int tt = warp; tt < ROUTE_CHUNK; tt += TOPK_WARPS) {
        const int t = t_begin + tt;
        if (t >= T) break;
        const float *srow = scores + (int64_t)t * E;
        float best_v = -INFINITY;
        int best_i = INT_MAX;
        for (int e = lane; e < E; e += 32) {
            float s = srow[e];
            row[e] = s;
            float v;
            if (isnan(s)) {
                ++nan_count;
                v = -INFINITY;
            } else {
                v = s + bias_s[e];
            }
            if (beats(v, e, best_v, best_i)) { best_v = v; best_i = e; }
        }
        __syncwarp();
        uint32_t taken[MAX_E / 32 / 32] = {0, 0, 0, 0};
        int my_e = 0;
        for (int j = 0; j < k; ++j) {
            float v = best_v;
            int i = best_i;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, v, o);
                int oi = __shfl_xor_sync(0xffffffffu, i, o);
                if (beats(ov, oi, v, i)) { v = ov; i = oi; }
            }
            if (lane == j) my_e = i;
            if ((i & 31) == lane) {          // the owner drops the winner and rescans
                const int q = i >> 5;
                taken[q >> 5] |= 1u << (q & 31);
                best_v = -INFINITY;
                best_i = INT_MAX;
                int qq = 0;
                for (int e = lane; e < E; e += 32, ++qq) {
                    if (taken[qq >> 5] & (1u << (qq & 31))) continue;
                    float s = row[e];
                    float bv = isnan(s) ? -INFINITY : s + bias_s[e];
                    if (beats(bv, e, best_v, best_i)) { best_v = bv; best_i = e; }
                }
            }
        }
        float s_raw = 0.f;
        if (lane < k) {
            s_raw = row[my_e];
            if (isnan(s_raw)) s_raw = 0.f;
        }
        const float sum = warp_sum(s_raw);
        if (lane < k) {
            topk_idx[(int64_t)t * k + lane] = my_e;
            topk_w[(int64_t)t * k + lane] = sum > 0.f ? s_raw / sum : 1.0f / (float)k;
            atomicAdd(&cnt[my_e], 1);
        }
        __syncwarp();
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nan_count += __shfl_xor_sync(0xffffffffu, nan_count, o);
    if (lane == 0 && nan_count && status) atomicAdd(&status[ST_NAN], nan_count);
    __syncthreads();
    int32_t *cc = chunk_counts + (int64_t)blockIdx.x * E;
    for (int i = tid; i < E; i += blockDim.x) cc[i] = cnt[i];
}

// One block: per expert, turn chunk counts into exclusive chunk bases; then the exclusive
// scan of the expert totals.
__global__ void __launch_bounds__(1024)
scan_kernel(int32_t *__restrict__ cc, int nchunks, int E, int32_t *__restrict__ counts,
            int32_t *__restrict__ offsets) {
    __shared__ int32_t tot[MAX_E];
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        int c = 0;
        for (; c + 8 <= nchunks; c += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = cc[(int64_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                cc[(int64_t)(c + u) * E + e] = run;
                run += v[u];
            }
        }
        for (; c < nchunks; ++c) {
            int v = cc[(int64_t)c * E + e];
            cc[(int64_t)c * E + e] = run;
            run += v;
        }
        counts[e] = run;
        tot[e] = run;
    }
    __syncthreads();
    const int base = tid * 4;
    int loc[4], s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        loc[i] = (base + i < E) ? tot[base + i] : 0;
        s += loc[i];
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = warp_tot[lane], inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        warp_tot[lane] = inc - v;
    }
    __syncthreads();
    int run = warp_tot[w] + incl - s;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (base + i < E) offsets[base + i] = run;
        run += loc[i];
    }
    if (tid == blockDim.x - 1) offsets[E] = run;
}

// One block per chunk: walk the chunk's tokens in order; lane j places slot j.  The k
// experts of one token are distinct, so the lanes of one step never share a counter.
__global__ void __launch_bounds__(128)
scatter_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ chunk_base,
               const int32_t *__restrict__ offsets, int T, int E, int k,
               int32_t *__restrict__ perm, int32_t *__restrict__ slot_pos) {
    extern __shared__ int32_t next[];
    const int32_t *cb = chunk_base + (int64_t)blockIdx.x * E;
    for (int i = threadIdx.x; i < E; i += blockDim.x) next[i] = offsets[i] + cb[i];
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int t0 = blockIdx.x * ROUTE_CHUNK;
    const int t1 = min(T, t0 + ROUTE_CHUNK);
    for (int t = t0; t < t1; ++t) {
        if (lane < k) {
            const int e = topk_idx[(int64_t)t * k + lane];
            const int pos = next[e];
            next[e] = pos + 1;
            perm[pos] = t;
            slot_pos[(int64_t)t * k + lane] = pos;
        }
        __syncwarp();
    }
}

}  // namespace

int launch_topk(const float *scores, const float *bias, int T, int E, int k, int32_t *topk_idx,
                float *topk_w, int32_t *chunk_counts, int32_t *status, cudaStream_t st) {
    const int nchunks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    if (nchunks == 0) return SLMOE_OK;
    const size_t smem = (size_t)(2 + TOPK_WARPS) * E * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return fail(SLMOE_ECUDA, "topk smem attribute: %s", cudaGetErrorString(e));
    }
    topk_kernel<<<nchunks, TOPK_WARPS * 32, smem, st>>>(scores, bias, T, E, k, topk_idx, topk_w,
                                                        chunk_counts, status);
    return check_launch("topk");
}

int launch_scan(int32_t *chunk_counts, int nchunks, int E, int32_t *counts, int32_t *offsets,
                cudaStream_t st) {
    scan_kernel<<<1, 1024, 0, st>>>(chunk_counts, nchunks, E, counts, offsets);
    return check_launch("scan");
}

int launch_scatter(const int32_t *topk_idx, const int32_t *chunk_base, const int32_t *offsets,
                   int T, int E, int k, int32_t *perm, int32_t *slot_pos, cudaStream_t st) {
    const int nchunks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    if (nchunks == 0) return SLMOE_OK;
    scatter_kernel<<<nchunks, 128, E * sizeof(int32_t), st>>>(topk_idx, chunk_base, offsets, T, E,
                                                              k, perm, slot_pos);
    return check_launch("scatter");
}

}  // namespace slmoe
