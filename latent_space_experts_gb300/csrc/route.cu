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

constexpr int TOPK_MAX_WARPS = 16;    // one token per warp when shared memory allows
constexpr int LIST = 4;              // candidates each lane keeps in registers

__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}

// Insert (v, i) into a lane's descending candidate list of LIST entries.
__device__ __forceinline__ void list_insert(float (&lv)[LIST], int (&li)[LIST], float v, int i) {
    if (!beats(v, i, lv[LIST - 1], li[LIST - 1])) return;
    lv[LIST - 1] = v;
    li[LIST - 1] = i;
#pragma unroll
    for (int p = LIST - 1; p > 0; --p) {
        if (beats(lv[p], li[p], lv[p - 1], li[p - 1])) {
            float tv = lv[p]; lv[p] = lv[p - 1]; lv[p - 1] = tv;
            int ti = li[p]; li[p] = li[p - 1]; li[p - 1] = ti;
        }
    }
}

// One block per chunk of ROUTE_CHUNK tokens, one warp per token (fewer warps, looping, when
// E is too large for a staging row per warp).  Lane l owns the
// experts e = l, l + 32, ...; it keeps its best LIST (biased score, index) pairs in
// registers.  Each of the k rounds takes the warp-wide best head (ties to the lower index)
// and the owning lane pops it; a lane whose list runs dry rescans its experts for the best
// ones that its last popped pair beats (everything above that was taken already).
__global__ void __launch_bounds__(TOPK_MAX_WARPS * 32)
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
    const int n_local = lane < E ? (E - lane + 31) / 32 : 0;
    int nan_count = 0;
    const int nwarps = blockDim.x >> 5;
    for (int tt = warp; tt < ROUTE_CHUNK; tt += nwarps) {
        const int t = t_begin + tt;
        if (t >= T) break;
        const float *srow = scores + (int64_t)t * E;
        float lv[LIST];
        int li[LIST];
#pragma unroll
        for (int p = 0; p < LIST; ++p) { lv[p] = -INFINITY; li[p] = INT_MAX; }
        // stage the row in shared memory with independent loads first (latency once per
        // batch, not once per element), then build the candidate lists from it
        for (int e0 = lane; e0 < E; e0 += 32 * 16) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = (e0 + 32 * u < E) ? __ldcs(srow + e0 + 32 * u) : 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (e0 + 32 * u < E) row[e0 + 32 * u] = v[u];
        }
        for (int e = lane; e < E; e += 32) {
            const float s = row[e];
            float v;
            if (isnan(s)) { ++nan_count; v = -INFINITY; } else { v = s + bias_s[e]; }
            list_insert(lv, li, v, e);
        }
        __syncwarp();
        int popped = 0;
        int my_e = 0;
        for (int j = 0; j < k; ++j) {
            float v = lv[0];
            int i = li[0];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                const int oi = __shfl_xor_sync(0xffffffffu, i, o);
                if (beats(ov, oi, v, i)) { v = ov; i = oi; }
            }
            if (lane == j) my_e = i;
            if (li[0] == i) {                    // this lane owned the winner: pop it
                const float last_v = lv[0];
                const int last_i = li[0];
#pragma unroll
                for (int p = 0; p < LIST - 1; ++p) { lv[p] = lv[p + 1]; li[p] = li[p + 1]; }
                lv[LIST - 1] = -INFINITY;
                li[LIST - 1] = INT_MAX;
                ++popped;
                if (li[0] == INT_MAX && popped < n_local) {
                    for (int e = lane; e < E; e += 32) {
                        const float s = row[e];
                        const float bv = isnan(s) ? -INFINITY : s + bias_s[e];
                        if (beats(last_v, last_i, bv, e)) list_insert(lv, li, bv, e);
                    }
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

// Per-expert exclusive scan of the chunk counts (chunk_counts becomes the chunk bases) and
// the expert totals.  One block per 32 experts (lane = expert); warp w covers a contiguous
// range of chunks; the warps' partial sums are scanned in shared memory.
constexpr int SCAN_WARPS = 32;
constexpr int SCAN_UNROLL = 8;
__global__ void __launch_bounds__(SCAN_WARPS * 32)
scan_kernel(int32_t *__restrict__ cc, int nchunks, int E, int32_t *__restrict__ counts) {
    __shared__ int32_t part[SCAN_WARPS][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const bool ok = e < E;
    const int per = (nchunks + SCAN_WARPS - 1) / SCAN_WARPS;
    const int c0 = w * per, c1 = min(nchunks, c0 + per);
    int sum = 0;
    for (int c = c0; c < c1; c += SCAN_UNROLL) {
        int v[SCAN_UNROLL];
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) v[u] = (ok && c + u < c1) ? cc[(int64_t)(c + u) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) sum += v[u];
    }
    part[w][lane] = sum;
    __syncthreads();
    int base = 0;
    for (int ww = 0; ww < w; ++ww) base += part[ww][lane];
    if (w == SCAN_WARPS - 1 && ok) counts[e] = base + sum;
    int run = base;
    for (int c = c0; c < c1; c += SCAN_UNROLL) {
        int v[SCAN_UNROLL];
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) v[u] = (ok && c + u < c1) ? cc[(int64_t)(c + u) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) {
            if (ok && c + u < c1) cc[(int64_t)(c + u) * E + e] = run;
            run += v[u];
        }
    }
}

// One block per chunk.  The block first scans the expert totals into offsets (block 0 also
// writes them out), then one warp walks the chunk's tokens in order; lane j places slot j.
// The k experts of one token are distinct, so the lanes of one step never share a counter.
__global__ void __launch_bounds__(256)
scatter_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ chunk_base,
               const int32_t *__restrict__ counts, int T, int E, int k,
               int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
               int32_t *__restrict__ slot_pos) {
    extern __shared__ int32_t next[];              // [E]
    __shared__ int32_t wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    // exclusive scan of counts[0..E): thread-contiguous runs, then a warp/block scan
    const int per = (E + 255) / 256;
    const int b0 = tid * per;
    int loc = 0;
    for (int i = 0; i < per; ++i)
        if (b0 + i < E) loc += counts[b0 + i];
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int wbase = 0;
    for (int i = 0; i < w; ++i) wbase += wsum[i];
    int run = wbase + incl - loc;
    const int32_t *cb = chunk_base + (int64_t)blockIdx.x * E;
    for (int i = 0; i < per; ++i) {
        const int e = b0 + i;
        if (e < E) {
            if (blockIdx.x == 0) offsets[e] = run;
            next[e] = run + cb[e];
            run += counts[e];
        }
    }
    if (blockIdx.x == 0 && tid == 255) offsets[E] = run;
    __syncthreads();
    if (tid >= 32) return;
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
    // bias + counters + one staging row per warp must fit in 227 KB of shared memory
    int warps = (int)(232448 / ((size_t)4 * E)) - 2;
    warps = warps > TOPK_MAX_WARPS ? TOPK_MAX_WARPS : (warps < 1 ? 1 : warps);
    const size_t smem = (size_t)(2 + warps) * E * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "topk smem attribute: %s", cudaGetErrorString(e));
    topk_kernel<<<nchunks, warps * 32, smem, st>>>(scores, bias, T, E, k, topk_idx, topk_w, chunk_counts, status);
    return check_launch("topk");
}

int launch_scan(int32_t *chunk_counts, int nchunks, int E, int32_t *counts, cudaStream_t st) {
    scan_kernel<<<(E + 31) / 32, SCAN_WARPS * 32, 0, st>>>(chunk_counts, nchunks, E, counts);
    return check_launch("scan");
}

int launch_scatter(const int32_t *topk_idx, const int32_t *chunk_base, const int32_t *counts, int T,
                   int E, int k, int32_t *offsets, int32_t *perm, int32_t *slot_pos, cudaStream_t st) {
    const int nchunks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    if (nchunks == 0) return SLMOE_OK;
    scatter_kernel<<<nchunks, 256, E * sizeof(int32_t), st>>>(topk_idx, chunk_base, counts, T, E, k,
                                                              offsets, perm, slot_pos);
    return check_launch("scatter");
}

}  // namespace slmoe
