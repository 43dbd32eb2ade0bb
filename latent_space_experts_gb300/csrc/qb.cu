// Quantile Balancing: per-expert score histograms and the bias update.
//
// K3 architecture write-up, 负载均衡优化: scores in [0, 1] are binned (1000 bins suffice), the
// target quantile is read from the binned distribution, and histograms add across
// micro-batches and machines.  The bias update (b_e <- mean(q) - q_e) is this library's
// fixed reading; the pages defer the exact rule to a technical report.
//
// Histogram design.  scores [T, E] fp32 is streamed once from HBM.  The experts are cut
// into slabs of 32 (one 128-byte line per row: lane = expert), and each slab is counted by
// one thread-block cluster of P CTAs that split the tokens (P from the SMs' cluster
// occupancy).  Each CTA keeps 32-bit counters [bin][32 experts] in shared memory, so the 32
// lanes of an atomic always hit 32 distinct banks, plus one extra row that counts NaN
// scores; every lane keeps 32 row loads in flight, and a score's counter row takes a few
// full-rate FP32 / integer instructions (qb_bin).  At the end the cluster adds its CTAs'
// counters through distributed shared memory and each bin of global memory is read and
// written exactly once, coalesced: no global atomics and no partial histograms in HBM.
#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace slmoe {
namespace {

constexpr int QB_SLAB = 32;
constexpr int QB_MAX_CLUSTER = 8;

// Counter row of a score: min(nbins - 1, max(0, floor(fl32(s * nbins)))), and the extra row
// nbins for NaN.  The floor is taken exactly on the FP32 pipe: the product is clamped to
// [0, nbins - 1] with NaN kept, and adding 2^23 rounded toward minus infinity leaves floor(q)
// in the low mantissa bits (exact for q < 2^23).  Any NaN bit pattern lies above every bin
// and is capped at nbins.
__device__ __forceinline__ uint32_t qb_bin(float v, float nb, float top_f, uint32_t nbins) {
    const float p = __fmul_rn(v, nb);
    float q;
    asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(q) : "f"(p));
    asm("min.NaN.f32 %0, %0, %1;" : "+f"(q) : "f"(top_f));
    const uint32_t bits = __float_as_uint(__fadd_rd(q, 8388608.0f));
    return min(bits - 0x4B000000u, nbins);
}


// Staging tile of the flush: [32 experts][QB_SB + 1] u32 (odd pitch: conflict-free both ways).
constexpr int QB_SB = 224;
constexpr size_t QB_STAGE_BYTES = (size_t)QB_SLAB * (QB_SB + 1) * 4;
constexpr int QB_THREADS = 1024;
constexpr int QB_UNROLL = 32;

__device__ __forceinline__ void cp_async4(uint32_t *dst, const uint32_t *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}

// Load hist rows [cb, cb + nbc) of the slab's experts into the staging tile (consecutive
// threads on consecutive bins of one expert: coalesced), asynchronously; the NaN row's slot
// starts at 0.
__device__ __forceinline__ void qb_stage_load(uint32_t *stage, const uint32_t *hist, int e0, int ne, int nbins,
                                              int cb, int nbc) {
    for (int i = threadIdx.x; i < ne * nbc; i += blockDim.x) {
        const int e = i / nbc, bl = i - e * nbc, b = cb + bl;
        uint32_t *dst = stage + e * (QB_SB + 1) + bl;
        if (b < nbins) cp_async4(dst, hist + (int64_t)(e0 + e) * nbins + b);
        else *dst = 0u;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Histogram of one slab of 32 experts over this CTA's share of the tokens (see the file
// comment), then the cluster's reduction into hist.  CTA `rank` of the cluster owns counter
// rows [b_lo, b_hi) of the slab (the NaN row nbins included) and settles them in chunks of
// QB_SB rows: (0) the chunk's hist values are loaded into the staging tile, coalesced (for
// the first chunk this is issued before the counting and lands meanwhile); (1) threads with
// lane = expert add the P CTAs' counters of those rows (local and distributed shared memory,
// all ranks' loads in flight at once) into the tile; (2) the tile is stored back into hist,
// coalesced, and the NaN row goes to status[0].  Each CTA arrives at a closing cluster
// barrier once its last reads of the other CTAs' counters are done and waits on it just
// before it exits, so that every CTA's counters stay alive until the whole cluster has read
// them while the stores of (2) overlap the other CTAs' reads.  P = the cluster size.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
template <int P>
__global__ void __launch_bounds__(QB_THREADS, 1)
qb_hist_kernel(const float *__restrict__ scores, int64_t T, int E, int nbins,
               uint32_t *__restrict__ hist, int32_t *status) {
    extern __shared__ uint32_t hs[];                 // [nbins + 1][QB_SLAB], then the staging tile
    uint32_t *stage = hs + (nbins + 1) * QB_SLAB;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nwarps = QB_THREADS / 32;
    const int e0 = blockIdx.x * QB_SLAB;
    const int ne = min(QB_SLAB, E - e0);
    const float nb = (float)nbins, top_f = (float)(nbins - 1);
    const int64_t per_t = (T + P - 1) / P;
    const int64_t t0 = min(T, rank * per_t);
    const int64_t t1 = min(T, t0 + per_t);
    const int nrows = nbins + 1;
    const int per_b = (nrows + P - 1) / P;
    const int b_lo = min(nrows, rank * per_b), b_hi = min(nrows, b_lo + per_b);

    qb_stage_load(stage, hist, e0, ne, nbins, b_lo, min(QB_SB, b_hi - b_lo));

    // counting: lane = expert; each lane keeps QB_UNROLL row loads in flight.  The first batch
    // is issued before the counters are cleared.
    const bool active = lane < ne;
    const float *col = scores + e0 + (active ? lane : 0);
    uint32_t *h = hs + lane;
    int64_t t = t0 + warp;
    const bool full_batch = active && t + (QB_UNROLL - 1) * nwarps < t1;
    float v[QB_UNROLL];
    if (full_batch) {
#pragma unroll
        for (int u = 0; u < QB_UNROLL; ++u) v[u] = __ldcs(col + (t + u * nwarps) * (int64_t)E);
    }
    {
        uint4 *h4 = reinterpret_cast<uint4 *>(hs);
        for (int i = threadIdx.x; i < nrows * QB_SLAB / 4; i += QB_THREADS) h4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (full_batch) {
        for (;;) {
#pragma unroll
            for (int u = 0; u < QB_UNROLL; ++u) atomicAdd(h + qb_bin(v[u], nb, top_f, nbins) * QB_SLAB, 1u);
            t += QB_UNROLL * nwarps;
            if (t + (QB_UNROLL - 1) * nwarps >= t1) break;
#pragma unroll
            for (int u = 0; u < QB_UNROLL; ++u) v[u] = __ldcs(col + (t + u * nwarps) * (int64_t)E);
        }
    }
    if (active)
        for (; t < t1; t += nwarps) atomicAdd(h + qb_bin(__ldcs(col + t * (int64_t)E), nb, top_f, nbins) * QB_SLAB, 1u);
    asm volatile("cp.async.wait_all;" ::: "memory");
    cluster.sync();

    // the cluster's reduction of the owned rows: every load of a chunk (CH per thread from
    // each of the P CTAs) is issued before the first is used
    const uint32_t *src[P];
#pragma unroll
    for (int r = 0; r < P; ++r) src[r] = cluster.map_shared_rank(hs, r);
    // loads per thread and rank in flight: 7 x 1024 >= QB_SB x QB_SLAB; fewer for larger P, as
    // many as the 64 registers of a 1024-thread block hold without spilling
    constexpr int CH = P <= 4 ? 7 : P == 5 ? 5 : 3;
    bool overflow = false, arrived = false;
    uint32_t nan_count = 0;
    for (int cb = b_lo; cb < b_hi; cb += QB_SB) {
        const int nbc = min(QB_SB, b_hi - cb);
        if (cb != b_lo) {
            qb_stage_load(stage, hist, e0, ne, nbins, cb, nbc);
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncthreads();
        }
        for (int i0 = threadIdx.x; i0 < nbc * QB_SLAB; i0 += CH * QB_THREADS) {
            uint32_t c[CH][P];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int i = i0 + k * QB_THREADS;
#pragma unroll
                for (int r = 0; r < P; ++r) c[k][r] = i < nbc * QB_SLAB ? src[r][cb * QB_SLAB + i] : 0u;
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int i = i0 + k * QB_THREADS;
                if (i < nbc * QB_SLAB && (i & 31) < ne) {
                    uint32_t *slot = stage + (i & 31) * (QB_SB + 1) + (i >> 5);
                    uint64_t sum = *slot;
#pragma unroll
                    for (int r = 0; r < P; ++r) sum += c[k][r];
                    if (sum > 0xffffffffull) {
                        if (cb + (i >> 5) < nbins) overflow = true;
                        sum = 0xffffffffull;
                    }
                    *slot = (uint32_t)sum;
                }
            }
        }
        if (cb + QB_SB >= b_hi) {       // this CTA's last reads of the other CTAs' counters
            cluster_arrive_release();
            arrived = true;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < ne * nbc; i += QB_THREADS) {
            const int e = i / nbc, bl = i - e * nbc, b = cb + bl;
            const uint32_t val = stage[e * (QB_SB + 1) + bl];
            if (b < nbins) hist[(int64_t)(e0 + e) * nbins + b] = val;
            else nan_count += val;
        }
        __syncthreads();
    }
    // other CTAs of the cluster may still be reading this CTA's counters (a CTA that owns no
    // rows gets here at once): no CTA leaves before all of them are done
    if (!arrived) cluster_arrive_release();
    cluster_wait_acquire();
    if (status) {
        if (nan_count) atomicAdd(&status[ST_NAN], (int)nan_count);
        if (overflow) atomicExch(&status[ST_OVERFLOW], 1);
    }
}

// One cluster of P CTAs (16 where the device can place such a cluster, else 8); CTA r owns a
// contiguous range of experts and each warp takes
// one expert at a time.  Lane l holds the expert's bins l*B .. l*B + B - 1 in registers
// (16-byte loads when the rows allow); an inclusive warp scan of the lanes' sums gives the
// cumulative counts.  The arithmetic avoids fp64 (a small fraction of the fp32 rate on this
// part) without giving up exactness where it matters:
//   r = (1 - k/E) N = N - N k / E;  with N k = E qd + rm (integer division),
//   ceil(r) = N - qd exactly, so "first bin with C_j >= r" is an integer search, and
//   r - C_{j-1} = (N - qd - C_{j-1}) - rm / E is an integer minus a fraction in [0, 1),
//   so q = (j + (r - C_{j-1}) / h_j) / nbins is formed in fp32 with an error below 3e-7.
// The mean over experts is an exact fixed-point sum (q * 2^31 rounded to an integer, added in
// int64 in any order, so the result does not depend on the order), shared across the
// cluster through distributed shared memory.  No global scratch.
constexpr int QBU_CTAS = 16;                 // largest cluster tried
constexpr int QBU_MIN_CTAS = 8;
constexpr int QBU_MAXB = 1024 / 32;          // bins per lane (nbins <= 1024)
constexpr int QBU_THREADS = 512;
constexpr int QBU_MAX_PER_CTA = 8192 / QBU_MIN_CTAS;
constexpr float QBU_FIX = 2147483648.0f;     // 2^31

__global__ void __launch_bounds__(QBU_THREADS, 1)
qb_update_kernel(const uint32_t *__restrict__ hist, int E, int nbins, int k,
                 float *__restrict__ q_out, float *__restrict__ bias) {
    __shared__ float q_s[QBU_MAX_PER_CTA];
    __shared__ long long red[QBU_THREADS / 32];
    __shared__ long long part;
    cg::cluster_group cluster = cg::this_cluster();
    const int P = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (E + P - 1) / P;
    const int e0 = min(E, rank * per), e1 = min(E, e0 + per);
    const int B = (nbins + 31) / 32;             // bins owned by each lane, contiguous
    const int b0 = lane * B;
    // 16-byte loads: each lane's first bin and each expert's row start on a 16-byte boundary
    const bool vec = (B % 4) == 0 && (nbins % 4) == 0 && ((uintptr_t)hist & 15u) == 0;
    for (int e = e0 + w; e < e1; e += QBU_THREADS / 32) {
        const uint32_t *h = hist + (int64_t)e * nbins + b0;
        uint32_t v[QBU_MAXB];
        if (vec) {
#pragma unroll
            for (int i = 0; i < QBU_MAXB; i += 4) {
                uint4 t = make_uint4(0, 0, 0, 0);
                if (i < B && b0 + i < nbins) t = __ldg(reinterpret_cast<const uint4 *>(h + i));
                v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < QBU_MAXB; ++i) v[i] = (i < B && b0 + i < nbins) ? __ldg(h + i) : 0u;
        }
        unsigned long long S = 0;
#pragma unroll
        for (int i = 0; i < QBU_MAXB; ++i) S += v[i];
        unsigned long long inc = S;              // inclusive scan of the lanes' sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        const unsigned long long N = __shfl_sync(0xffffffffu, inc, 31);
        const unsigned long long nk = N * (unsigned long long)k;
        const unsigned long long qd = nk / (unsigned long long)E;
        const unsigned long long rm = nk - qd * (unsigned long long)E;
        const unsigned long long rc = N - qd;    // ceil(r); r > 0 exactly when rc >= 1
        float q = 0.0f;
        if (rc >= 1) {
            const unsigned m = __ballot_sync(0xffffffffu, inc >= rc);
            const int l = __ffs(m) - 1;          // the lane whose bins hold rank r
            float qq = 0.0f;
            if (lane == l) {
                unsigned long long C = inc - S;  // cumulative count before this lane's bins
                int j = b0;
                unsigned long long prev = C, hj = 1;
                bool found = false;
#pragma unroll
                for (int i = 0; i < QBU_MAXB; ++i) {
                    const unsigned long long before = C;
                    C += v[i];
                    const bool hit = !found && i < B && C >= rc;
                    if (hit) { j = b0 + i; prev = before; hj = v[i]; }
                    found = found || hit;
                }
                const float frac = (float)(rc - prev) - (float)rm / (float)E;
                qq = ((float)j + frac / (float)hj) / (float)nbins;
            }
            q = __shfl_sync(0xffffffffu, qq, l);
        }
        if (lane == 0) q_s[e - e0] = q;
    }
    __syncthreads();
    long long fx = 0;
    for (int i = tid; i < e1 - e0; i += blockDim.x) fx += __float2ll_rn(q_s[i] * QBU_FIX);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fx += __shfl_xor_sync(0xffffffffu, fx, o);
    if (lane == 0) red[w] = fx;
    __syncthreads();
    if (tid == 0) {
        long long t = 0;
        for (int i = 0; i < QBU_THREADS / 32; ++i) t += red[i];
        part = t;
    }
    cluster.sync();
    long long pv[QBU_CTAS];
#pragma unroll
    for (int r = 0; r < QBU_CTAS; ++r) pv[r] = r < P ? *cluster.map_shared_rank(&part, r) : 0;
    long long total = 0;
#pragma unroll
    for (int r = 0; r < QBU_CTAS; ++r) total += pv[r];
    const float cbar = (float)(total / E) * (1.0f / QBU_FIX);
    for (int e = e0 + tid; e < e1; e += blockDim.x) {
        const float qe = q_s[e - e0];
        bias[e] = cbar - qe;
        if (q_out) q_out[e] = qe;
    }
    cluster.sync();
}

}  // namespace

// Cluster size P (CTAs per 32-expert slab) of a histogram launch.  Every CTA needs a whole SM
// and a cluster's CTAs must share one GPC, so how many clusters of a given size fit at once
// depends on how the SMs are grouped (cudaOccupancyMaxActiveClusters): 28 clusters of 5 may
// need two waves where 28 clusters of 4 fit in one.  P minimises waves / P (the per-CTA work
// falls as 1 / P), fewer waves breaking ties.  Cached per device, kernel and shape.
using QbHistFn = void (*)(const float *, int64_t, int, int, uint32_t *, int32_t *);
static const QbHistFn kQbHist[QB_MAX_CLUSTER + 1] = {nullptr,           qb_hist_kernel<1>, qb_hist_kernel<2>,
                                                     qb_hist_kernel<3>, qb_hist_kernel<4>, qb_hist_kernel<5>,
                                                     qb_hist_kernel<6>, qb_hist_kernel<7>, qb_hist_kernel<8>};

static int qb_cluster_size(int nslabs, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, nslabs, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int best = 1;
    double best_cost = 1e30;
    int best_waves = 1 << 30;
    for (int P = 1; P <= QB_MAX_CLUSTER; ++P) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(nslabs, P, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = P;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kQbHist[P], &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            continue;
        }
        const int waves = (nslabs + n - 1) / n;
        const double cost = (double)waves / P;
        if (cost < best_cost - 1e-12 || (cost < best_cost + 1e-12 && waves < best_waves)) {
            best = P;
            best_cost = cost;
            best_waves = waves;
        }
    }
    cache[key] = best;
    return best;
}

int launch_qb_histogram(const float *scores, int64_t T, int E, int nbins, uint32_t *hist,
                        int32_t *status, cudaStream_t st) {
    if (T <= 0) return SLMOE_OK;
    const size_t smem = (size_t)QB_SLAB * (nbins + 1) * sizeof(uint32_t) + QB_STAGE_BYTES;
    for (int p = 1; p <= QB_MAX_CLUSTER; ++p) {
        cudaError_t e = cudaFuncSetAttribute(kQbHist[p], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb smem attribute: %s", cudaGetErrorString(e));
    }
    cudaError_t e;
    const int nslabs = (E + QB_SLAB - 1) / QB_SLAB;
    const int P = qb_cluster_size(nslabs, QB_THREADS, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nslabs, P, 1);
    cfg.blockDim = dim3(QB_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = P;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kQbHist[P], scores, T, E, nbins, hist, status);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb histogram launch: %s", cudaGetErrorString(e));
    return check_launch("qb_histogram");
}

// Cluster size of the bias update: 16 CTAs when the device can place a cluster of 16 such
// CTAs (a non-portable size), else 8.  Looked up once per device.
static int qb_update_cluster_size() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int P = QBU_MIN_CTAS;
    if (cudaFuncSetAttribute(qb_update_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(QBU_CTAS, 1, 1);
        cfg.blockDim = dim3(QBU_THREADS, 1, 1);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = QBU_CTAS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, qb_update_kernel, &cfg) == cudaSuccess && n >= 1) P = QBU_CTAS;
    }
    cudaGetLastError();
    cache[dev] = P;
    return P;
}

int launch_qb_update(const uint32_t *hist, int E, int nbins, int k, float *q_out, float *bias,
                     cudaStream_t st) {
    const int P = qb_update_cluster_size();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P, 1, 1);
    cfg.blockDim = dim3(QBU_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, qb_update_kernel, hist, E, nbins, k, q_out, bias);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb update launch: %s", cudaGetErrorString(e));
    return check_launch("qb_update");
}

// ---------------------------------------------------------------- fixed-step (SignSGD) update
// The rule QB replaces ([K3-news] §02: K2 moves each expert's selection bias by a fixed step,
// up or down): bias[e] += step * sign(N - E * counts[e]), N = sum of the counts, i.e. the sign
// of (mean load - load of e), taken in exact int64 arithmetic; bias is left untouched where
// the load equals the mean.  One block: the threads sum the counts (int64), then each updates
// its experts with one fp32 add.
constexpr int SG_THREADS = 1024;

__global__ void __launch_bounds__(SG_THREADS) signsgd_update_kernel(const int32_t *__restrict__ counts, int E,
                                                                    float step, float *__restrict__ bias) {
    __shared__ long long wsum[SG_THREADS / 32];
    __shared__ long long total;
    long long acc = 0;
    for (int e = threadIdx.x; e < E; e += SG_THREADS) acc += counts[e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) wsum[w] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long t = 0;
        for (int i = 0; i < SG_THREADS / 32; ++i) t += wsum[i];
        total = t;
    }
    __syncthreads();
    const long long N = total;
    for (int e = threadIdx.x; e < E; e += SG_THREADS) {
        const long long diff = N - (long long)E * counts[e];
        if (diff > 0) bias[e] = __fadd_rn(bias[e], step);
        else if (diff < 0) bias[e] = __fadd_rn(bias[e], -step);
    }
}

int launch_signsgd_update(const int32_t *counts, int E, float step, float *bias, cudaStream_t st) {
    signsgd_update_kernel<<<1, SG_THREADS, 0, st>>>(counts, E, step, bias);
    return check_launch("signsgd_update");
}

}  // namespace slmoe
