// Quantile Balancing: per-expert score histograms and the bias update.
//
// K3 architecture write-up, 负载均衡优化: scores in [0, 1] are binned (1000 bins suffice), the
// target quantile is read from the binned distribution, and histograms add across
// micro-batches and machines.  The bias update (b_e <- mean(q) - q_e) is this library's
// fixed reading; the pages defer the exact rule to a technical report.
//
// Histogram design.  scores [T, E] fp32 is streamed once from HBM.  The experts are cut
// into slabs of 32 (one 128-byte line per row: lane = expert), and each slab is counted by
// one thread-block cluster of P CTAs that split the tokens (P is chosen so that the
// clusters fill the SMs).  Each CTA keeps 32-bit counters [bin][32 experts] in shared
// memory, so the 32 lanes of an atomic always hit 32 distinct banks, and keeps 32 row
// loads in flight per lane.  At the end the cluster adds its CTAs' counters through
// distributed shared memory and each bin of global memory is read-modified-written by
// exactly one thread: no global atomics and no partial histograms in HBM.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace slmoe {
namespace {

constexpr int QB_SLAB = 32;
constexpr int QB_THREADS = 1024;
constexpr int QB_MAX_CLUSTER = 8;
constexpr int QB_UNROLL = 32;

__global__ void __launch_bounds__(QB_THREADS, 1)
qb_hist_kernel(const float *__restrict__ scores, int64_t T, int E, int nbins,
               uint32_t *__restrict__ hist, int32_t *status) {
    extern __shared__ uint32_t hs[];                 // [nbins][QB_SLAB]
    cg::cluster_group cluster = cg::this_cluster();
    const int P = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = QB_THREADS / 32;
    const int e0 = blockIdx.x * QB_SLAB;
    const int ne = min(QB_SLAB, E - e0);
    const float nb = (float)nbins;
    const int top = nbins - 1;
    int nan_count = 0;
    bool overflow = false;

    for (int i = tid; i < QB_SLAB * nbins; i += QB_THREADS) hs[i] = 0u;
    __syncthreads();
    const int64_t per = (T + P - 1) / P;
    const int64_t t0 = rank * per;
    const int64_t t1 = min(T, t0 + per);
    if (lane < ne) {
        const float *col = scores + e0 + lane;
        uint32_t *h = hs + lane;
        int64_t t = t0 + warp;
        for (; t + (QB_UNROLL - 1) * nwarps < t1; t += QB_UNROLL * nwarps) {
            float v[QB_UNROLL];
#pragma unroll
            for (int u = 0; u < QB_UNROLL; ++u) v[u] = __ldcs(col + (t + u * nwarps) * (int64_t)E);
#pragma unroll
            for (int u = 0; u < QB_UNROLL; ++u) {
                // one IEEE fp32 round-to-nearest multiply, floor, clamp to [0, nbins-1]
                const int b = min(max(__float2int_rd(__fmul_rn(v[u], nb)), 0), top);
                if (isnan(v[u])) ++nan_count;
                else atomicAdd(&h[b * QB_SLAB], 1u);
            }
        }
        for (; t < t1; t += nwarps) {
            const float v = __ldcs(col + t * (int64_t)E);
            const int b = min(max(__float2int_rd(__fmul_rn(v, nb)), 0), top);
            if (isnan(v)) ++nan_count;
            else atomicAdd(&h[b * QB_SLAB], 1u);
        }
    }
    cluster.sync();
    // each CTA of the cluster adds a share of the slab's bins across all CTAs
    const int total = ne * nbins;
    const int share = (total + P - 1) / P;
    const int f0 = rank * share, f1 = min(total, f0 + share);
    for (int f = f0 + tid; f < f1; f += QB_THREADS) {
        const int b = f / ne, e = f - b * ne;
        uint64_t sum = 0;
        for (int r = 0; r < P; ++r) sum += cluster.map_shared_rank(hs, r)[b * QB_SLAB + e];
        if (sum) {
            uint32_t *g = hist + (int64_t)(e0 + e) * nbins + b;
            uint64_t nv = (uint64_t)*g + sum;
            if (nv > 0xffffffffull) { overflow = true; nv = 0xffffffffull; }
            *g = (uint32_t)nv;
        }
    }
    cluster.sync();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nan_count += __shfl_xor_sync(0xffffffffu, nan_count, o);
    if (status) {
        if (lane == 0 && nan_count) atomicAdd(&status[ST_NAN], nan_count);
        if (overflow) atomicExch(&status[ST_OVERFLOW], 1);
    }
}

// One cluster of QBU_CTAS CTAs; CTA r owns a contiguous range of experts.  A warp loads an
// expert's whole histogram into registers up front (lane l holds bins l, l + 32, ...), then
// walks the 32-bin chunks with an inclusive warp scan until the cumulative count reaches
// r = (1 - k/E) N_e, and interpolates inside that bin, in fp64.  The mean over experts is a
// fixed-order sum: per CTA in shared memory, then across the cluster's CTAs in rank order
// through distributed shared memory.  No global scratch.
constexpr int QBU_CTAS = 8;
constexpr int QBU_MAXB = 1024 / 32;          // bins per lane (nbins <= 1024)
constexpr int QBU_THREADS = 512;
constexpr int QBU_STAGE_WORDS = (QBU_THREADS / 32) * QBU_MAXB * 33;

__global__ void __launch_bounds__(QBU_THREADS, 1)
qb_update_kernel(const uint32_t *__restrict__ hist, int E, int nbins, int k,
                 float *__restrict__ q_out, float *__restrict__ bias) {
    // dynamic shared memory: per-warp staging tiles, then q of this CTA's experts
    extern __shared__ uint32_t dyn[];
    __shared__ double red[QBU_THREADS / 32];
    __shared__ double part;
    uint32_t *stage = dyn;
    double *q_s = reinterpret_cast<double *>(dyn + QBU_STAGE_WORDS);
    cg::cluster_group cluster = cg::this_cluster();
    const int P = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (E + P - 1) / P;
    const int e0 = rank * per, e1 = min(E, e0 + per);
    const double p = 1.0 - (double)k / (double)E;
    const int B = (nbins + 31) / 32;             // bins owned by each lane, contiguous
    const int b0 = lane * B;
    // per-warp staging tile: bin b at word b + b / 32 (one pad word per 32 bins) so that the
    // coalesced stores and the lane-contiguous reads are both free of bank conflicts
    uint32_t *tile = stage + w * (QBU_MAXB * 33);
    for (int e = e0 + w; e < e1; e += QBU_THREADS / 32) {
        const uint32_t *h = hist + (int64_t)e * nbins;
        uint32_t ld[QBU_MAXB];                   // all loads first: one memory latency
#pragma unroll
        for (int i = 0; i < QBU_MAXB; ++i) {
            const int b = i * 32 + lane;
            ld[i] = (i < B && b < nbins) ? __ldg(h + b) : 0u;
        }
#pragma unroll
        for (int i = 0; i < QBU_MAXB; ++i)
            if (i < B) tile[i * 32 + lane + i] = ld[i];
        __syncwarp();
        uint32_t v[QBU_MAXB];
        unsigned long long S = 0;
#pragma unroll
        for (int i = 0; i < QBU_MAXB; ++i) {
            const int b = b0 + i;
            v[i] = (i < B) ? tile[b + (b >> 5)] : 0u;
            S += v[i];
        }
        __syncwarp();
        unsigned long long inc = S;              // inclusive scan of the lanes' sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        const unsigned long long N = __shfl_sync(0xffffffffu, inc, 31);
        const double r = p * (double)N;
        double q = 0.0;
        if (r > 0.0) {
            // C_j >= r  <=>  C_j >= ceil(r) for integer counts: the search is integer-only
            // (fp64 is slow on this part) and decides exactly as the fp64 comparison would
            const unsigned long long rc = (unsigned long long)ceil(r);
            const unsigned m = __ballot_sync(0xffffffffu, inc >= rc);
            const int l = __ffs(m) - 1;          // the lane whose bins hold rank r
            double qq = 0.0;
            if (lane == l) {
                unsigned long long C = inc - S;  // cumulative count before this lane's bins
                int j = 0;
                unsigned long long prev = C, hj = 1;
                bool done = false;
#pragma unroll
                for (int i = 0; i < QBU_MAXB; ++i) {
                    if (!done && i < B) {
                        const unsigned long long before = C;
                        C += v[i];
                        if (C >= rc) { j = b0 + i; prev = before; hj = v[i]; done = true; }
                    }
                }
                qq = ((double)j + (r - (double)prev) / (double)hj) / (double)nbins;
            }
            q = __shfl_sync(0xffffffffu, qq, l);
        }
        if (lane == 0) q_s[e - e0] = q;
    }
    __syncthreads();
    double s = 0.0;
    for (int i = tid; i < e1 - e0; i += blockDim.x) s += q_s[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[w] = s;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int i = 0; i < QBU_THREADS / 32; ++i) t += red[i];
        part = t;
    }
    cluster.sync();
    double total = 0.0;
    for (int r = 0; r < P; ++r) total += *cluster.map_shared_rank(&part, r);
    const double cbar = total / (double)E;
    for (int e = e0 + tid; e < e1; e += blockDim.x) {
        bias[e] = (float)(cbar - q_s[e - e0]);
        if (q_out) q_out[e] = (float)q_s[e - e0];
    }
    cluster.sync();
}

}  // namespace

int launch_qb_histogram(const float *scores, int64_t T, int E, int nbins, uint32_t *hist,
                        int32_t *status, cudaStream_t st) {
    if (T <= 0) return SLMOE_OK;
    const size_t smem = (size_t)QB_SLAB * nbins * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(qb_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb smem attribute: %s", cudaGetErrorString(e));
    const int nslabs = (E + QB_SLAB - 1) / QB_SLAB;
    int P = sm_count() / nslabs;
    P = P < 1 ? 1 : (P > QB_MAX_CLUSTER ? QB_MAX_CLUSTER : P);
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
    e = cudaLaunchKernelEx(&cfg, qb_hist_kernel, scores, T, E, nbins, hist, status);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb histogram launch: %s", cudaGetErrorString(e));
    return check_launch("qb_histogram");
}

int launch_qb_update(const uint32_t *hist, int E, int nbins, int k, float *q_out, float *bias,
                     cudaStream_t st) {
    const size_t smem = QBU_STAGE_WORDS * sizeof(uint32_t) +
                        (size_t)((E + QBU_CTAS - 1) / QBU_CTAS) * sizeof(double);
    cudaError_t e = cudaFuncSetAttribute(qb_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb update smem: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(QBU_CTAS, 1, 1);
    cfg.blockDim = dim3(QBU_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = QBU_CTAS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, qb_update_kernel, hist, E, nbins, k, q_out, bias);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "qb update launch: %s", cudaGetErrorString(e));
    return check_launch("qb_update");
}

}  // namespace slmoe
