// Backward pass of the Stable LatentMoE layer, bf16 layer type (sm_103a).
//
// The gradient is the chain rule of the forward (K3 architecture write-up, SiTU激活优化 /
// 归一化策略调整; the concept note's 训练基础设施 trains this layer), run against the
// intermediates a forward call leaves in its workspace.  The contractions reuse the forward's
// tcgen05 kernels (tc_gemm.cu): the dense kernel with MN-major operands and fp32, accumulating
// or SiTU-GLU-derivative epilogues for the dense gradients, and the grouped kernel over the
// forward's work lists for the routed experts' pre-activations (recomputed in fp32: near
// saturation the derivatives of SiTU and of the soft cap change by a few per cent across one
// bf16 step of their argument), dh with the SiTU-GLU derivative, and the x_lat gradient of
// each slot.  This file adds the routed experts' weight gradients (wgrad_kernel: per expert,
// K = the expert's own rows) and the memory-bound steps as plain kernels: RMSNorm + combine
// backward (dc, the gradient of each expert output, of each gate weight, and per-block dgamma
// sums), the per-token sum of the k slot gradients of x_lat, and the router (gate
// renormalisation, sigmoid, the router's share of dx and dW_r).  Every reduction runs in a
// fixed order, so results do not depend on scheduling.
#include <cuda_bf16.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_gemm.h"
#include "tcgen05.cuh"
#include "tmap.h"

namespace slmoe {
namespace {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- routed weight gradients
// wgrad_kernel: for each expert e, C_e^T = A_e^T B_e with K = the expert's own rows in
// expert-sorted order (offsets[e] .. offsets[e + 1]): a tile is 128 M (A's features: the MMA's
// M, the gradient's contiguous dimension) x 256 N (B's features), K in blocks of 64.  A and B
// are stored [rows, features] (MN-major operands); A's rows may be gathered through an index,
// B's are contiguous and come by TMA in 64 x 64 boxes.  Four loader warps fill a 4-stage ring
// (A by cp.async, 16-byte chunks zero-filled past the segment), one thread issues the MMAs
// into a double-buffered TMEM accumulator, and eight epilogue warps (two per lane quadrant,
// half the columns each) drain the fp32 tile transposed: 16 gradient rows (tile columns) at a
// time, each warp stages its 32 M lanes of them in shared memory ([16 rows][32 M], two 2 KB
// buffers per warp) and its first lane writes them by TMA (a 32 x 16 box of the gradient seen
// as [E * N rows, M], full 128-byte lines; added in by a TMA reduction when accumulating), so
// that no warp waits on another.  The kernel is bound by
// those fp32 writes (19.7 GB at K3): stored by the epilogue warps themselves they stalled the
// warps on the memory system (4.3 TB/s, where a plain store stream of the same pattern
// reaches 6.5 TB/s).
constexpr int WG_BN = 256;
constexpr int WG_STAGES = 4;
constexpr int WG_A_BYTES = 128 * 128;              // 128 M x 64 K
constexpr int WG_B_BYTES = WG_BN * 128;            // 256 N x 64 K
constexpr int WG_STAGE = WG_A_BYTES + WG_B_BYTES;
constexpr int WG_LOADERS = 128;                    // warps 0-3
constexpr int WG_MMA_WARP = 4;
constexpr int WG_EPI_WARP0 = 5;                    // warps 5-12
constexpr int WG_EPI_WARPS = 8;
constexpr int WG_THREADS = (WG_EPI_WARP0 + WG_EPI_WARPS) * 32;
constexpr int WG_Q = 4;
constexpr int WG_O_CHUNK = 16 * 32 * 4;             // 16 gradient rows x 32 M, fp32
constexpr int WG_O_BYTES = 2 * WG_EPI_WARPS * WG_O_CHUNK;   // two buffers per epilogue warp
constexpr int WG_SMEM = WG_STAGES * WG_STAGE + WG_O_BYTES + 1024 + 512;
static_assert(WG_SMEM <= 232448, "shared memory");
constexpr int WG_BAND = 8;                         // M tiles per band of an expert's tile order
constexpr int A_MN_ = 1, B_MN_ = 2;                // tc_dense_gemm operand majorness

// One operand as stored: lines of ld elements; index (nullable) maps a line number to the
// stored line.
struct BOp {
    const bf16 *p;
    long long ld;
    const int32_t *index;
};

struct WArgs {
    BOp A, B;
    int M, N;                // per expert: gradient tile space M x N
    int tiles_m, tiles_n;    // 128 x 256 tiles
    int units;               // E * tiles_m * tiles_n
    const int32_t *offsets;  // per-expert row segments [E + 1]
    int *counter;            // zeroed work counter
    float *C;                // expert e's gradient at C + e * cstride, stored [N][M] (row pitch ldc)
    long long ldc, cstride;
    int accumulate;          // add into C instead of storing
    int32_t *status;
    unsigned long long wait_limit_ns;
};

struct WItem {
    int e, m0, n0, mv, nv, kr0, klen;   // e < 0: end of work
};

__device__ __forceinline__ WItem fetch_item(const WArgs &a) {
    WItem it;
    it.e = -1;
    const int u = atomicAdd(a.counter, 1);
    if (u >= a.units) return it;
    const int per = a.tiles_m * a.tiles_n;
    it.e = u / per;
    // bands of WG_BAND M tiles, M fastest inside a band: the tiles in flight share B strips
    const int t = u - it.e * per;
    const int per_band = WG_BAND * a.tiles_n;
    const int band = t / per_band;
    const int m_first = band * WG_BAND;
    const int bm = min(WG_BAND, a.tiles_m - m_first);
    const int r = t - band * per_band;
    it.m0 = (m_first + r % bm) * 128;
    it.n0 = (r / bm) * WG_BN;
    it.mv = min(128, a.M - it.m0);
    it.nv = min(WG_BN, a.N - it.n0);
    it.kr0 = a.offsets[it.e];
    it.klen = a.offsets[it.e + 1] - it.kr0;
    return it;
}

// The A tile of one stage (64 K rows x 128 M, MN-major: a line of 64 M values per K row, two
// 64-wide groups, 128-byte swizzle) by cp.async; t = loader thread 0..127.  Thread t copies
// chunk t % 16 of K rows t / 16 + 8 i (i < 8): a_lines gives the stored lines of those rows
// (through the index when A is gathered; rows past the segment repeat its first row and are
// zero-filled), so that the index loads of the next K block can be in flight while this one
// is issued.
__device__ __forceinline__ void a_lines(const BOp &op, int kr0, int k0, int klen, int t, int (&lines)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int kr = (t >> 4) + 8 * i;
        const int krow = kr0 + k0 + (k0 + kr < klen ? kr : 0);
        lines[i] = op.index ? op.index[krow] : krow;
    }
}
__device__ __forceinline__ void load_a(uint32_t sbase, const BOp &op, int m0, int mv, int k0, int klen, int t,
                                       const int (&lines)[8]) {
    const int w = t & 15;
    const int g = w >> 3, c = w & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int kr = (t >> 4) + 8 * i;
        const bool ok = k0 + kr < klen && 64 * g + 8 * c < mv;
        const long long col = ok ? m0 + 64 * g + 8 * c : m0;
        const uint32_t dst = sbase + g * 8192 + (kr >> 3) * 1024 + (kr & 7) * 128 + ((c ^ (kr & 7)) << 4);
        const bf16 *src = op.p + (long long)lines[i] * op.ld + (ok ? col : 0);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16u : 0u)
                     : "memory");
    }
}

// B rows past the expert's segment (TMA boxes of 64 K rows) hold other experts' values; they
// meet the zero-filled rows of A past the segment, so they add nothing.
// cmap: the gradients as one fp32 matrix [E * N rows, M] (expert e's row n at e * N + n),
// boxes of 32 x 16, no swizzle.
__global__ void __launch_bounds__(WG_THREADS, 1) wgrad_kernel(const __grid_constant__ CUtensorMap bmap,
                                                              const __grid_constant__ CUtensorMap cmap,
                                                              const WArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sO = smem + WG_STAGES * WG_STAGE;        // output staging
    WItem *q_items = reinterpret_cast<WItem *>(sO + WG_O_BYTES);
    uint64_t *q_full = reinterpret_cast<uint64_t *>(q_items + WG_Q);
    uint64_t *q_empty = q_full + WG_Q;
    uint64_t *full = q_empty + WG_Q;
    uint64_t *empty = full + WG_STAGES;
    uint64_t *tfull = empty + WG_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_drain + 1);
    volatile WaitCtl *wc = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < WG_Q; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 4 + 1 + WG_EPI_WARPS);   // loader warps, MMA thread, epilogue warps
        }
        for (int s = 0; s < WG_STAGES; ++s) {
            mbar_init(&full[s], WG_LOADERS + 1);             // A's cp.async arrivals + B's TMA
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], WG_EPI_WARPS);
        }
        mbar_init(mma_drain, 1);
        wait_ctl_init(wc, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == WG_MMA_WARP) tmem_alloc(tmem_slot, 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;

    auto pop = [&](int &qs, uint32_t &qp, WItem &it, bool warp_wide) -> bool {
        if (!mbar_wait(&q_full[qs], qp, wc)) return false;
        it = q_items[qs];
        if (warp_wide) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qs]);
        } else {
            mbar_arrive(&q_empty[qs]);
        }
        if (++qs == WG_Q) { qs = 0; qp ^= 1; }
        return true;
    };

    int l_stage = 0;                  // loader ring position, kept for the drain of TMA copies
    uint32_t l_phase = 0;
    bool l_wrapped = false;
    if (warp < 4) {
        // ------------------------------------------------ loaders (warp 0 lane 0 also fetches)
        const int t = threadIdx.x;
        int qs = 0, fs = 0;
        int &stage = l_stage;
        uint32_t qp = 0, fp = 0;
        uint32_t &phase = l_phase;
        for (;;) {
            if (warp == 0) {
                int ok = 1;
                if (lane == 0) {
                    const WItem nx = fetch_item(a);
                    if (mbar_wait(&q_empty[fs], fp ^ 1, wc)) {
                        q_items[fs] = nx;
                        mbar_arrive(&q_full[fs]);
                    } else {
                        ok = 0;
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (++fs == WG_Q) { fs = 0; fp ^= 1; }
            }
            WItem it;
            if (!pop(qs, qp, it, true)) break;
            if (it.e < 0) break;
            const int nkb = (it.klen + 63) / 64;
            bool aborted = false;
            int lines[8];
            if (nkb > 0) a_lines(a.A, it.kr0, 0, it.klen, t, lines);
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1, wc)) { aborted = true; break; }
                const uint32_t sa = su32(smem + stage * WG_STAGE);
                const uint32_t sb = sa + WG_A_BYTES;
                load_a(sa, a.A, it.m0, it.mv, kb * 64, it.klen, t, lines);
                if (kb + 1 < nkb) a_lines(a.A, it.kr0, (kb + 1) * 64, it.klen, t, lines);
                if (t == 0) {
                    mbar_expect_tx(&full[stage], WG_B_BYTES);
#pragma unroll
                    for (int g = 0; g < WG_BN / 64; ++g)
                        tma_load_2d(sb + g * 8192, &bmap, &full[stage], it.n0 + 64 * g, it.kr0 + kb * 64);
                }
                cp_async_arrive_noinc(&full[stage]);
                if (++stage == WG_STAGES) { stage = 0; phase ^= 1; l_wrapped = true; }
            }
            if (aborted) break;
        }
        cp_async_wait_all();
    } else if (warp == WG_MMA_WARP) {
        if (lane == 0) {
            int qs = 0, stage = 0, buf = 0;
            uint32_t qp = 0, phase = 0, tph = 0;
            constexpr uint32_t IDESC = idesc_bf16(128, WG_BN) | (1u << 15) | (1u << 16);   // A, B MN-major
            for (;;) {
                WItem it;
                if (!pop(qs, qp, it, false)) break;
                if (it.e < 0) break;
                const int nkb = (it.klen + 63) / 64;
                if (nkb == 0) continue;                    // nothing to accumulate (empty expert)
                if (!mbar_wait(&tempty[buf], tph ^ 1, wc)) break;
                tc_after();
                const uint32_t d = tmem_base + buf * 256;
                bool aborted = false;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, wc)) { aborted = true; break; }
                    fence_proxy_async();
                    tc_after();
                    const uint32_t sa = su32(smem + stage * WG_STAGE);
                    const uint32_t sb = sa + WG_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma(d, mn_desc(sa + kk * 2048, 8192), mn_desc(sb + kk * 2048, 8192), IDESC,
                             (kb > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == WG_STAGES) { stage = 0; phase ^= 1; }
                }
                if (aborted) break;
                umma_commit(&tfull[buf]);
                if (++buf == 2) { buf = 0; tph ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue: warp w drains TMEM lanes
        // 32 (w % 4) .. + 31 (tile rows M of that quadrant), columns 128 h .. 128 h + 127
        const int q = warp & 3;
        const int h = (warp - WG_EPI_WARP0) >> 2;
        const int i = q * 32 + lane;
        uint8_t *stg_w = sO + (warp - WG_EPI_WARP0) * 2 * WG_O_CHUNK;   // this warp's two buffers
        int ocnt = 0;
        int qs = 0, buf = 0;
        uint32_t qp = 0, tph = 0;
        for (;;) {
            WItem it;
            if (!pop(qs, qp, it, true)) break;
            if (it.e < 0) break;
            const int nkb = (it.klen + 63) / 64;
            const bool row_ok = i < it.mv;
            const int m = it.m0 + i;
            const int c_end = min(it.nv, 128 * h + 128);
            float *C = a.C + (long long)it.e * a.cstride;
            if (nkb == 0) {
                // an expert without rows: its weight-gradient tile is zero (stored unless adding)
                if (!a.accumulate && row_ok)
                    for (int j = 128 * h; j < c_end; ++j) C[(long long)(it.n0 + j) * a.ldc + m] = 0.f;
                continue;
            }
            if (!mbar_wait(&tfull[buf], tph, wc)) break;
            tc_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + buf * 256;
            const int grow0 = it.e * a.N + it.n0;       // the tile's first row in cmap
            const bool warp_ok = it.m0 + q * 32 < a.M;  // the warp's 32 M lanes start inside M
            for (int c0 = 128 * h; c0 < c_end; c0 += 64) {
                uint32_t r[4][16];
#pragma unroll
                for (int u = 0; u < 4; ++u) TMEM_LD16(tb + c0 + 16 * u, r[u]);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cu = c0 + 16 * u;
                    if (cu >= c_end) break;                  // the same for every warp of the half
                    if (c_end - cu < 16) {
                        // a partial block of gradient rows (N not a multiple of 16): direct
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (row_ok && j < c_end - cu) {
                                float *o = C + (long long)(it.n0 + cu + j) * a.ldc + m;
                                *o = __uint_as_float(r[u][j]) + (a.accumulate ? *o : 0.f);
                            }
                        continue;
                    }
                    float *stg = reinterpret_cast<float *>(stg_w + (ocnt & 1) * WG_O_CHUNK);
                    if (lane == 0) bulk_wait_read1();   // the write two chunks back has read this buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 16; ++j) stg[j * 32 + lane] = __uint_as_float(r[u][j]);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0 && warp_ok) {   // columns past M are cut off by the map's bounds
                        if (a.accumulate) tma_reduce_add_2d(&cmap, su32(stg), it.m0 + q * 32, grow0 + cu);
                        else tma_store_2d(&cmap, su32(stg), it.m0 + q * 32, grow0 + cu);
                        bulk_commit();
                    }
                    ++ocnt;
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            if (++buf == 2) { buf = 0; tph ^= 1; }
        }
    }
    bulk_wait_all();   // output writes read shared memory until they complete
    __syncthreads();
    if (wc->abort) {   // let copies and MMAs in flight finish before TMEM is freed
        if (threadIdx.x == 0) drain_ring(full, WG_STAGES, l_stage, l_phase, l_wrapped);
        if (warp == WG_MMA_WARP && lane == 0) {
            umma_commit(mma_drain);
            mbar_wait_drain(mma_drain, 0);
        }
        __syncthreads();
    }
    if (warp == WG_MMA_WARP) {
        tc_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && wc->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// ---------------------------------------------------------------- memory-bound steps
__global__ void f32_to_bf16_kernel(const float *__restrict__ in, bf16 *__restrict__ out, long long n) {
    for (long long i = (blockIdx.x * (long long)blockDim.x + threadIdx.x) * 4; i < n;
         i += (long long)gridDim.x * blockDim.x * 4) {
        if (i + 4 <= n) {
            const float4 v = *reinterpret_cast<const float4 *>(in + i);
            *reinterpret_cast<uint2 *>(out + i) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
        } else {
            for (long long j = i; j < n; ++j) out[j] = __float2bfloat16_rn(in[j]);
        }
    }
}

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
}

// RMSNorm + combine backward, RB_TOK tokens per block in order, 8 features per thread and
// chunk (16-byte loads and stores).  Per token: c = sum_j g_j y_e (fp32, slot order, as the
// forward combine), r = sqrt(mean c^2 + eps), A = sum_i gamma_i dz_i c_i;
// dc = gamma dz / r - c A / (n r^3); the expert-row gradient g_j dc (bf16, at the row's
// position in expert order), the gate-weight gradient dc . y_e(t, j), and the block's dgamma
// sum of dz c / r (one row per block, added across blocks in order by dgamma_reduce_kernel).
constexpr int RB_TOK = 32;
constexpr int RB_MAXCH = 4;          // 8-feature chunks per thread: d_latent <= 8 * 256 * 4
template <int MAXCH>
__global__ void __launch_bounds__(256) rms_combine_bwd_kernel(
    const bf16 *__restrict__ y_e, const float *__restrict__ topk_w, const int32_t *__restrict__ slot_pos,
    const float *__restrict__ gamma, const float *__restrict__ dz, int T, int dl, int k, float eps,
    bf16 *__restrict__ dye, float *__restrict__ dg, float *__restrict__ dgamma_part) {
    constexpr int GRP = 8 / MAXCH;   // slot rows loaded together: 8 loads in flight per thread
    __shared__ float red[64];
    __shared__ float redk[8][32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nch = dl / 8;
    float dgp[MAXCH][8];
#pragma unroll
    for (int u = 0; u < MAXCH; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) dgp[u][v] = 0.f;
    const int t0 = blockIdx.x * RB_TOK;
    for (int t = t0; t < min(T, t0 + RB_TOK); ++t) {
        const int32_t *sp = slot_pos + (long long)t * k;
        const float *gw = topk_w + (long long)t * k;
        const float *dzt = dz + (long long)t * dl;
        float cv[MAXCH][8];
        float ss = 0.f, A = 0.f;
#pragma unroll
        for (int u = 0; u < MAXCH; ++u)
#pragma unroll
            for (int v = 0; v < 8; ++v) cv[u][v] = 0.f;
        // the slots' rows GRP at a time, all loaded before any is added; the adds stay in slot
        // order
        for (int j0 = 0; j0 < k; j0 += GRP) {
            uint4 qv[MAXCH][GRP];
#pragma unroll
            for (int g = 0; g < GRP; ++g) {
                const long long r0 = j0 + g < k ? (long long)sp[j0 + g] * dl : 0;
#pragma unroll
                for (int u = 0; u < MAXCH; ++u) {
                    const int ch = tid + u * 256;
                    if (j0 + g < k && ch < nch) qv[u][g] = *reinterpret_cast<const uint4 *>(y_e + r0 + 8 * ch);
                }
            }
#pragma unroll
            for (int g = 0; g < GRP; ++g) {
                if (j0 + g >= k) break;
                const float wj = gw[j0 + g];
#pragma unroll
                for (int u = 0; u < MAXCH; ++u) {
                    if (tid + u * 256 >= nch) continue;
                    const bf16 *b = reinterpret_cast<const bf16 *>(&qv[u][g]);
#pragma unroll
                    for (int v = 0; v < 8; ++v) cv[u][v] += wj * __bfloat162float(b[v]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < MAXCH; ++u) {
            const int ch = tid + u * 256;
            if (ch < nch) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    ss += cv[u][v] * cv[u][v];
                    A += gamma[8 * ch + v] * dzt[8 * ch + v] * cv[u][v];
                }
            }
        }
        ss = block_sum(ss, red);
        A = block_sum(A, red + 32);
        const float r = sqrtf(ss / (float)dl + eps);
        const float ir = 1.0f / r;
        const float coef = A / ((float)dl * r * r * r);
        float dc[MAXCH][8];
#pragma unroll
        for (int u = 0; u < MAXCH; ++u) {
            const int ch = tid + u * 256;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float dzv = ch < nch ? dzt[8 * ch + v] : 0.f;
                const float gm = ch < nch ? gamma[8 * ch + v] : 0.f;
                dc[u][v] = gm * dzv * ir - cv[u][v] * coef;
                dgp[u][v] += dzv * cv[u][v] * ir;
            }
        }
        // slot by slot: dy_e = g_j dc, and the gate-weight gradient's partial dot product,
        // summed over the warp at once (no per-slot accumulators held across the slots); the
        // rows are read again GRP slots at a time, loads first
        for (int j0 = 0; j0 < k; j0 += GRP) {
            uint4 qv[MAXCH][GRP];
#pragma unroll
            for (int g = 0; g < GRP; ++g) {
                const long long r0 = j0 + g < k ? (long long)sp[j0 + g] * dl : 0;
#pragma unroll
                for (int u = 0; u < MAXCH; ++u) {
                    const int ch = tid + u * 256;
                    if (j0 + g < k && ch < nch) qv[u][g] = *reinterpret_cast<const uint4 *>(y_e + r0 + 8 * ch);
                }
            }
#pragma unroll
            for (int g = 0; g < GRP; ++g) {
                if (j0 + g >= k) break;
                const int j = j0 + g;
                const float gj = gw[j];
                const long long r0 = (long long)sp[j] * dl;
                float dot = 0.f;
#pragma unroll
                for (int u = 0; u < MAXCH; ++u) {
                    const int ch = tid + u * 256;
                    if (ch >= nch) continue;
                    const bf16 *b = reinterpret_cast<const bf16 *>(&qv[u][g]);
#pragma unroll
                    for (int v = 0; v < 8; ++v) dot += dc[u][v] * __bfloat162float(b[v]);
                    *reinterpret_cast<uint4 *>(dye + r0 + 8 * ch) =
                        make_uint4(pack_bf16(gj * dc[u][0], gj * dc[u][1]), pack_bf16(gj * dc[u][2], gj * dc[u][3]),
                                   pack_bf16(gj * dc[u][4], gj * dc[u][5]), pack_bf16(gj * dc[u][6], gj * dc[u][7]));
                }
                dot = warp_sum(dot);
                if (lane == 0) redk[w][j] = dot;
            }
        }
        __syncthreads();
        if (tid < k) {
            float sum = 0.f;
            for (int i = 0; i < (int)(blockDim.x >> 5); ++i) sum += redk[i][tid];
            dg[(long long)t * k + tid] = sum;
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < MAXCH; ++u) {
        const int ch = tid + u * 256;
        if (ch < nch)
#pragma unroll
            for (int v = 0; v < 8; ++v) dgamma_part[(long long)blockIdx.x * dl + 8 * ch + v] = dgp[u][v];
    }
}

__global__ void dgamma_reduce_kernel(const float *__restrict__ part, int nblk, int dl, float *dgamma,
                                     int accumulate) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= dl) return;
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += part[(long long)b * dl + i];
    dgamma[i] = s + (accumulate ? dgamma[i] : 0.f);
}

// dx_lat[t] = sum_j dxe[slot_pos[t, j]] (fp32 rows, added in slot order), stored bf16; 8 values
// per thread.
__global__ void slot_reduce_kernel(const float *__restrict__ dxe, const int32_t *__restrict__ slot_pos, int T,
                                   int dl, int k, bf16 *__restrict__ out) {
    const int per_row = dl / 8;
    const long long total = (long long)T * per_row;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / per_row), c = (int)(idx - (long long)t * per_row);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < k; ++j) {
            const float *src = dxe + (long long)slot_pos[(long long)t * k + j] * dl + 8 * c;
            const float4 v0 = *reinterpret_cast<const float4 *>(src);
            const float4 v1 = *reinterpret_cast<const float4 *>(src + 4);
            acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
            acc[4] += v1.x; acc[5] += v1.y; acc[6] += v1.z; acc[7] += v1.w;
        }
        *reinterpret_cast<uint4 *>(out + (long long)t * dl + 8 * c) =
            make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                       pack_bf16(acc[6], acc[7]));
    }
}

// Router backward of one token per block.  g_j = s_j / S over the chosen experts, so
// ds_j = (dg_j - sum_i g_i dg_i) / S; dlogit_j = ds_j s_j (1 - s_j).  The token's dx gains
// sum_j dlogit_j W_r[e_j] (fp32); dlogit is also written at the pair's expert-order position
// for the router's weight gradient.
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
    const int32_t *__restrict__ slot_pos, const float *__restrict__ dg, const float *__restrict__ W_r, int E,
    int d, int k, float *__restrict__ dx, float *__restrict__ dl_perm) {
    __shared__ float dl_s[32];
    __shared__ int e_s[32];
    const int t = blockIdx.x, tid = threadIdx.x;
    if (tid < 32) {
        const bool on = tid < k;
        const int e = on ? topk_idx[(long long)t * k + tid] : 0;
        const float s = on ? scores[(long long)t * E + e] : 0.f;
        const float g = on ? topk_w[(long long)t * k + tid] : 0.f;
        const float dgj = on ? dg[(long long)t * k + tid] : 0.f;
        const float S = warp_sum(s);
        const float gd = warp_sum(g * dgj);
        const float dl = on ? (dgj - gd) / S * s * (1.0f - s) : 0.f;
        dl_s[tid] = dl;
        e_s[tid] = e;
        if (on) dl_perm[slot_pos[(long long)t * k + tid]] = dl;
    }
    __syncthreads();
    float *row = dx + (long long)t * d;
    for (int i = 4 * tid; i < d; i += 4 * blockDim.x) {
        float4 acc = *reinterpret_cast<const float4 *>(row + i);
        for (int j = 0; j < k; ++j) {
            const float4 w = *reinterpret_cast<const float4 *>(W_r + (long long)e_s[j] * d + i);
            acc.x += dl_s[j] * w.x; acc.y += dl_s[j] * w.y; acc.z += dl_s[j] * w.z; acc.w += dl_s[j] * w.w;
        }
        *reinterpret_cast<float4 *>(row + i) = acc;
    }
}

// dW_r[e] (+)= sum over expert e's rows p (expert order) of dlogit(p) x[perm[p]]; grid
// (E, column blocks), four columns per thread, rows in order.
__global__ void __launch_bounds__(256) router_wgrad_kernel(const bf16 *__restrict__ x, const int32_t *__restrict__ perm,
                                                           const int32_t *__restrict__ offsets,
                                                           const float *__restrict__ dl_perm, int d, float *dW_r,
                                                           int accumulate) {
    const int e = blockIdx.x;
    const int i = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (i >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
        const float w = dl_perm[p];
        const uint2 v = *reinterpret_cast<const uint2 *>(x + (long long)perm[p] * d + i);
        const bf16 *b = reinterpret_cast<const bf16 *>(&v);
        acc.x += w * __bfloat162float(b[0]);
        acc.y += w * __bfloat162float(b[1]);
        acc.z += w * __bfloat162float(b[2]);
        acc.w += w * __bfloat162float(b[3]);
    }
    float *o = dW_r + (long long)e * d + i;
    if (accumulate) {
        const float4 p = *reinterpret_cast<const float4 *>(o);
        acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
    }
    *reinterpret_cast<float4 *>(o) = acc;
}

// ---------------------------------------------------------------- host side
// Expert e's gradient C_e [N][M] = (A_e^T B_e)^T over its rows: A [rows, M] (optionally gathered
// through a_index), B [rows, N] contiguous (b_rows in all).
int launch_wgrad(int E, int M, int N, const void *A, long long lda, const int32_t *a_index, const void *B,
                 long long ldb, long long b_rows, const int32_t *offsets, float *C, int accumulate, int *counter,
                 int32_t *status, cudaStream_t st) {
    WArgs a = {};
    a.A.p = static_cast<const bf16 *>(A); a.A.ld = lda; a.A.index = a_index;
    a.B.p = static_cast<const bf16 *>(B); a.B.ld = ldb; a.B.index = nullptr;
    a.M = M; a.N = N;
    a.tiles_m = (M + 127) / 128;
    a.tiles_n = (N + WG_BN - 1) / WG_BN;
    a.units = E * a.tiles_m * a.tiles_n;
    a.offsets = offsets;
    a.counter = counter;
    a.C = C; a.ldc = M; a.cstride = (long long)M * N;
    a.accumulate = accumulate;
    a.status = status;
    cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WG_SMEM);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "smem attribute: %s", cudaGetErrorString(e));
    if (a.units == 0) return SLMOE_OK;
    CUtensorMap bmap;   // B stored [b_rows, N] (MN-major), 64 x 64 boxes, 128-byte swizzle
    int rc = tmap_encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, b_rows, N, ldb, 64, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    CUtensorMap cmap;   // the gradients, [E * N, M] fp32, 32 x 16 boxes
    if ((rc = tmap_encode_2d(&cmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, (long long)E * N, M, M, 32, 16,
                             CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;
    const int sms = sm_count();
    wgrad_kernel<<<a.units < sms ? a.units : sms, WG_THREADS, WG_SMEM, st>>>(bmap, cmap, a);
    return check_launch("wgrad_kernel");
}

}  // namespace

// Bytes of backward workspace (see tc_backward for the regions).
size_t backward_workspace_bytes(const slmoe_config *c, BwdLayout *L) {
    const size_t T = c->T, d = c->d, dl = c->d_latent, E = c->E, k = c->k, I = c->I, Is = c->I_shared;
    const size_t Tk = T * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + (bytes ? bytes : 1) + 255) / 256 * 256;
        return at;
    };
    BwdLayout l = {};
    l.dy_b = take(T * d * 2);
    l.dz = take(T * dl * 4);
    l.dye = take(Tk * dl * 2);
    l.dg = take(Tk * 4);
    l.gu = take(Tk * 2 * I * 4);
    l.dgu = take(Tk * 2 * I * 2);
    l.dxe = take(Tk * dl * 4);
    l.dx_lat = take(T * dl * 2);
    l.gu_s = take(T * 2 * Is * 4);
    l.dgu_s = take(T * 2 * Is * 2);
    l.dl_perm = take(Tk * 4);
    l.nblk = (T + RB_TOK - 1) / RB_TOK;
    l.dgamma_part = take(l.nblk * dl * 4);
    l.counters = take(32 * 4);
    l.cap_dglu = (I + 127) / 128 * (E + (Tk + GROUPED_PASS - 1) / GROUPED_PASS);
    l.items_dglu = take(l.cap_dglu * 16);
    l.cap_dxe = (dl + 255) / 256 * (E + (Tk + GROUPED_PASS - 1) / GROUPED_PASS);
    l.items_dxe = take(l.cap_dxe * 16);
    l.total = off;
    if (L) *L = l;
    return off;
}

int tc_backward(const slmoe_config *c, const void *x, const slmoe_weights *w, const float *dy, float *dx,
                const slmoe_grads *g, int accumulate, const FwdSaved &fs, char *ws, int32_t *status,
                cudaStream_t st) {
    const int T = c->T, d = c->d, dl = c->d_latent, E = c->E, k = c->k, I = c->I;
    const int ns = c->n_shared, Is = c->I_shared;
    const long long Tk = (long long)T * k;
    BwdLayout L;
    backward_workspace_bytes(c, &L);
    bf16 *dy_b = reinterpret_cast<bf16 *>(ws + L.dy_b);
    float *dz = reinterpret_cast<float *>(ws + L.dz);
    bf16 *dye = reinterpret_cast<bf16 *>(ws + L.dye);
    float *dg = reinterpret_cast<float *>(ws + L.dg);
    float *gu = reinterpret_cast<float *>(ws + L.gu);
    bf16 *dgu = reinterpret_cast<bf16 *>(ws + L.dgu);
    float *dxe = reinterpret_cast<float *>(ws + L.dxe);
    bf16 *dx_lat = reinterpret_cast<bf16 *>(ws + L.dx_lat);
    float *gu_s = reinterpret_cast<float *>(ws + L.gu_s);
    bf16 *dgu_s = reinterpret_cast<bf16 *>(ws + L.dgu_s);
    float *dl_perm = reinterpret_cast<float *>(ws + L.dl_perm);
    float *dgamma_part = reinterpret_cast<float *>(ws + L.dgamma_part);
    int *cnt = reinterpret_cast<int *>(ws + L.counters);
    int rc;
    if (cudaMemsetAsync(cnt, 0, 32 * sizeof(int), st) != cudaSuccess ||
        cudaMemsetAsync(dx, 0, (size_t)T * d * sizeof(float), st) != cudaSuccess)
        return check_launch("memset");
    const int sms = sm_count();

    // dy in bf16 for the tensor cores
    {
        const long long n = (long long)T * d;
        const long long blocks = (n / 4 + 255) / 256 < 8LL * sms ? (n / 4 + 255) / 256 : 8LL * sms;
        f32_to_bf16_kernel<<<(int)(blocks > 0 ? blocks : 1), 256, 0, st>>>(dy, dy_b, n);
        if ((rc = check_launch("f32_to_bf16"))) return rc;
    }
    auto opnd = [](const void *p, long long pitch) { TcOperand o; o.p = p; o.pitch = pitch; return o; };
    // up-projection: dz = dy W_out (fp32; W_out stored [d, d_l] is MN-major here),
    // dW_out (+)= dy^T z (both operands MN-major)
    if ((rc = tc_dense_gemm(B_MN_, T, dl, d, opnd(dy_b, d), opnd(w->W_out, dl), dz, dl, 0, nullptr, status, cnt + 0,
                            st)))
        return rc;
    if ((rc = tc_dense_gemm(A_MN_ | B_MN_, d, dl, T, opnd(dy_b, d), opnd(fs.z, dl), g->dW_out, dl, accumulate, nullptr,
                            status, cnt + 1, st)))
        return rc;
    // shared experts
    for (int s = 0; s < ns; ++s) {
        const bf16 *W13s = static_cast<const bf16 *>(w->W13_s) + (size_t)s * 2 * Is * d;
        const bf16 *W2s = static_cast<const bf16 *>(w->W2_s) + (size_t)s * d * Is;
        int *cs = cnt + 2 + 5 * s;
        // pre-activations gu_s = x W13_s^T (recomputed, fp32)
        if ((rc = tc_dense_gemm(0, T, 2 * Is, d, opnd(x, d), opnd(W13s, d), gu_s, 2 * Is, 0, nullptr, status, cs + 0,
                                st)))
            return rc;
        // dh_s = dy W2_s (W2_s stored [d, I_s]), turned into [dg | du] by the SiTU-GLU derivative
        TcDglu dgl;
        dgl.gu = gu_s; dgl.ld_gu = 2 * Is; dgl.F = Is; dgl.dgu = dgu_s; dgl.ld_dgu = 2 * Is;
        dgl.beta1 = c->beta1; dgl.beta2 = c->beta2;
        if ((rc = tc_dense_gemm(B_MN_, T, Is, d, opnd(dy_b, d), opnd(W2s, Is), nullptr, 0, 0, &dgl, status, cs + 1, st)))
            return rc;
        // dW2_s (+)= dy^T h_s  (h_s from the forward)
        if ((rc = tc_dense_gemm(A_MN_ | B_MN_, d, Is, T, opnd(dy_b, d), opnd(fs.h_s + (size_t)s * Is, (long long)ns * Is),
                                g->dW2_s + (size_t)s * d * Is, Is, accumulate, nullptr, status, cs + 2, st)))
            return rc;
        // dx += [dg | du] W13_s  (W13_s stored [2 I_s, d]);  dW13_s (+)= [dg | du]^T x
        if ((rc = tc_dense_gemm(B_MN_, T, d, 2 * Is, opnd(dgu_s, 2 * Is), opnd(W13s, d), dx, d, 1, nullptr, status,
                                cs + 3, st)))
            return rc;
        if ((rc = tc_dense_gemm(A_MN_ | B_MN_, 2 * Is, d, T, opnd(dgu_s, 2 * Is), opnd(x, d),
                                g->dW13_s + (size_t)s * 2 * Is * d, d, accumulate, nullptr, status, cs + 4, st)))
            return rc;
    }
    // RMSNorm + combine backward
    {
        // 8-feature chunks per thread: as few as d_latent needs (registers bound the blocks per SM)
        const int nch = (dl / 8 + 255) / 256;
        auto kern = nch <= 1 ? rms_combine_bwd_kernel<1> : nch <= 2 ? rms_combine_bwd_kernel<2> : rms_combine_bwd_kernel<RB_MAXCH>;
        kern<<<(int)L.nblk, 256, 0, st>>>(fs.y_e, fs.topk_w, fs.slot_pos, w->gamma, dz, T, dl, k, c->eps, dye, dg,
                                          dgamma_part);
        if ((rc = check_launch("rms_combine_bwd"))) return rc;
        dgamma_reduce_kernel<<<(dl + 255) / 256, 256, 0, st>>>(dgamma_part, (int)L.nblk, dl, g->dgamma, accumulate);
        if ((rc = check_launch("dgamma_reduce"))) return rc;
    }
    // routed experts on the forward's grouped kernel: pre-activations (the forward's gate|up
    // list), dh -> [dg | du] (a list of 128-feature blocks of I, alternating between two
    // accumulator sets), x_lat rows (256-feature blocks of d_latent)
    // (a single-list build writes its count and a zero after it: counters 28-29 and 30-31)
    int4 *items_dglu = reinterpret_cast<int4 *>(ws + L.items_dglu);
    int4 *items_dxe = reinterpret_cast<int4 *>(ws + L.items_dxe);
    if ((rc = tc_worklist_single(fs.counts, fs.offsets, E, (I + 127) / 128, items_dglu, cnt + 28, (int)L.cap_dglu, st)))
        return rc;
    if ((rc = tc_worklist_single(fs.counts, fs.offsets, E, (dl + 255) / 256, items_dxe, cnt + 30, (int)L.cap_dxe, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_GU32, c, w->W13, fs.x_lat, fs.perm, fs.items1, fs.n_items, cnt + 17, gu, nullptr,
                             nullptr, status, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_DGLU, c, w->W2, dye, nullptr, items_dglu, cnt + 28, cnt + 18, nullptr, gu, dgu,
                             status, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_DXE, c, w->W13, dgu, nullptr, items_dxe, cnt + 30, cnt + 19, dxe, nullptr,
                             nullptr, status, st)))
        return rc;
    // routed weight gradients, K = the expert's rows, computed transposed so that each lane
    // (an M index) stores along a row of the gradient:
    //   dW2[e]^T  [I, d_l]  = h^T dy_e             (A = h, B = dy_e by TMA)
    //   dW13[e]^T [d_l, 2I] = x_lat[perm]^T [dg|du] (A = x_lat gathered, B = [dg|du] by TMA)
    if ((rc = launch_wgrad(E, I, dl, fs.h, I, nullptr, dye, dl, Tk, fs.offsets, g->dW2, accumulate, cnt + 23,
                           status, st)))
        return rc;
    if ((rc = launch_wgrad(E, dl, 2 * I, fs.x_lat, dl, fs.perm, dgu, 2 * I, Tk, fs.offsets, g->dW13, accumulate,
                           cnt + 24, status, st)))
        return rc;
    // dx_lat = sum over the token's k rows; then the latent down-projection
    {
        const long long n = (long long)T * (dl / 8);
        const long long blocks = (n + 255) / 256 < 8LL * sms ? (n + 255) / 256 : 8LL * sms;
        slot_reduce_kernel<<<(int)(blocks > 0 ? blocks : 1), 256, 0, st>>>(dxe, fs.slot_pos, T, dl, k, dx_lat);
        if ((rc = check_launch("slot_reduce"))) return rc;
    }
    if ((rc = tc_dense_gemm(B_MN_, T, d, dl, opnd(dx_lat, dl), opnd(w->W_in, d), dx, d, 1, nullptr, status, cnt + 25,
                            st)))
        return rc;
    if ((rc = tc_dense_gemm(A_MN_ | B_MN_, dl, d, T, opnd(dx_lat, dl), opnd(x, d), g->dW_in, d, accumulate, nullptr,
                            status, cnt + 26, st)))
        return rc;
    // router
    router_bwd_kernel<<<T, 256, 0, st>>>(fs.scores, fs.topk_idx, fs.topk_w, fs.slot_pos, dg, w->W_r, E, d, k, dx,
                                         dl_perm);
    if ((rc = check_launch("router_bwd"))) return rc;
    router_wgrad_kernel<<<dim3(E, (d / 4 + 255) / 256), 256, 0, st>>>(static_cast<const bf16 *>(x), fs.perm,
                                                                    fs.offsets, dl_perm, d, g->dW_r, accumulate);
    if ((rc = check_launch("router_wgrad"))) return rc;
    (void)Tk;
    return SLMOE_OK;
}

}  // namespace slmoe
