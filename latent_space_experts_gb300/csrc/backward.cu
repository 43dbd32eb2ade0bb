// Backward pass of the Stable LatentMoE layer, bf16 layer type (sm_103a).
//
// The gradient is the chain rule of the forward (K3 architecture write-up, SiTU激活优化 /
// 归一化策略调整; the concept note's 训练基础设施 trains this layer), run against the
// intermediates a forward call leaves in its workspace.  Every contraction goes through one
// tcgen05 kernel, bgemm_kernel:
//
//  * a tile is 128 rows (the MMA's M) x up to 256 columns (N), K in blocks of 64;
//  * four loader warps fill a 4-stage ring with cp.async (16-byte chunks, zero-filled past
//    the edges), writing each operand either K-major (a row of 64 K values per 128-byte line)
//    or MN-major (a line of 64 M or N values per K row), both in the 128-byte swizzle, so
//    dgrad and wgrad read W and the activations as they are stored, without transposes;
//  * one thread issues tcgen05.mma (M = 128, K = 16) into a double-buffered TMEM
//    accumulator; four epilogue warps drain it while the next tile accumulates;
//  * work comes from a global counter in three modes: dense tiles (banded for L2 reuse),
//    per-expert token passes from a device-built list (the routed experts' dgrad, with the
//    weights as M: "swap AB"), and per-expert weight-gradient tiles whose K is the expert's
//    own segment of rows in expert-sorted order;
//  * epilogues: fp32 store or accumulate (optionally transposed), bf16 store, and the
//    SiTU-GLU derivative, which turns dh into [dg | du] using the recomputed pre-activations
//    (kept in fp32: near saturation the derivatives of SiTU and of the soft cap change by a
//    few per cent across one bf16 step of their argument).
//
// The memory-bound steps are plain kernels: RMSNorm + combine backward (dc, the gradient of
// each expert output, of each gate weight, and per-block dgamma sums), the per-token sum of
// the k expert-row gradients of x_lat, and the router (gate renormalisation, sigmoid, the
// router's share of dx and dW_r).  Every reduction runs in a fixed order, so results do not
// depend on scheduling.
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

constexpr int BG_BN = 256;
constexpr int BG_STAGES = 4;
constexpr int BG_A_BYTES = 128 * 128;              // 128 M x 64 K
constexpr int BG_B_BYTES = BG_BN * 128;            // 256 N x 64 K
constexpr int BG_STAGE = BG_A_BYTES + BG_B_BYTES;
constexpr int BG_LOADERS = 128;                    // warps 0-3
constexpr int BG_MMA_WARP = 4;
constexpr int BG_EPI_WARP0 = 5;                    // warps 5-8
constexpr int BG_THREADS = 9 * 32;
constexpr int BG_Q = 4;
constexpr int BG_STG_LD = 65;                      // fp32 staging row of 64 columns (+1 against bank conflicts)
constexpr int BG_STG = 4 * 32 * BG_STG_LD * 4;     // one 32 x 64 staging tile per epilogue warp
constexpr int BG_SMEM = BG_STAGES * BG_STAGE + BG_STG + 1024 + 512;
constexpr int BG_BAND = 8;                         // row tiles per band of the dense tile order

enum { BG_DENSE = 0, BG_PASS = 1, BG_WGRAD = 2 };
constexpr int A_MN_ = 1, B_MN_ = 2;   // tc_dense_gemm operand majorness
enum { BE_F32 = 0, BE_BF16 = 1, BE_DGLU = 2 };

// One operand as stored: lines of ld elements; a grouped operand's expert e starts estride
// elements further on; index (nullable) maps a line number to the stored line.
struct BOp {
    const bf16 *p;
    long long ld;
    long long estride;
    const int32_t *index;
};

struct BArgs {
    BOp A, B;
    int M, N, K;             // dense: the GEMM; pass: M features per expert, K; wgrad: M x N per expert
    int tiles_m, tiles_n;    // 128 x 256 tiles of M x N (dense, wgrad)
    int units;               // dense: tiles; wgrad: E * tiles; pass: list capacity
    const int4 *items;       // pass: {expert, M block, first row in expert order, rows}
    const int *n_items;      // pass: number of items (device)
    const int32_t *offsets;  // wgrad: per-expert row segments [E + 1]
    int *counter;            // zeroed work counter
    void *C;                 // output (fp32 or bf16); wgrad: expert e at C + e * cstride
    long long ldc, cstride;
    int out_t;               // 1: C[n][m] instead of C[m][n]
    int accumulate;          // fp32 epilogue: add into C instead of storing
    const float *gu;         // SiTU-GLU derivative: fp32 pre-activations [rows, 2F] (gate | up)
    long long ld_gu;
    int F;
    bf16 *dgu;               // ... and its output [rows, 2F]
    long long ld_dgu;
    float beta1, beta2;
    int32_t *status;
    unsigned long long wait_limit_ns;
};

struct BItem {
    int e, m0, n0, mv, nv, kr0, klen;   // e < 0: end of work
};

__device__ __forceinline__ void band_tile(int tile, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_band = BG_BAND * tiles_n;
    const int band = tile / per_band;
    const int m_first = band * BG_BAND;
    const int bm = min(BG_BAND, tiles_m - m_first);
    const int r = tile - band * per_band;
    tm = m_first + r % bm;
    tn = r / bm;
}

template <int MODE>
__device__ __forceinline__ BItem fetch_item(const BArgs &a) {
    BItem it;
    it.e = -1;
    const int u = atomicAdd(a.counter, 1);
    if (MODE == BG_PASS) {
        if (u >= *a.n_items || u >= a.units) return it;
        const int4 v = a.items[u];
        it.e = v.x;
        it.m0 = v.y * 128;
        it.mv = min(128, a.M - it.m0);
        it.n0 = v.z;
        it.nv = v.w;
        it.kr0 = 0;
        it.klen = a.K;
        return it;
    }
    if (u >= a.units) return it;
    const int per = a.tiles_m * a.tiles_n;
    int tm, tn;
    if (MODE == BG_DENSE) {
        band_tile(u, a.tiles_m, a.tiles_n, tm, tn);
        it.e = 0;
        it.kr0 = 0;
        it.klen = a.K;
    } else {
        it.e = u / per;
        band_tile(u - it.e * per, a.tiles_m, a.tiles_n, tm, tn);
        it.kr0 = a.offsets[it.e];
        it.klen = a.offsets[it.e + 1] - it.kr0;
    }
    it.m0 = tm * 128;
    it.n0 = tn * BG_BN;
    it.mv = min(128, a.M - it.m0);
    it.nv = min(BG_BN, a.N - it.n0);
    return it;
}

// Copies of one operand tile (extent x 64 K) for one stage.  t = loader thread 0..127.
//  K-major: line r = row r of the tile (M or N index), chunk c = K values 8c..8c+7.
//  MN-major: line (g, kr) = K row kr of the 64-wide group g, chunk c = values 64g+8c..+7.
template <bool MN, int EXTENT>
__device__ __forceinline__ void load_tile(uint32_t sbase, const BOp &op, int e, int mn0, int mnv, int kr0,
                                          int k0, int klen, int t) {
    constexpr int CHUNKS = EXTENT * 8;                  // 16-byte chunks of the tile
    const bf16 *base = op.p + (long long)e * op.estride;
#pragma unroll 4
    for (int q = t; q < CHUNKS; q += BG_LOADERS) {
        int line, c;
        long long src_line;
        bool ok;
        uint32_t dst;
        long long col;
        if (!MN) {
            line = q >> 3;
            c = q & 7;
            ok = line < mnv && k0 + 8 * c < klen;
            const int row = mn0 + (line < mnv ? line : 0);
            src_line = op.index ? op.index[row] : row;
            col = k0 + 8 * c;
            dst = sbase + (line >> 3) * 1024 + (line & 7) * 128 + ((c ^ (line & 7)) << 4);
        } else {
            // 64 K rows x (EXTENT / 64) groups x 8 chunks; consecutive threads walk one K row
            const int per_row = EXTENT / 8;              // chunks per K row
            const int kr = q / per_row;
            const int w = q - kr * per_row;
            const int g = w >> 3;
            c = w & 7;
            ok = k0 + kr < klen && 64 * g + 8 * c < mnv;
            const int krow = kr0 + k0 + (k0 + kr < klen ? kr : 0);
            src_line = op.index ? op.index[krow] : krow;
            col = mn0 + 64 * g + 8 * c;
            dst = sbase + g * 8192 + (kr >> 3) * 1024 + (kr & 7) * 128 + ((c ^ (kr & 7)) << 4);
            if (!ok) col = mn0;
        }
        const bf16 *src = base + src_line * op.ld + (ok ? col : 0);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16u : 0u)
                     : "memory");
    }
}

__device__ __forceinline__ float situ_f(float g, float b1) {
    return b1 * tanhf(g / b1) * (1.0f / (1.0f + expf(-g)));
}
__device__ __forceinline__ float situ_grad_f(float g, float b1) {
    const float th = tanhf(g / b1);
    const float sg = 1.0f / (1.0f + expf(-g));
    return (1.0f - th * th) * sg + b1 * th * sg * (1.0f - sg);
}

// B_TMA: the B operand (MN-major, stored rows in expert order) comes by TMA in 64 x 64 boxes
// from bmap; rows past the expert's segment then hold other experts' values, which meet the
// zero-filled rows of A past the segment, so they add nothing.
template <int EPI, bool A_MN, bool B_MN, int MODE, bool B_TMA = false>
__global__ void __launch_bounds__(BG_THREADS, 1) bgemm_kernel(const __grid_constant__ CUtensorMap bmap,
                                                              const BArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *stg_all = reinterpret_cast<float *>(smem + BG_STAGES * BG_STAGE);
    BItem *q_items = reinterpret_cast<BItem *>(smem + BG_STAGES * BG_STAGE + BG_STG);
    uint64_t *q_full = reinterpret_cast<uint64_t *>(q_items + BG_Q);
    uint64_t *q_empty = q_full + BG_Q;
    uint64_t *full = q_empty + BG_Q;
    uint64_t *empty = full + BG_STAGES;
    uint64_t *tfull = empty + BG_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_drain + 1);
    volatile WaitCtl *wc = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < BG_Q; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 4 + 1 + 4);   // loader warps, MMA thread, epilogue warps
        }
        for (int s = 0; s < BG_STAGES; ++s) {
            mbar_init(&full[s], BG_LOADERS + (B_TMA ? 1 : 0));
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(mma_drain, 1);
        wait_ctl_init(wc, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == BG_MMA_WARP) tmem_alloc(tmem_slot, 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;

    auto pop = [&](int &qs, uint32_t &qp, BItem &it, bool warp_wide) -> bool {
        if (!mbar_wait(&q_full[qs], qp, wc)) return false;
        it = q_items[qs];
        if (warp_wide) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qs]);
        } else {
            mbar_arrive(&q_empty[qs]);
        }
        if (++qs == BG_Q) { qs = 0; qp ^= 1; }
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
                    const BItem nx = fetch_item<MODE>(a);
                    if (mbar_wait(&q_empty[fs], fp ^ 1, wc)) {
                        q_items[fs] = nx;
                        mbar_arrive(&q_full[fs]);
                    } else {
                        ok = 0;
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (++fs == BG_Q) { fs = 0; fp ^= 1; }
            }
            BItem it;
            if (!pop(qs, qp, it, true)) break;
            if (it.e < 0) break;
            const int nkb = (it.klen + 63) / 64;
            bool aborted = false;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1, wc)) { aborted = true; break; }
                const uint32_t sa = su32(smem + stage * BG_STAGE);
                const uint32_t sb = sa + BG_A_BYTES;
                load_tile<A_MN, 128>(sa, a.A, it.e, it.m0, it.mv, it.kr0, kb * 64, it.klen, t);
                if (B_TMA) {
                    if (t == 0) {
                        mbar_expect_tx(&full[stage], BG_B_BYTES);
#pragma unroll
                        for (int g = 0; g < BG_BN / 64; ++g)
                            tma_load_2d(sb + g * 8192, &bmap, &full[stage], it.n0 + 64 * g, it.kr0 + kb * 64);
                    }
                } else {
                    load_tile<B_MN, BG_BN>(sb, a.B, it.e, it.n0, it.nv, it.kr0, kb * 64, it.klen, t);
                }
                cp_async_arrive_noinc(&full[stage]);
                if (++stage == BG_STAGES) { stage = 0; phase ^= 1; l_wrapped = true; }
            }
            if (aborted) break;
        }
        cp_async_wait_all();
    } else if (warp == BG_MMA_WARP) {
        if (lane == 0) {
            int qs = 0, stage = 0, buf = 0;
            uint32_t qp = 0, phase = 0, tph = 0;
            for (;;) {
                BItem it;
                if (!pop(qs, qp, it, false)) break;
                if (it.e < 0) break;
                const int nkb = (it.klen + 63) / 64;
                if (nkb == 0) continue;                    // nothing to accumulate (empty expert)
                const int n16 = (MODE == BG_PASS ? it.nv : BG_BN) + 15 & ~15;
                const uint32_t idesc = idesc_bf16(128, n16) | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
                if (!mbar_wait(&tempty[buf], tph ^ 1, wc)) break;
                tc_after();
                const uint32_t d = tmem_base + buf * 256;
                bool aborted = false;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, wc)) { aborted = true; break; }
                    fence_proxy_async();
                    tc_after();
                    const uint32_t sa = su32(smem + stage * BG_STAGE);
                    const uint32_t sb = sa + BG_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = A_MN ? mn_desc(sa + kk * 2048, 8192) : sdesc(sa + kk * 32);
                        const uint64_t bd = B_MN ? mn_desc(sb + kk * 2048, 8192) : sdesc(sb + kk * 32);
                        umma(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == BG_STAGES) { stage = 0; phase ^= 1; }
                }
                if (aborted) break;
                umma_commit(&tfull[buf]);
                if (++buf == 2) { buf = 0; tph ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue: warp w drains TMEM lanes
        // 32 (w % 4) .. + 31, i.e. tile rows (M) of that quadrant
        const int q = warp & 3;
        const int i = q * 32 + lane;
        int qs = 0, buf = 0;
        uint32_t qp = 0, tph = 0;
        for (;;) {
            BItem it;
            if (!pop(qs, qp, it, true)) break;
            if (it.e < 0) break;
            const int nkb = (it.klen + 63) / 64;
            const bool row_ok = i < it.mv;
            const int m = it.m0 + i;
            if (nkb == 0) {
                // an expert without rows: its weight-gradient tile is zero (stored unless adding)
                if (EPI == BE_F32 && !a.accumulate && row_ok) {
                    float *C = static_cast<float *>(a.C) + (long long)it.e * a.cstride;
                    for (int j = 0; j < it.nv; ++j)
                        C[a.out_t ? (long long)(it.n0 + j) * a.ldc + m : (long long)m * a.ldc + it.n0 + j] = 0.f;
                }
                continue;
            }
            if (!mbar_wait(&tfull[buf], tph, wc)) break;
            tc_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + buf * 256;
            if (EPI == BE_F32 && !a.out_t) {
                // 64 columns at a time through a 32 x 64 staging tile: each lane writes its row,
                // then the warp stores one row at a time as two 128-byte runs (coalesced)
                float *stg = stg_all + (warp - BG_EPI_WARP0) * 32 * BG_STG_LD;
                float *C = static_cast<float *>(a.C) + (long long)it.e * (MODE == BG_WGRAD ? a.cstride : 0);
                for (int c0 = 0; c0 < it.nv; c0 += 64) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) TMEM_LD16(tb + c0 + 16 * u, r[u]);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int j = 0; j < 16; ++j) stg[lane * BG_STG_LD + 16 * u + j] = __uint_as_float(r[u][j]);
                    __syncwarp();
                    // eight rows at a time: all staging reads (and, when adding, all reads of C)
                    // issued before the stores, so the latencies overlap
                    const bool c_ok[2] = {c0 + lane < it.nv, c0 + lane + 32 < it.nv};
#pragma unroll 1
                    for (int rr0 = 0; rr0 < 32; rr0 += 8) {
                        float v[8][2];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int h = 0; h < 2; ++h) v[i][h] = stg[(rr0 + i) * BG_STG_LD + lane + 32 * h];
                        if (a.accumulate) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int mi = q * 32 + rr0 + i;
                                const float *row = C + (long long)(it.m0 + mi) * a.ldc + it.n0 + c0;
#pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    if (mi < it.mv && c_ok[h]) v[i][h] += row[lane + 32 * h];
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int mi = q * 32 + rr0 + i;
                            float *row = C + (long long)(it.m0 + mi) * a.ldc + it.n0 + c0;
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                if (mi < it.mv && c_ok[h]) row[lane + 32 * h] = v[i][h];
                        }
                    }
                    __syncwarp();
                }
            } else
            for (int c = 0; c < it.nv; c += 16) {
                uint32_t r[16];
                TMEM_LD16(tb + c, r);
                tmem_wait_ld();
                if (!row_ok) continue;
                const int nj = min(16, it.nv - c);
                if (EPI == BE_F32) {
                    float *C = static_cast<float *>(a.C) + (long long)it.e * (MODE == BG_WGRAD ? a.cstride : 0);
                    if (!a.out_t) {
                        float *row = C + (long long)m * a.ldc + it.n0 + c;
                        if (nj == 16 && (a.ldc & 3) == 0) {
#pragma unroll
                            for (int v = 0; v < 16; v += 4) {
                                float4 o = make_float4(__uint_as_float(r[v]), __uint_as_float(r[v + 1]),
                                                       __uint_as_float(r[v + 2]), __uint_as_float(r[v + 3]));
                                if (a.accumulate) {
                                    const float4 p = *reinterpret_cast<const float4 *>(row + v);
                                    o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
                                }
                                *reinterpret_cast<float4 *>(row + v) = o;
                            }
                        } else {
                            for (int j = 0; j < nj; ++j)
                                row[j] = __uint_as_float(r[j]) + (a.accumulate ? row[j] : 0.f);
                        }
                    } else {   // lanes are consecutive m: every store is one 128-byte run
                        float *o = C + (long long)(it.n0 + c) * a.ldc + m;
                        float v[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
                        if (a.accumulate) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < nj) v[j] += o[(long long)j * a.ldc];
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < nj) o[(long long)j * a.ldc] = v[j];
                    }
                } else if (EPI == BE_BF16) {
                    bf16 *C = static_cast<bf16 *>(a.C);
                    if (!a.out_t) {
                        bf16 *row = C + (long long)m * a.ldc + it.n0 + c;
                        for (int j = 0; j < nj; ++j) row[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
                    } else {
                        for (int j = 0; j < nj; ++j)
                            C[(long long)(it.n0 + c + j) * a.ldc + m] = __float2bfloat16_rn(__uint_as_float(r[j]));
                    }
                } else {   // BE_DGLU: the accumulator is dh; rows x features by orientation
                    for (int j = 0; j < nj; ++j) {
                        const long long row = a.out_t ? (long long)(it.n0 + c + j) : (long long)m;
                        const int f = a.out_t ? m : it.n0 + c + j;
                        const float dh = __uint_as_float(r[j]);
                        const float g = a.gu[row * a.ld_gu + f];
                        const float u = a.gu[row * a.ld_gu + a.F + f];
                        const float tu = tanhf(u / a.beta2);
                        const float cap = a.beta2 * tu;
                        a.dgu[row * a.ld_dgu + f] = __float2bfloat16_rn(dh * cap * situ_grad_f(g, a.beta1));
                        a.dgu[row * a.ld_dgu + a.F + f] =
                            __float2bfloat16_rn(dh * situ_f(g, a.beta1) * (1.0f - tu * tu));
                    }
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            if (++buf == 2) { buf = 0; tph ^= 1; }
        }
    }
    __syncthreads();
    if (wc->abort) {   // let copies and MMAs in flight finish before TMEM is freed
        if (B_TMA && threadIdx.x == 0) drain_ring(full, BG_STAGES, l_stage, l_phase, l_wrapped);
        if (warp == BG_MMA_WARP && lane == 0) {
            umma_commit(mma_drain);
            mbar_wait_drain(mma_drain, 0);
        }
        __syncthreads();
    }
    if (warp == BG_MMA_WARP) {
        tc_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && wc->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// Token passes of at most cap rows per expert (balanced), times nmb M blocks: the work list of
// a grouped dgrad GEMM, built on the device from the expert counts and offsets.
__global__ void __launch_bounds__(1024) pass_list_kernel(const int32_t *__restrict__ counts,
                                                         const int32_t *__restrict__ offsets, int E, int nmb,
                                                         int cap, int4 *__restrict__ items, int *n_items,
                                                         int max_items) {
    __shared__ int base_s[4096 + 1];
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = tid * per;
    int loc = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) loc += nmb * ((counts[e] + cap - 1) / cap);
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int base = incl - loc;
    for (int i = 0; i < w; ++i) base += wsum[i];
    for (int e = e0; e < e0 + per && e < E; ++e) {
        base_s[e] = base;
        base += nmb * ((counts[e] + cap - 1) / cap);
    }
    if (tid == blockDim.x - 1) *n_items = min(base, max_items);
    __syncthreads();
    for (int e = w; e < E; e += blockDim.x >> 5) {
        const int n = counts[e], off = offsets[e];
        const int np = (n + cap - 1) / cap;
        if (np == 0) continue;
        const int chunk = (n + np - 1) / np;
        for (int j = lane; j < nmb * np; j += 32) {
            const int mb = j / np, pass = j - mb * np;
            const int c0 = pass * chunk;
            if (base_s[e] + j < max_items)
                items[base_s[e] + j] = make_int4(e, mb, off + c0, min(chunk, n - c0));
        }
    }
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
constexpr int RB_TOK = 16;
constexpr int RB_MAXCH = 4;          // 8-feature chunks per thread: d_latent <= 8 * 256 * 4
__global__ void __launch_bounds__(256) rms_combine_bwd_kernel(
    const bf16 *__restrict__ y_e, const float *__restrict__ topk_w, const int32_t *__restrict__ slot_pos,
    const float *__restrict__ gamma, const float *__restrict__ dz, int T, int dl, int k, float eps,
    bf16 *__restrict__ dye, float *__restrict__ dg, float *__restrict__ dgamma_part) {
    __shared__ float red[64];
    __shared__ float redk[8][32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nch = dl / 8;
    float dgp[RB_MAXCH][8];
#pragma unroll
    for (int u = 0; u < RB_MAXCH; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) dgp[u][v] = 0.f;
    const int t0 = blockIdx.x * RB_TOK;
    for (int t = t0; t < min(T, t0 + RB_TOK); ++t) {
        const int32_t *sp = slot_pos + (long long)t * k;
        const float *gw = topk_w + (long long)t * k;
        const float *dzt = dz + (long long)t * dl;
        float cv[RB_MAXCH][8];
        float ss = 0.f, A = 0.f;
#pragma unroll
        for (int u = 0; u < RB_MAXCH; ++u) {
            const int ch = tid + u * 256;
#pragma unroll
            for (int v = 0; v < 8; ++v) cv[u][v] = 0.f;
            if (ch < nch) {
                for (int j = 0; j < k; ++j) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(y_e + (long long)sp[j] * dl + 8 * ch);
                    const bf16 *b = reinterpret_cast<const bf16 *>(&q);
#pragma unroll
                    for (int v = 0; v < 8; ++v) cv[u][v] += gw[j] * __bfloat162float(b[v]);
                }
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
        float dgl[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) dgl[j] = 0.f;
#pragma unroll
        for (int u = 0; u < RB_MAXCH; ++u) {
            const int ch = tid + u * 256;
            if (ch >= nch) continue;
            float dc[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float dzv = dzt[8 * ch + v];
                dc[v] = gamma[8 * ch + v] * dzv * ir - cv[u][v] * coef;
                dgp[u][v] += dzv * cv[u][v] * ir;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < k) {
                    const long long rw = (long long)sp[j] * dl + 8 * ch;
                    const uint4 q = *reinterpret_cast<const uint4 *>(y_e + rw);
                    const bf16 *b = reinterpret_cast<const bf16 *>(&q);
                    float dot = 0.f;
#pragma unroll
                    for (int v = 0; v < 8; ++v) dot += dc[v] * __bfloat162float(b[v]);
                    dgl[j] += dot;
                    const float gj = gw[j];
                    *reinterpret_cast<uint4 *>(dye + rw) =
                        make_uint4(pack_bf16(gj * dc[0], gj * dc[1]), pack_bf16(gj * dc[2], gj * dc[3]),
                                   pack_bf16(gj * dc[4], gj * dc[5]), pack_bf16(gj * dc[6], gj * dc[7]));
                }
            }
        }
        // all k gate-weight sums at once: warp sums, then one thread per slot over the warps
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < k) {
                const float v = warp_sum(dgl[j]);
                if (lane == 0) redk[w][j] = v;
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
    for (int u = 0; u < RB_MAXCH; ++u) {
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
template <int EPI, bool AMN, bool BMN, int MODE, bool B_TMA = false>
int launch_bg(BArgs a, cudaStream_t st, long long b_rows = 0) {
    auto kern = bgemm_kernel<EPI, AMN, BMN, MODE, B_TMA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BG_SMEM);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "smem attribute: %s", cudaGetErrorString(e));
    if (MODE != BG_PASS && a.units == 0) return SLMOE_OK;
    CUtensorMap bmap;
    memset(&bmap, 0, sizeof(bmap));
    if (B_TMA) {   // B stored [b_rows, N] (MN-major), 64 x 64 boxes, 128-byte swizzle
        int rc = tmap_encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.B.p, b_rows, a.N, a.B.ld, 64, 64,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
    }
    const int sms = sm_count();
    const int grid = (MODE != BG_PASS && a.units < sms) ? a.units : sms;
    kern<<<grid, BG_THREADS, BG_SMEM, st>>>(bmap, a);
    return check_launch("bgemm_kernel");
}

BArgs dense_args(int M, int N, int K, BOp A, BOp B, void *C, long long ldc, int accumulate, int *counter,
                 int32_t *status) {
    BArgs a = {};
    a.A = A;
    a.B = B;
    a.M = M;
    a.N = N;
    a.K = K;
    a.tiles_m = (M + 127) / 128;
    a.tiles_n = (N + BG_BN - 1) / BG_BN;
    a.units = a.tiles_m * a.tiles_n;
    a.C = C;
    a.ldc = ldc;
    a.accumulate = accumulate;
    a.counter = counter;
    a.status = status;
    return a;
}

BOp op(const void *p, long long ld, long long estride = 0, const int32_t *index = nullptr) {
    BOp o;
    o.p = static_cast<const bf16 *>(p);
    o.ld = ld;
    o.estride = estride;
    o.index = index;
    return o;
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
    const size_t cap1 = (2 * I + 127) / 128 * (E + (Tk + BG_BN - 1) / BG_BN);
    const size_t cap2 = (I + 127) / 128 * (E + (Tk + BG_BN - 1) / BG_BN);
    const size_t cap3 = (dl + 127) / 128 * (E + (Tk + BG_BN - 1) / BG_BN);
    l.cap1 = cap1;
    l.cap2 = cap2;
    l.cap3 = cap3;
    l.items1 = take(cap1 * 16);
    l.items2 = take(cap2 * 16);
    l.items3 = take(cap3 * 16);
    l.cap_dglu = (I + 255) / 256 * (E + (Tk + GROUPED_PASS - 1) / GROUPED_PASS);
    l.items_dglu = take(l.cap_dglu * 16);
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
    int4 *items1 = reinterpret_cast<int4 *>(ws + L.items1);
    int4 *items2 = reinterpret_cast<int4 *>(ws + L.items2);
    int4 *items3 = reinterpret_cast<int4 *>(ws + L.items3);
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
        rms_combine_bwd_kernel<<<(int)L.nblk, 256, 0, st>>>(fs.y_e, fs.topk_w, fs.slot_pos, w->gamma, dz, T, dl, k,
                                                               c->eps, dye, dg, dgamma_part);
        if ((rc = check_launch("rms_combine_bwd"))) return rc;
        dgamma_reduce_kernel<<<(dl + 255) / 256, 256, 0, st>>>(dgamma_part, (int)L.nblk, dl, g->dgamma, accumulate);
        if ((rc = check_launch("dgamma_reduce"))) return rc;
    }
    // routed experts on the forward's grouped kernel: pre-activations (the forward's gate|up
    // list), dh -> [dg | du] (a list of 256-feature blocks of I), x_lat rows (the down list)
    int4 *items_dglu = reinterpret_cast<int4 *>(ws + L.items_dglu);
    if ((rc = tc_worklist_single(fs.counts, fs.offsets, E, (I + 255) / 256, items_dglu, cnt + 28, (int)L.cap_dglu, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_GU32, c, w->W13, fs.x_lat, fs.perm, fs.items1, fs.n_items, cnt + 17, gu, nullptr,
                             nullptr, status, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_DGLU, c, w->W2, dye, nullptr, items_dglu, cnt + 28, cnt + 18, nullptr, gu, dgu,
                             status, st)))
        return rc;
    if ((rc = tc_grouped_bwd(TC_BWD_DXE, c, w->W13, dgu, nullptr, fs.items2, fs.n_items + 1, cnt + 19, dxe, nullptr,
                             nullptr, status, st)))
        return rc;
    // routed weight gradients, K = the expert's rows, computed transposed so that each lane
    // (an M index) stores along a row of the gradient:
    //   dW2[e]^T  [I, d_l]  = h^T dy_e             (A = h, B = dy_e by TMA)
    //   dW13[e]^T [d_l, 2I] = x_lat[perm]^T [dg|du] (A = x_lat gathered, B = [dg|du] by TMA)
    {
        BArgs a = dense_args(I, dl, 0, op(fs.h, I), op(dye, dl), g->dW2, I, accumulate, cnt + 23, status);
        a.offsets = fs.offsets; a.units = E * a.tiles_m * a.tiles_n; a.cstride = (long long)dl * I; a.out_t = 1;
        if ((rc = launch_bg<BE_F32, true, true, BG_WGRAD, true>(a, st, Tk))) return rc;
        BArgs b = dense_args(dl, 2 * I, 0, op(fs.x_lat, dl, 0, fs.perm), op(dgu, 2 * I), g->dW13, dl, accumulate,
                             cnt + 24, status);
        b.offsets = fs.offsets; b.units = E * b.tiles_m * b.tiles_n; b.cstride = (long long)2 * I * dl; b.out_t = 1;
        if ((rc = launch_bg<BE_F32, true, true, BG_WGRAD, true>(b, st, Tk))) return rc;
    }
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
