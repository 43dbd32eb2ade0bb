// tcgen05 / TMEM / TMA kernels of the bf16 layer type (sm_103a).
//
// Three persistent, warp-specialised kernels carry every contraction of the layer; in each,
// one thread issues TMA loads, one thread issues tcgen05.mma (M = 128, K = 16) into TMEM,
// and epilogue warps read the accumulators back with tcgen05.ld.
//
//  * dense_kernel  C[T, N] = epi(A[T, K] B[N, K]^T) with A = activations, B = weights, both
//    loaded by TMA into 128-byte-swizzled shared memory.  A tile is two 128-row sub-tiles
//    sharing one weight tile of BN rows (256; 64 for a batch of one row tile), with a
//    single-buffered accumulator drained by 8 epilogue warps.  K may be cut into up to four
//    segments, each with its own pair of tensor maps, added into one accumulator (used for
//    y = z W_out^T + sum_s h_s W2_s^T).  Epilogues: bf16 store, fp32 store and SiTU-GLU
//    (gate rows in the first half of the weight tile, up rows in the second).
//
//  * router_kernel  the router logits over three bf16 pieces of W_r with the TMEM
//    accumulator drained into fp32 registers every few K blocks, then sigmoid(logit + mu);
//    a small batch splits the K blocks over several CTAs per tile (router_kernel<true>)
//    and a reduce kernel adds their fp32 sums before the sigmoid.
//
//  * grouped_kernel  the routed experts, with the weights as the MMA's M operand
//    ("swap AB"): a work item is an expert, a block of output features (128 for gate|up,
//    whose gate and up rows make the two M sub-tiles; 256 for down) and a pass of up to 192
//    of its tokens (N rounded to 16).  The tokens' rows are gathered by index with cp.async
//    into the same swizzled layout a TMA load would produce, so the weights - the bytes that
//    bound this step - stream from HBM once per expert while the few tokens of each expert
//    cost a 16-wide MMA column granule instead of a 128-row tile.
//    Epilogues: SiTU-GLU -> h (expert gate/up), bf16 store -> y_e (expert down).
//
// Every wait on an mbarrier is bounded (%globaltimer); on expiry the kernel sets a shared
// abort flag and every role leaves its loop; the TMA producer then waits (bounded) for the
// copies it issued and the MMA thread for its MMAs, status[2] is set and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"
#include "ptx.cuh"
#include "tc_gemm.h"
#include "tcgen05.cuh"
#include "mx.cuh"
#include "tmap.h"

namespace slmoe {
namespace {

// Tile ids flow from the producer thread to the MMA thread and the epilogue warps through a
// TQ-slot shared-memory queue guarded by mbarriers.  The producer draws ids from a global
// counter when one is given (dynamic scheduling: a CTA that starts late, while another
// kernel still holds its SM, simply takes fewer tiles), else walks the static sequence
// blockIdx.x, blockIdx.x + gridDim.x, ...; an id >= tiles ends every role's loop.
constexpr int TQ = 2;
__device__ __forceinline__ bool tq_push(int *ids, uint64_t *full, uint64_t *empty, int &slot, uint32_t &ph,
                                        int tile, volatile WaitCtl *abort_flag) {
    if (!mbar_wait(&empty[slot], ph ^ 1, abort_flag)) return false;
    ids[slot] = tile;
    mbar_arrive(&full[slot]);
    if (++slot == TQ) { slot = 0; ph ^= 1; }
    return true;
}
// pop for a single consumer thread (arrives itself) or a warp (lane 0 arrives after the warp read)
__device__ __forceinline__ bool tq_pop(int *ids, uint64_t *full, uint64_t *empty, int &slot, uint32_t &ph,
                                       int &tile, volatile WaitCtl *abort_flag, bool warp_wide) {
    if (!mbar_wait(&full[slot], ph, abort_flag)) return false;
    tile = ids[slot];
    if (warp_wide) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[slot]);
    } else {
        mbar_arrive(&empty[slot]);
    }
    if (++slot == TQ) { slot = 0; ph ^= 1; }
    return true;
}

// ---------------------------------------------------------------- dense kernel
constexpr int EPI_BF16 = 0, EPI_GLU = 1, EPI_F32 = 3;
// Backward epilogues: dense SiTU-GLU derivative (rows = tokens); grouped (rows = features):
// fp32 gate|up pre-activations, fp32 transposed store, SiTU-GLU derivative.
constexpr int EPI_DGLU = 4, EPI_GU32 = 5, EPI_F32T = 6, EPI_DGLU_T = 7;
// MXFP8 store (the MXFP4 layer's latent activations): codes [rows, N] and E8M0 scales
// [rows, N / 32], N a multiple of 32.
constexpr int EPI_MX8 = 8;
// Operand majorness of the dense kernel (template MAJ): bit 0 = A MN-major, bit 1 = B MN-major.
// An MN-major operand is stored [K rows, M (or N) columns]; TMA loads it in 64 x 64 boxes.
constexpr int A_MN = 1, B_MN = 2;

struct TmaPack {
    CUtensorMap a[4];
    CUtensorMap b[4];
    CUtensorMap c;      // staged output [M, N]: boxes of 32 rows x 128 bytes, 128-byte swizzle
};

struct DenseArgs {
    int M, N;              // output rows and columns (GLU: h columns)
    int nseg;
    int kblocks[4];        // 64-wide K blocks per segment
    int glu_up_row;        // GLU: B-map row of the up half of h column n is n + glu_up_row
    int tiles_n, tiles;
    void *C;
    long long ldc;
    const float *mu;       // router: logit offset per column (nullable)
    float beta1, beta2;
    int32_t *status;
    int *counter;          // nullable: global tile counter (zeroed) for dynamic scheduling
    // router split K: tile t covers output tile t % tiles_mn and the K blocks of split
    // t / tiles_mn of ksplit; the raw fp32 sums go to partial[split][row][col] (row stride ldp)
    int ksplit, tiles_mn;
    float *partial;
    long long ldp;
    unsigned long long wait_limit_ns;   // 0 = the default limit of every bounded wait
    // failure-path check only: the producer issues no copies, so the MMA thread's wait on
    // the first stage can only run out (nothing is in flight when the kernel aborts)
    int stall_producer;
    int accumulate;        // EPI_F32: add into C instead of storing
    // EPI_DGLU: dh (the accumulator) -> [dg | du] from the fp32 pre-activations gu [rows, 2F]
    const float *gu;
    long long ld_gu;
    int F;
    __nv_bfloat16 *dgu;
    long long ld_dgu;
    float dbeta1, dbeta2;
    uint8_t *scales;       // EPI_MX8: block scales, ld_scales bytes per row
    long long ld_scales;
};

// Tile order of the dense kernel: bands of DENSE_BAND row tiles, rows fastest inside a band,
// so that the tiles in flight at once (about one per SM) share a few activation strips and a
// few weight strips that stay in L2, and each weight strip is read from HBM once per band
// instead of once per row tile.
constexpr int DENSE_BAND = 8;
__device__ __forceinline__ void dense_tile_mn(int tile, int tiles, int tiles_n, int &tm, int &tn) {
    const int tiles_m = tiles / tiles_n;
    const int per_band = DENSE_BAND * tiles_n;
    const int band = tile / per_band;
    const int m_first = band * DENSE_BAND;
    const int bm = min(DENSE_BAND, tiles_m - m_first);    // the last band may be short
    const int r = tile - band * per_band;
    tm = m_first + r % bm;
    tn = r / bm;
}

// A tile is MSUB row sub-tiles of 128 (the MMA's M) sharing one weight tile of BN rows, so a
// 64-wide K block is MSUB * 16 KB of activations + BN * 128 bytes of weights feeding MSUB * 4
// MMAs: with MSUB = 2 a stage (64 KB) covers 1024 MMA cycles and three stages cover the
// ~3000-cycle latency of a loaded L2, where single-row-tile stages (48 KB, 512 cycles) left
// the tensor pipe waiting a third of the time.  At BN = 256 the sub-tiles' accumulators fill
// the 512 TMEM columns, so the accumulator is single-buffered; each sub-tile has its own 4
// epilogue warps to drain it quickly.  (BN = 64, for a batch of one row tile, keeps the same
// structure in 128 columns.)
template <int BN, int EPI, int PACC>
struct DenseCfg {
    static constexpr int BM = 128, BK = 64, MSUB = 2, BM_TILE = BM * MSUB;
    static constexpr int A_BYTES = BM * BK * 2;           // one row sub-tile
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE = MSUB * A_BYTES + B_BYTES;
    static constexpr int STAGES = (196 * 1024) / STAGE;
    static constexpr int BN_OUT = EPI == EPI_GLU ? BN / 2 : BN;
    static constexpr int ACC = BN * PACC;                 // columns of one sub-tile's accumulator
    static constexpr int NBUF = 1;
    static constexpr int TMEM_COLS = MSUB * ACC;
    static constexpr int EPI_WARPS = 4 * MSUB;
    static constexpr int THREADS = (2 + EPI_WARPS) * 32;  // TMA, MMA, epilogue
    // staged output: a 4 KB tile per epilogue warp (32 rows x 128 bytes: 32 fp32 or 64 bf16
    // columns), written to the output by TMA; bf16 outputs need tiles of at least 64 columns.
    // (The SiTU-GLU output staged the same way measured no faster: its drain is its math.)
    static constexpr bool STAGE_OUT = EPI == EPI_F32 || (EPI == EPI_BF16 && BN_OUT >= 64);
    static constexpr int O_BYTES = STAGE_OUT ? EPI_WARPS * 4096 : 0;
    static constexpr int SMEM = STAGES * STAGE + O_BYTES + 1024 + 256;
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS >= 32 && TMEM_COLS <= 512 && STAGES >= 3,
                  "dense tile shape");
};

// [dg, du] of h = SiTU(g) * b2 tanh(u / b2) for an upstream dh (fp32, CUDA math functions):
// with t = tanh(g / b1) and s = sigmoid(g), SiTU = b1 t s and SiTU' = (1 - t^2) s + b1 t s (1 - s);
// the soft cap's derivative is 1 - tanh(u / b2)^2.  Each transcendental is evaluated once.
__device__ __forceinline__ void dglu(float dh, float g, float u, float b1, float b2, float &dg, float &du) {
    const float th = tanhf(g / b1);
    const float sg = 1.0f / (1.0f + expf(-g));
    const float tu = tanhf(u / b2);
    const float bts = b1 * th * sg;                       // SiTU(g)
    dg = dh * (b2 * tu) * ((1.0f - th * th) * sg + bts * (1.0f - sg));
    du = dh * bts * (1.0f - tu * tu);
}

template <int BN, int EPI, int PACC, int MAJ = 0>
__global__ void __launch_bounds__(DenseCfg<BN, EPI, PACC>::THREADS, 1) dense_kernel(const __grid_constant__ TmaPack maps,
                                                                                  const DenseArgs a) {
    using Cfg = DenseCfg<BN, EPI, PACC>;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sO = smem + STAGES * Cfg::STAGE;         // output staging
    uint64_t *full = reinterpret_cast<uint64_t *>(sO + Cfg::O_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *tq_full = tempty + 2;
    uint64_t *tq_empty = tq_full + TQ;
    uint64_t *mma_drain = tq_empty + TQ;
    int *tq_ids = reinterpret_cast<int *>(mma_drain + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tq_ids + TQ);
    volatile WaitCtl *abort_flag = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int p_stage = 0;                  // the TMA producer's ring position, kept for the drain
    uint32_t p_phase = 0;
    bool p_wrapped = false;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        mbar_init(mma_drain, 1);
        for (int q = 0; q < TQ; ++q) {
            mbar_init(&tq_full[q], 1);
            mbar_init(&tq_empty[q], 1 + Cfg::EPI_WARPS);
        }
        wait_ctl_init(abort_flag, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int &stage = p_stage;
        uint32_t &phase = p_phase;
        int qs = 0, it = 0;
        uint32_t qp = 0;
        for (;;) {
            const int tile = a.counter ? atomicAdd(a.counter, 1) : (int)blockIdx.x + (it++) * (int)gridDim.x;
            if (!tq_push(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag)) goto done;
            if (tile >= a.tiles) break;
            int tm, tn;
            dense_tile_mn(tile, a.tiles, a.tiles_n, tm, tn);
            const int m0 = tm * Cfg::BM_TILE;
            const int n0 = tn * Cfg::BN_OUT;
            for (int s = 0; s < a.nseg; ++s) {
                for (int kb = 0; kb < a.kblocks[s]; ++kb) {
                    if (a.stall_producer) continue;
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) goto done;
                    mbar_expect_tx(&full[stage], Cfg::STAGE);
                    const uint32_t sa = su32(smem + stage * Cfg::STAGE);
                    const uint32_t sb = sa + Cfg::MSUB * Cfg::A_BYTES;
#pragma unroll
                    for (int j = 0; j < Cfg::MSUB; ++j) {
                        if (MAJ & A_MN) {
                            tma_load_2d(sa + j * Cfg::A_BYTES, &maps.a[s], &full[stage], m0 + j * Cfg::BM, kb * Cfg::BK);
                            tma_load_2d(sa + j * Cfg::A_BYTES + 8192, &maps.a[s], &full[stage], m0 + j * Cfg::BM + 64,
                                        kb * Cfg::BK);
                        } else {
                            tma_load_2d(sa + j * Cfg::A_BYTES, &maps.a[s], &full[stage], kb * Cfg::BK, m0 + j * Cfg::BM);
                        }
                    }
                    if (MAJ & B_MN) {
#pragma unroll
                        for (int g = 0; g < BN / 64; ++g)
                            tma_load_2d(sb + g * 8192, &maps.b[s], &full[stage], n0 + 64 * g, kb * Cfg::BK);
                    } else if (EPI == EPI_GLU) {
                        tma_load_2d(sb, &maps.b[s], &full[stage], kb * Cfg::BK, n0);
                        tma_load_2d(sb + (BN / 2) * 128, &maps.b[s], &full[stage], kb * Cfg::BK,
                                    n0 + a.glu_up_row);
                    } else {
                        tma_load_2d(sb, &maps.b[s], &full[stage], kb * Cfg::BK, n0);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; p_wrapped = true; }
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC =
            idesc_bf16(128, BN) | ((MAJ & A_MN) ? (1u << 15) : 0u) | ((MAJ & B_MN) ? (1u << 16) : 0u);
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        uint32_t bphase = 0;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            int tile;
            if (!tq_pop(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag, false)) goto done;
            if (tile >= a.tiles) break;
            if (!mbar_wait(&tempty[buf], bphase ^ 1, abort_flag)) goto done;
            tc_after();
            int kg = 0;
            for (int s = 0; s < a.nseg; ++s) {
                for (int kb = 0; kb < a.kblocks[s]; ++kb, ++kg) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) goto done;
                    tc_after();
                    const uint32_t sa = su32(smem + stage * Cfg::STAGE);
                    const uint32_t sb = sa + Cfg::MSUB * Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = (MAJ & B_MN) ? mn_desc(sb + kk * 2048, 8192) : sdesc(sb + kk * 32);
#pragma unroll
                        for (int j = 0; j < Cfg::MSUB; ++j) {
                            const uint32_t aj = sa + j * Cfg::A_BYTES;
                            const uint64_t ad = (MAJ & A_MN) ? mn_desc(aj + kk * 2048, 8192) : sdesc(aj + kk * 32);
                            umma(tmem_base + j * Cfg::ACC + (kg % PACC) * BN, ad, bd, IDESC,
                                 (kg >= PACC || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            umma_commit(&tfull[buf]);
            if (++buf == Cfg::NBUF) { buf = 0; bphase ^= 1; }
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue warps: warp w drains TMEM
        // lane quarter w % 4 of row sub-tile (w - 2) / 4
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int sub = (warp - 2) >> 2;
        const int row_in_tile = sub * Cfg::BM + q * 32 + lane;
            int buf = 0;
        uint32_t bphase = 0;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            int tile;
            if (!tq_pop(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag, true)) goto done;
            if (tile >= a.tiles) break;
            if (!mbar_wait(&tfull[buf], bphase, abort_flag)) goto done;
            tc_after();
            int tm, tn;
            dense_tile_mn(tile, a.tiles, a.tiles_n, tm, tn);
            const int row = tm * Cfg::BM_TILE + row_in_tile;
            const int n0 = tn * Cfg::BN_OUT;
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + sub * Cfg::ACC;
            const bool row_ok = row < a.M;
            if (EPI == EPI_MX8) {
                // 32-column chunks: one MXFP8 block of this thread's row per chunk
                uint8_t *C = static_cast<uint8_t *>(a.C) + (long long)row * a.ldc;
                uint8_t *S = a.scales + (long long)row * a.ld_scales;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r0[16], r1[16];
                    TMEM_LD16(tb + c, r0);
                    TMEM_LD16(tb + c + 16, r1);
                    tmem_wait_ld();
                    const int n = n0 + c;
                    if (row_ok && n < a.N) {
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            v[i] = __uint_as_float(r0[i]);
                            v[16 + i] = __uint_as_float(r1[i]);
                        }
                        uint32_t w[8];
                        S[n >> 5] = (uint8_t)mx8_quant32(v, w);
                        *reinterpret_cast<uint4 *>(C + n) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(C + n + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else if (EPI == EPI_BF16 && Cfg::STAGE_OUT) {
                // 64 columns at a time: the warp's 32 rows staged in shared memory (128-byte
                // swizzle) and written by one TMA store
                uint8_t *stg = sO + (warp - 2) * 4096;
                uint8_t *rowp = stg + lane * 128;
                const int row0w = tm * Cfg::BM_TILE + sub * Cfg::BM + q * 32;
#pragma unroll 1
                for (int c = 0; c < BN; c += 64) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) TMEM_LD16(tb + c + 16 * u, r[u]);
                    if (lane == 0) bulk_wait_read0();   // the warp's last store has read the tile
                    __syncwarp();
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int hv = 0; hv < 2; ++hv) {
                            const uint32_t *x = r[u] + 8 * hv;
                            *reinterpret_cast<uint4 *>(rowp + (((2 * u + hv) ^ (lane & 7)) << 4)) = make_uint4(
                                pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                        }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0 && row0w < a.M && n0 + c < a.N) {   // the map's bounds cut the rest
                        tma_store_2d(&maps.c, su32(stg), n0 + c, row0w);
                        bulk_commit();
                    }
                }
            } else if (EPI == EPI_BF16) {
                __nv_bfloat16 *C = static_cast<__nv_bfloat16 *>(a.C) + (long long)row * a.ldc;
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t r[16];
                    TMEM_LD16(tb + c, r);
                    tmem_wait_ld();
                    const int n = n0 + c;
                    if (row_ok) {
                        if (n + 16 <= a.N) {
                            uint4 v0 = make_uint4(pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                                  pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                                  pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                                  pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7])));
                            uint4 v1 = make_uint4(pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9])),
                                                  pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11])),
                                                  pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13])),
                                                  pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15])));
                            *reinterpret_cast<uint4 *>(C + n) = v0;
                            *reinterpret_cast<uint4 *>(C + n + 8) = v1;
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)   // static indices keep r in registers
                                if (n + i < a.N) C[n + i] = __float2bfloat16_rn(__uint_as_float(r[i]));
                        }
                    }
                }
            } else if (EPI == EPI_F32) {
                // 32 columns at a time: the warp's 32 rows staged in shared memory (the 128-byte
                // swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8)) and written by one TMA
                // store, or added in by a TMA reduction, instead of 16-byte stores to 32 rows
                uint8_t *stg = sO + (warp - 2) * 4096;
                uint8_t *rowp = stg + lane * 128;
                const int row0w = tm * Cfg::BM_TILE + sub * Cfg::BM + q * 32;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r0[16], r1[16];
                    TMEM_LD16(tb + c, r0);
                    TMEM_LD16(tb + c + 16, r1);
                    if (lane == 0) bulk_wait_read0();   // the warp's last store has read the tile
                    __syncwarp();
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        *reinterpret_cast<uint4 *>(rowp + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
                        *reinterpret_cast<uint4 *>(rowp + (((j + 4) ^ (lane & 7)) << 4)) =
                            make_uint4(r1[4 * j], r1[4 * j + 1], r1[4 * j + 2], r1[4 * j + 3]);
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0 && row0w < a.M && n0 + c < a.N) {   // the map's bounds cut the rest
                        if (a.accumulate) tma_reduce_add_2d(&maps.c, su32(stg), n0 + c, row0w);
                        else tma_store_2d(&maps.c, su32(stg), n0 + c, row0w);
                        bulk_commit();
                    }
                }
            } else if (EPI == EPI_DGLU) {
                // rows are tokens, columns features f: gate at f, up at F + f; 16 columns at a
                // time with 16-byte loads of the pre-activations and 16-byte stores of [dg | du]
                // when the rows allow it (F, the pitches and n 16-element aligned)
                const float *gr = a.gu + (long long)row * a.ld_gu;
                __nv_bfloat16 *dr = a.dgu + (long long)row * a.ld_dgu;
                const bool vec = ((a.F | a.ld_gu | a.ld_dgu) & 15) == 0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t r[16];
                    TMEM_LD16(tb + c, r);
                    tmem_wait_ld();
                    const int n = n0 + c;
                    if (!row_ok) continue;
                    if (vec && n + 16 <= a.N) {
                        float g[16], u[16], dg[16], du[16];
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 gv = *reinterpret_cast<const float4 *>(gr + n + i);
                            const float4 uv = *reinterpret_cast<const float4 *>(gr + a.F + n + i);
                            g[i] = gv.x; g[i + 1] = gv.y; g[i + 2] = gv.z; g[i + 3] = gv.w;
                            u[i] = uv.x; u[i + 1] = uv.y; u[i + 2] = uv.z; u[i + 3] = uv.w;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) dglu(__uint_as_float(r[i]), g[i], u[i], a.dbeta1, a.dbeta2, dg[i], du[i]);
                        uint32_t pg[8], pu[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            pg[i] = pack_bf16(dg[2 * i], dg[2 * i + 1]);
                            pu[i] = pack_bf16(du[2 * i], du[2 * i + 1]);
                        }
                        *reinterpret_cast<uint4 *>(dr + n) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
                        *reinterpret_cast<uint4 *>(dr + n + 8) = make_uint4(pg[4], pg[5], pg[6], pg[7]);
                        *reinterpret_cast<uint4 *>(dr + a.F + n) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
                        *reinterpret_cast<uint4 *>(dr + a.F + n + 8) = make_uint4(pu[4], pu[5], pu[6], pu[7]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (n + i >= a.N) continue;
                            float dg, du;
                            dglu(__uint_as_float(r[i]), gr[n + i], gr[a.F + n + i], a.dbeta1, a.dbeta2, dg, du);
                            dr[n + i] = __float2bfloat16_rn(dg);
                            dr[a.F + n + i] = __float2bfloat16_rn(du);
                        }
                    }
                }
            } else if (EPI == EPI_GLU) {
                __nv_bfloat16 *C = static_cast<__nv_bfloat16 *>(a.C) + (long long)row * a.ldc;
                const float ib1 = 1.0f / a.beta1, ib2 = 1.0f / a.beta2;
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 16) {
                    uint32_t g[16], u[16];
                    TMEM_LD16(tb + c, g);
                    TMEM_LD16(tb + BN / 2 + c, u);
                    tmem_wait_ld();
                    const int n = n0 + c;
                    if (row_ok) {
                        float h[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            h[i] = situ_glu_fast(__uint_as_float(g[i]), __uint_as_float(u[i]), ib1, a.beta1,
                                                 ib2, a.beta2);
                        if (n + 16 <= a.N) {
                            uint4 v0 = make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]),
                                                  pack_bf16(h[4], h[5]), pack_bf16(h[6], h[7]));
                            uint4 v1 = make_uint4(pack_bf16(h[8], h[9]), pack_bf16(h[10], h[11]),
                                                  pack_bf16(h[12], h[13]), pack_bf16(h[14], h[15]));
                            *reinterpret_cast<uint4 *>(C + n) = v0;
                            *reinterpret_cast<uint4 *>(C + n + 8) = v1;
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)   // static indices keep h in registers
                                if (n + i < a.N) C[n + i] = __float2bfloat16_rn(h[i]);
                        }
                    }
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            if (++buf == Cfg::NBUF) { buf = 0; bphase ^= 1; }
        }
    }
done:
    if (Cfg::STAGE_OUT) bulk_wait_all();   // output stores read shared memory until they complete
    __syncthreads();
    if (abort_flag->abort) {   // every role has stopped: let copies and MMAs in flight finish
        if (warp == 0 && lane == 0) drain_ring(full, STAGES, p_stage, p_phase, p_wrapped);
        if (warp == 1 && lane == 0) {
            umma_commit(mma_drain);
            mbar_wait_drain(mma_drain, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    if (threadIdx.x == 0 && abort_flag->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// ---------------------------------------------------------------- router logits
// C[T, E] = sigmoid(x . (W_hi + W_mid + W_lo)^T + mu) in fp32.  The three bf16 weight pieces
// are three K segments added into one accumulator.  To keep the logits fp32-faithful, the
// MMA accumulates only RT_DRAIN K blocks into a fresh TMEM buffer; two epilogue
// warpgroups (columns 0..111 and 112..223) drain each such partial sum into fp32 registers
// (round-to-nearest adds) while the next chunk fills the other buffer, so no tensor-core
// accumulation chain is longer than 4 * RT_DRAIN MMA steps.  BN = 224 tiles E = 896 exactly.
constexpr int RT_BN = 224, RT_HALF = RT_BN / 2, RT_DRAIN = 8;
constexpr int RT_STAGE = 128 * 128 + RT_BN * 128;
constexpr int RT_STAGES = 5;
constexpr int RT_SMEM = RT_STAGES * RT_STAGE + 1024 + 256;
constexpr int RT_THREADS = 320;               // TMA, MMA, 8 epilogue warps

template <int N>
__device__ __forceinline__ void drain_add(uint32_t taddr, float *acc) {
    // N x 16 columns: issue all loads, one wait, then add
    uint32_t r[N][16];
#pragma unroll
    for (int b = 0; b < N; ++b) TMEM_LD16(taddr + 16 * b, r[b]);
    tmem_wait_ld();
#pragma unroll
    for (int b = 0; b < N; ++b)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[16 * b + i] += __uint_as_float(r[b][i]);
}

// Output tile and K range (global K blocks [g0, g1) over the three pieces) of a router tile
// id; with SPLIT, tile t covers output tile t % tiles_mn and split t / tiles_mn of ksplit.
template <bool SPLIT>
__device__ __forceinline__ void router_tile(const DenseArgs &a, int tile, int ktot, int &m0, int &n0, int &g0,
                                            int &g1) {
    int mn = tile, ks = 0;
    if (SPLIT) {
        ks = tile / a.tiles_mn;
        mn = tile - ks * a.tiles_mn;
    }
    m0 = (mn / a.tiles_n) * 128;
    n0 = (mn % a.tiles_n) * RT_BN;
    g0 = SPLIT ? (int)((long long)ks * ktot / a.ksplit) : 0;
    g1 = SPLIT ? (int)((long long)(ks + 1) * ktot / a.ksplit) : ktot;
}

template <bool SPLIT>
__global__ void __launch_bounds__(RT_THREADS, 1) router_kernel(const __grid_constant__ TmaPack maps,
                                                               const DenseArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + RT_STAGES * RT_STAGE);
    uint64_t *empty = full + RT_STAGES;
    uint64_t *tfull = empty + RT_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *tq_full = tempty + 2;
    uint64_t *tq_empty = tq_full + TQ;
    uint64_t *mma_drain = tq_empty + TQ;
    int *tq_ids = reinterpret_cast<int *>(mma_drain + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tq_ids + TQ);
    volatile WaitCtl *abort_flag = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(mma_drain, 1);
        for (int s = 0; s < RT_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);
        }
        for (int q = 0; q < TQ; ++q) {
            mbar_init(&tq_full[q], 1);
            mbar_init(&tq_empty[q], 9);
        }
        wait_ctl_init(abort_flag, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;
    int ktot = 0;
    for (int s = 0; s < a.nseg; ++s) ktot += a.kblocks[s];

    if (warp == 0 && lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool wrapped = false;
        int qs = 0, it = 0;
        uint32_t qp = 0;
        for (;;) {
            const int tile = a.counter ? atomicAdd(a.counter, 1) : (int)blockIdx.x + (it++) * (int)gridDim.x;
            if (!tq_push(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag)) goto producer_out;
            if (tile >= a.tiles) break;
            int m0, n0, g0, g1;
            router_tile<SPLIT>(a, tile, ktot, m0, n0, g0, g1);
            for (int s = 0, g = 0; s < a.nseg; ++s) {
                for (int kb = 0; kb < a.kblocks[s]; ++kb, ++g) {
                    if (SPLIT && (g < g0 || g >= g1)) continue;
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) goto producer_out;
                    mbar_expect_tx(&full[stage], RT_STAGE);
                    const uint32_t sa = su32(smem + stage * RT_STAGE);
                    tma_load_2d(sa, &maps.a[s], &full[stage], kb * 64, m0);
                    tma_load_2d(sa + 128 * 128, &maps.b[s], &full[stage], kb * 64, n0);
                    if (++stage == RT_STAGES) { stage = 0; phase ^= 1; wrapped = true; }
                }
            }
        }
    producer_out:   // wait (bounded) until every copy issued has landed
        drain_ring(full, RT_STAGES, stage, phase, wrapped);
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t IDESC = idesc_bf16(128, RT_BN);
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        uint32_t bphase = 0;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            int tile;
            if (!tq_pop(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag, false)) goto mma_out;
            if (tile >= a.tiles) break;
            int m0, n0, g0, g1;
            router_tile<SPLIT>(a, tile, ktot, m0, n0, g0, g1);
            const int klen = g1 - g0;
            int kg = 0;                               // K blocks of this tile so far
            for (int s = 0, g = 0; s < a.nseg; ++s) {
                for (int kb = 0; kb < a.kblocks[s]; ++kb, ++g) {
                    if (SPLIT && (g < g0 || g >= g1)) continue;
                    const bool first = (kg % RT_DRAIN) == 0;
                    if (first) {
                        if (!mbar_wait(&tempty[buf], bphase ^ 1, abort_flag)) goto mma_out;
                        tc_after();
                    }
                    if (!mbar_wait(&full[stage], phase, abort_flag)) goto mma_out;
                    tc_after();
                    const uint32_t d = tmem_base + buf * 256;
                    const uint32_t sa = su32(smem + stage * RT_STAGE);
                    const uint32_t sb = sa + 128 * 128;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma(d, sdesc(sa + kk * 32), sdesc(sb + kk * 32), IDESC, (!first || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == RT_STAGES) { stage = 0; phase ^= 1; }
                    if ((kg % RT_DRAIN) == RT_DRAIN - 1 || kg == klen - 1) {
                        umma_commit(&tfull[buf]);
                        if (++buf == 2) { buf = 0; bphase ^= 1; }
                    }
                    ++kg;
                }
            }
        }
    mma_out:        // wait (bounded) until every MMA issued has finished
        umma_commit(mma_drain);
        mbar_wait_drain(mma_drain, 0);
    } else if (warp >= 2) {
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;             // column half drained by this warp
        const int row_in_tile = q * 32 + lane;
        const int nchunks_all = (ktot + RT_DRAIN - 1) / RT_DRAIN;
        int buf = 0;
        uint32_t bphase = 0;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            int tile;
            if (!tq_pop(tq_ids, tq_full, tq_empty, qs, qp, tile, abort_flag, true)) goto done;
            if (tile >= a.tiles) break;
            int nchunks = nchunks_all;
            if constexpr (SPLIT) {
                int m0s, n0s, g0, g1;
                router_tile<true>(a, tile, ktot, m0s, n0s, g0, g1);
                nchunks = (g1 - g0 + RT_DRAIN - 1) / RT_DRAIN;
            }
            float acc[RT_HALF];
#pragma unroll
            for (int i = 0; i < RT_HALF; ++i) acc[i] = 0.f;
            for (int ch = 0; ch < nchunks; ++ch) {
                if (!mbar_wait(&tfull[buf], bphase, abort_flag)) goto done;
                tc_after();
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + buf * 256 + half * RT_HALF;
                drain_add<4>(tb, acc);
                drain_add<3>(tb + 64, acc + 64);
                tc_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                if (++buf == 2) { buf = 0; bphase ^= 1; }
            }
            if constexpr (SPLIT) {
                // raw fp32 logit sums of this split; router_splitk_reduce_kernel adds the
                // splits in order, then the offset and the sigmoid
                const int ks = tile / a.tiles_mn, mn = tile - ks * a.tiles_mn;
                const int row = (mn / a.tiles_n) * 128 + row_in_tile;
                const int n0 = (mn % a.tiles_n) * RT_BN + half * RT_HALF;
                if (row < a.M) {
                    float *P = a.partial + ((long long)ks * a.M + row) * a.ldp;
#pragma unroll
                    for (int i = 0; i < RT_HALF; ++i)
                        if (n0 + i < a.N) P[n0 + i] = acc[i];
                }
                continue;
            }
            const int row = (tile / a.tiles_n) * 128 + row_in_tile;
            const int n0 = (tile % a.tiles_n) * RT_BN + half * RT_HALF;
            if (row < a.M) {
                float *C = static_cast<float *>(a.C) + (long long)row * a.ldc;
                const bool vec = (a.ldc & 3) == 0;       // rows 16-byte aligned: float4 stores
#pragma unroll
                for (int i = 0; i < RT_HALF; i += 4) {
                    float o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int n = n0 + i + j;
                        const float v = acc[i + j] + ((a.mu && n < a.N) ? a.mu[n] : 0.f);
                        o[j] = 1.0f / (1.0f + expf(-v));
                    }
                    const int n = n0 + i;
                    if (vec && n + 4 <= a.N) {
                        *reinterpret_cast<float4 *>(C + n) = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (n + j < a.N) C[n + j] = o[j];
                    }
                }
            }
        }
    }
done:
    __syncthreads();
    if (warp == 1) {
        tc_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && abort_flag->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// ---------------------------------------------------------------- grouped (routed experts)
// A work item is (expert e, feature block fb, token pass): weight sub-tiles of 128 rows (the
// MMA's M) times the pass's tokens (N <= PASS, rounded to 16).  The weights stream from HBM
// through a ring of TMA loads (112-128 KB in flight); the pass's token rows are gathered from
// L2 by cp.async into a 4-deep ring, each gather thread signalling a stage with
// cp.async.mbarrier.arrive.noinc (the MMA thread fences the generic-proxy writes to the async
// proxy after its wait).  Items come from a list built on the device (expert-major, then
// feature block, then pass, so the passes of one weight tile are adjacent and the CTAs that
// take them together share it through L2) and are handed out dynamically through a global
// counter, so the heavy skew of expert loads cannot leave one CTA with all the hot experts.
// Both routed-expert GEMMs use 192-token passes drained by 8 or 12 epilogue warps.
//   Gate|up (K = d_latent): NSUB = 2 pairs the gate rows fb*128.. with the up rows I + fb*128..
//   for the fused SiTU-GLU in one accumulator set; its MMAs are long beside the drain.  (The
//   backward's grouped GEMMs take this form too, with two blocks of 128 features.)
//   Down (K = I = 512, DBUF): it drains as many fp32 values as it accumulates over a short K.
//   Timed per role, the single-set form spent 40 % of its MMA thread's time waiting for the
//   drain, and the drain's time was the epilogue warps' 2-byte y_e stores stalling on the
//   memory system (its tensor-memory loads took a few percent of it).  So each item is one
//   128-feature sub-tile in one of two accumulator sets (columns 0 and 256), and each half of
//   the epilogue warps stages 16 rows at a time in shared memory, from where one thread
//   stores them by TMA: the drain overlaps the next item's MMAs and never waits on a store.
//   (The staged stores with two sub-tiles and one set, or two sets of <= 128-token passes,
//   measured slower.)
constexpr int G_GATHER_THREADS = 128;
constexpr int G_TQ = 4;                           // item queue slots

template <bool DBUF>
struct GCfg {
    static constexpr int NSUB = DBUF ? DOWN_NSUB : 2;        // weight sub-tiles per item
    static constexpr int PASS = GROUPED_PASS;                // tokens per pass
    static constexpr int A_BYTES = NSUB * 128 * 128;
    static constexpr int A_STAGES = !DBUF ? 4 : NSUB == 1 ? 7 : 3;   // what shared memory leaves
    static constexpr int B_BYTES = PASS * 128;
    static constexpr int B_STAGES = 4;
    static constexpr int NBUF = DBUF && NSUB == 1 ? 2 : 1;   // accumulator sets, at columns 0 / 256
    static constexpr int SUB1_COL = 256;                     // sub-tile 1 (NSUB = 2)
    // epilogue warps per TMEM lane quadrant: three with one accumulator set, whose drain holds
    // up the MMAs (1.128 against 1.141 ms for expert gate|up at K3 with two; four, at 80
    // registers a thread, 1.18 ms), two with two sets
    static constexpr int EPI_WARPS = DBUF ? 8 : 12;
    static constexpr int GATHER_WARP0 = 2 + EPI_WARPS;
    static constexpr int THREADS = (2 + EPI_WARPS + 4) * 32;   // TMA, MMA, epilogue, 4 gather warps
    // DBUF: output staging, two 16-row x (128 NSUB)-feature bf16 chunks per half of the epilogue warps
    static constexpr int O_CHUNK = 16 * 128 * NSUB * 2;
    static constexpr int O_BYTES = DBUF ? 4 * O_CHUNK : 0;
    static constexpr int SMEM = A_STAGES * A_BYTES + B_STAGES * B_BYTES + O_BYTES + 1024 + 512;
    static_assert(SMEM <= 232448, "shared memory");
};

struct GroupedArgs {
    int kblocks;
    int a_rows_pe;        // rows of the weight view per expert
    int a_sub1;           // row offset of sub-tile 1 inside a feature block
    int a_fb_stride;      // rows between feature blocks
    const int4 *items;    // {e, fb | multi_pass << 16, first row in perm order, tokens}
    const int *n_items;
    int *counter;         // zeroed item counter
    const int32_t *b_index;               // nullable: token row = b_index[row]
    const __nv_bfloat16 *b_src;
    long long b_ld;
    int b_K;
    void *out;            // bf16 (forward epilogues) or fp32 (EPI_GU32, EPI_F32T)
    long long out_ld;
    int out_cols;         // features of the output (EPI_GU32 / EPI_DGLU_T: the up half's offset F)
    float beta1, beta2;
    int32_t *status;
    unsigned long long wait_limit_ns;   // 0 = the default limit of every bounded wait
    const float *gu;      // EPI_DGLU_T: fp32 pre-activations [rows, 2F]
    long long ld_gu;
    __nv_bfloat16 *dgu;   // EPI_DGLU_T: [dg | du] out, bf16 [rows, 2F]
    long long ld_dgu;
    // MXFP4 layer (grouped_mx_kernel): E8M0 block scales of the weight rows (a_scale_ld bytes
    // per row; rows at or past a_rows_total read scale 0), of the token rows (b_scale_ld bytes
    // per row of b_src) and of the MXFP8 output rows (EPI_GLU: out_scale_ld bytes per row)
    const uint8_t *a_scales;
    int a_scale_ld;
    long long a_rows_total;
    const uint8_t *b_scales;
    int b_scale_ld;
    uint8_t *out_scales;
    int out_scale_ld;
};

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(map), "r"(su32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}
// 8 x 8 transpose within each aligned group of 8 lanes (t = lane % 8): on entry v[i] is row t,
// column i of the group's matrix; on exit v[i] is row i, column t.  Three exchange stages
// (lane distance 4, 2, 1), each swapping the off-diagonal halves of 2 x 2 blocks.
__device__ __forceinline__ void transpose8(float (&v)[8], int t) {
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & s) continue;
            const bool hi = (t & s) != 0;
            const float send = hi ? v[i] : v[i | s];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            if (hi) v[i] = recv;
            else v[i | s] = recv;
        }
    }
}
// Work lists of both routed-expert GEMMs in one block: per expert ceil(n_e / cap) passes of
// balanced size (0 when n_e = 0) times nfb feature blocks.  The threads scan the experts'
// item counts into per-expert bases (kept in shared memory), then each warp writes one
// expert's items at a time with its lanes in parallel, so a hot expert's items do not fall
// to a single thread.
constexpr int WL_MAX_E = 4096;
__global__ void __launch_bounds__(1024)
worklist_kernel(const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets, int E,
                int nfb1, int cap1, int4 *__restrict__ items1, int nfb2, int cap2,
                int4 *__restrict__ items2, int *__restrict__ n_items, int max1, int max2) {
    __shared__ int wsum[2][32];
    __shared__ int ebase[2][WL_MAX_E];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = tid * per;
    const int caps[2] = {cap1, cap2}, nfbs[2] = {nfb1, nfb2};
    int loc[2] = {0, 0};
    for (int e = e0; e < e0 + per && e < E; ++e) {
        const int n = counts[e];
        loc[0] += nfb1 * ((n + cap1 - 1) / cap1);
        loc[1] += nfb2 * ((n + cap2 - 1) / cap2);
    }
    int incl[2] = {loc[0], loc[1]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int l = 0; l < 2; ++l) {
            const int v = __shfl_up_sync(0xffffffffu, incl[l], o);
            if (lane >= o) incl[l] += v;
        }
    }
    if (lane == 31) { wsum[0][w] = incl[0]; wsum[1][w] = incl[1]; }
    __syncthreads();
    int base[2] = {0, 0};
    for (int i = 0; i < w; ++i) { base[0] += wsum[0][i]; base[1] += wsum[1][i]; }
    base[0] += incl[0] - loc[0];
    base[1] += incl[1] - loc[1];
    if (tid == blockDim.x - 1) {
        n_items[0] = min(base[0] + loc[0], max1);
        n_items[1] = min(base[1] + loc[1], max2);
    }
    for (int e = e0; e < e0 + per && e < E; ++e) {
        const int n = counts[e];
#pragma unroll
        for (int l = 0; l < 2; ++l) {
            ebase[l][e] = base[l];
            base[l] += nfbs[l] * ((n + caps[l] - 1) / caps[l]);
        }
    }
    __syncthreads();
    int4 *lists[2] = {items1, items2};
    for (int e = w; e < E; e += blockDim.x >> 5) {
        const int n = counts[e], off = offsets[e];
#pragma unroll
        for (int l = 0; l < 2; ++l) {
            const int np = (n + caps[l] - 1) / caps[l];
            if (np == 0) continue;
            const int chunk = (n + np - 1) / np;
            const int multi = np > 1 ? 1 : 0;
            const int maxl = l == 0 ? max1 : max2;
            for (int j = lane; j < nfbs[l] * np; j += 32) {
                const int fb = j / np, pass = j - fb * np;
                const int c0 = pass * chunk;
                // the workspace holds the largest possible list; never write past it
                if (ebase[l][e] + j < maxl)
                    lists[l][ebase[l][e] + j] = make_int4(e, fb | (multi << 16), off + c0, min(chunk, n - c0));
            }
        }
    }
}

// AMN: the weights are MN-major (stored [K rows, features], the transposed use of a forward
// weight in the backward): each 128-feature sub-tile is two 64 x 64 TMA boxes; a_rows_pe is then
// the K rows per expert, a_fb_stride the features per block and a_sub1 the second sub-tile's
// feature offset.
template <int EPI, bool DBUF, bool AMN = false>
__global__ void __launch_bounds__(GCfg<DBUF>::THREADS, 1) grouped_kernel(const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap omap,
                                                               const GroupedArgs a) {
    using Cfg = GCfg<DBUF>;
    constexpr int AST = Cfg::A_STAGES, BST = Cfg::B_STAGES, NBUF = Cfg::NBUF, SUB1 = Cfg::SUB1_COL;
    constexpr bool TWO = Cfg::NSUB == 2;
    // staged output (TMA stores): the forward's expert down-projection
    constexpr bool STAGED = DBUF && EPI == EPI_BF16;
    static_assert(!DBUF || (EPI == EPI_BF16 && !AMN) || (EPI == EPI_DGLU_T && AMN),
                  "one sub-tile in two accumulator sets: expert down, and the backward's dh + SiTU-GLU derivative");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + AST * Cfg::A_BYTES;
    uint8_t *sO = sB + BST * Cfg::B_BYTES;     // DBUF output staging
    int4 *q_items = reinterpret_cast<int4 *>(sO + Cfg::O_BYTES);
    uint64_t *q_full = reinterpret_cast<uint64_t *>(q_items + G_TQ);
    uint64_t *q_empty = q_full + G_TQ;
    uint64_t *a_full = q_empty + G_TQ;
    uint64_t *a_empty = a_full + AST;
    uint64_t *b_full = a_empty + AST;
    uint64_t *b_empty = b_full + BST;
    uint64_t *tfull = b_empty + BST;
    uint64_t *tempty = tfull + NBUF;
    uint64_t *mma_drain = tempty + NBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_drain + 1);
    volatile WaitCtl *abort_flag = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int p_stage = 0;                  // the weight producer's ring position, kept for the drain
    uint32_t p_phase = 0;
    bool p_wrapped = false;
    if (threadIdx.x == 0) {
        mbar_init(mma_drain, 1);
        for (int s = 0; s < G_TQ; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1 + Cfg::EPI_WARPS + 4);   // MMA thread, epilogue, gather warps
        }
        for (int s = 0; s < AST; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < BST; ++s) {
            mbar_init(&b_full[s], G_GATHER_THREADS);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        wait_ctl_init(abort_flag, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;

    // consumers take the next item from the queue; a negative token count ends the loop
    auto pop = [&](int &qs, uint32_t &qp, int4 &it, bool warp_wide) -> bool {
        if (!mbar_wait(&q_full[qs], qp, abort_flag)) return false;
        it = q_items[qs];
        if (warp_wide) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qs]);
        } else {
            mbar_arrive(&q_empty[qs]);
        }
        if (++qs == G_TQ) { qs = 0; qp ^= 1; }
        return true;
    };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ item fetch + weights by TMA
        const uint64_t pol_first = policy_evict_first();
        const int n_items = *a.n_items;
        int &stage = p_stage;
        uint32_t &phase = p_phase;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            const int idx = atomicAdd(a.counter, 1);
            const int4 it = idx < n_items ? a.items[idx] : make_int4(0, 0, 0, -1);
            if (!mbar_wait(&q_empty[qs], qp ^ 1, abort_flag)) goto done;
            q_items[qs] = it;
            mbar_arrive(&q_full[qs]);
            if (++qs == G_TQ) { qs = 0; qp ^= 1; }
            if (it.w < 0) break;
            const int fb = it.y & 0xffff;
            const bool multi = (it.y >> 16) != 0;
            const int row0 = it.x * a.a_rows_pe + fb * a.a_fb_stride;
            for (int kb = 0; kb < a.kblocks; ++kb) {
                if (!mbar_wait(&a_empty[stage], phase ^ 1, abort_flag)) goto done;
                mbar_expect_tx(&a_full[stage], Cfg::A_BYTES);
                const uint32_t sa = su32(sA + stage * Cfg::A_BYTES);
                if (AMN) {         // features fb * stride (+ sub1), K rows of expert it.x
                    const int f0 = fb * a.a_fb_stride, kr = it.x * a.a_rows_pe + kb * 64;
#pragma unroll
                    for (int sub = 0; sub < Cfg::NSUB; ++sub)
#pragma unroll
                        for (int g = 0; g < 2; ++g)
                            tma_load_2d_hint(sa + sub * 128 * 128 + g * 8192, &wmap, &a_full[stage],
                                             f0 + sub * a.a_sub1 + 64 * g, kr, pol_first);
                } else if (multi) {   // other passes of this tile run alongside: normal L2 policy
                    tma_load_2d(sa, &wmap, &a_full[stage], kb * 64, row0);
                    if (TWO) tma_load_2d(sa + 128 * 128, &wmap, &a_full[stage], kb * 64, row0 + a.a_sub1);
                } else {           // streamed once
                    tma_load_2d_hint(sa, &wmap, &a_full[stage], kb * 64, row0, pol_first);
                    if (TWO)
                        tma_load_2d_hint(sa + 128 * 128, &wmap, &a_full[stage], kb * 64, row0 + a.a_sub1, pol_first);
                }
                if (++stage == AST) { stage = 0; phase ^= 1; p_wrapped = true; }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int as = 0, bs = 0, buf = 0, qs = 0;
        uint32_t aph = 0, bph = 0, tph = 0, qp = 0;
        for (;;) {
            int4 it;
            if (!pop(qs, qp, it, false)) goto done;
            if (it.w < 0) break;
            const uint32_t idesc = idesc_bf16(128, (it.w + 15) & ~15) | (AMN ? (1u << 15) : 0u);
            if (!mbar_wait(&tempty[buf], tph ^ 1, abort_flag)) goto done;
            tc_after();
            const uint32_t d = tmem_base + buf * 256;
            for (int kb = 0; kb < a.kblocks; ++kb) {
                if (!mbar_wait(&a_full[as], aph, abort_flag)) goto done;
                if (!mbar_wait(&b_full[bs], bph, abort_flag)) goto done;
                fence_proxy_async();
                tc_after();
                const uint32_t sa = su32(sA + as * Cfg::A_BYTES);
                const uint32_t sb = su32(sB + bs * Cfg::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    const uint64_t bd = sdesc(sb + kk * 32);
                    if (AMN) {
                        umma(d, mn_desc(sa + kk * 2048, 8192), bd, idesc, acc);
                        if (TWO) umma(d + SUB1, mn_desc(sa + 128 * 128 + kk * 2048, 8192), bd, idesc, acc);
                    } else {
                        umma(d, sdesc(sa + kk * 32), bd, idesc, acc);
                        if (TWO) umma(d + SUB1, sdesc(sa + 128 * 128 + kk * 32), bd, idesc, acc);
                    }
                }
                umma_commit(&a_empty[as]);
                umma_commit(&b_empty[bs]);
                if (++as == AST) { as = 0; aph ^= 1; }
                if (++bs == BST) { bs = 0; bph ^= 1; }
            }
            umma_commit(&tfull[buf]);
            if (++buf == NBUF) { buf = 0; tph ^= 1; }
        }
    } else if (warp >= 2 && warp < Cfg::GATHER_WARP0) {
        // ------------------------------------------------ epilogue: warp w reads TMEM lane
        // quadrant w % 4; the EPI_WARPS / 4 warps of a quadrant take alternate 16-column chunks
        constexpr int WPQ = Cfg::EPI_WARPS / 4;
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int lf = q * 32 + lane;                 // feature inside a 128-row sub-tile
        const float ib1 = 1.0f / a.beta1, ib2 = 1.0f / a.beta2;
        const bool lead = lane == 0 && ((warp - 2) & 3) == 0;   // issues a half's output stores
        int ocnt = 0;                                          // a half's staged chunks
        int buf = 0, qs = 0;
        uint32_t tph = 0, qp = 0;
        for (;;) {
            int4 it = make_int4(0, 0, 0, -1);
            bool okw = pop(qs, qp, it, true);
            if (okw && it.w >= 0) okw = mbar_wait(&tfull[buf], tph, abort_flag);
            // DBUF: the four warps of a half meet at named barriers inside an item, so they
            // leave together or go on together (one barrier per item, whatever each waited for)
            if (STAGED) okw = group_all(1 + half, okw);
            if (!okw) goto done;
            if (it.w < 0) break;
            const int fb = it.y & 0xffff, N = it.w, Np = (N + 15) & ~15;
            tc_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + buf * 256;
            // GLU / GU32: the sub-tiles are the gate and up rows of feature fb*128 + lf.
            // Otherwise they are features fb*256 + lf and fb*256 + 128 + lf (one sub-tile:
            // feature fb*128 + lf).
            constexpr bool GU_LAYOUT = EPI == EPI_GLU || EPI == EPI_GU32;
            const int f = (GU_LAYOUT || !TWO ? fb * 128 : fb * 256) + lf;
            const bool ok = f < a.out_cols;
            const bool ok1 = TWO && (GU_LAYOUT ? ok : f + 128 < a.out_cols);
            if constexpr (STAGED) {
                // one 128-feature sub-tile, rows of y_e: each half stages 16 rows at a time in
                // shared memory (two buffers) and one thread stores them by TMA, so that the
                // epilogue warps never wait on global stores (they held up the drain, and with
                // it the MMAs, far longer than the reads of tensor memory did)
                constexpr int OW = 128 * Cfg::NSUB;     // features of a staged row
                for (int c = half * 16; c < Np; c += 32) {
                    uint8_t *stg = sO + (half * 2 + (ocnt & 1)) * Cfg::O_CHUNK;
                    uint32_t r0[16], r1[16];
                    TMEM_LD16(tb + c, r0);
                    if (TWO) TMEM_LD16(tb + SUB1 + c, r1);
                    if (lead) bulk_wait_read1();   // the store two chunks back has read this buffer
                    group_sync(1 + half);
                    tmem_wait_ld();
                    __nv_bfloat16 *srow = reinterpret_cast<__nv_bfloat16 *>(stg) + lf;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        srow[j * OW] = __float2bfloat16_rn(__uint_as_float(r0[j]));
                        if (TWO) srow[j * OW + 128] = __float2bfloat16_rn(__uint_as_float(r1[j]));
                    }
                    fence_proxy_async();
                    group_sync(1 + half);
                    if (lead) {
                        const int rows = N - c < 16 ? N - c : 16;
                        if (rows == 16) {
                            tma_store_2d(&omap, su32(stg), fb * OW, it.z + c);
                        } else {   // the item's last rows: one bulk store each, clipped to d_out
                            const int cols = a.out_cols - fb * OW < OW ? a.out_cols - fb * OW : OW;
                            for (int r = 0; r < rows; ++r)
                                bulk_store(static_cast<__nv_bfloat16 *>(a.out) + (long long)(it.z + c + r) * a.out_ld +
                                               fb * OW,
                                           su32(stg) + r * OW * 2, (uint32_t)cols * 2);
                        }
                        bulk_commit();
                    }
                    ++ocnt;
                }
            } else
            for (int c = half * 16; c < Np; c += 16 * WPQ) {
                if (EPI == EPI_GLU) {
                    uint32_t g[16], v[16];
                    TMEM_LD16(tb + c, g);
                    TMEM_LD16(tb + SUB1 + c, v);
                    tmem_wait_ld();
                    // h of this lane's feature for 8 rows at a time, transposed within each group
                    // of 8 lanes so that a lane holds 8 consecutive features of one row: one
                    // 16-byte store per row and group instead of eight 2-byte stores
                    const int t8 = lane & 7, fg = f - t8;
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float hv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            hv[i] = situ_glu_fast(__uint_as_float(g[8 * h8 + i]), __uint_as_float(v[8 * h8 + i]), ib1,
                                                  a.beta1, ib2, a.beta2);
                        transpose8(hv, t8);
                        const int row = c + 8 * h8 + t8;
                        if (row < N && fg < a.out_cols) {   // out_cols is a multiple of 8
                            const uint4 pk = make_uint4(pack_bf16(hv[0], hv[1]), pack_bf16(hv[2], hv[3]),
                                                        pack_bf16(hv[4], hv[5]), pack_bf16(hv[6], hv[7]));
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                       ((long long)it.z + row) * a.out_ld + fg) = pk;
                        }
                    }
                } else if (EPI == EPI_DGLU_T) {
                    // dh of features f and f + 128 for 16 token rows: the rows' fp32 gate and up
                    // pre-activations are loaded first, all in flight together (they come from
                    // HBM), then [dg | du] is computed and stored
                    uint32_t r0[16], r1[16];
                    TMEM_LD16(tb + c, r0);
                    if (TWO) TMEM_LD16(tb + SUB1 + c, r1);
                    tmem_wait_ld();
                    const int F = a.out_cols;
#pragma unroll
                    for (int j0 = 0; j0 < 16; j0 += 8) {   // 8 rows at a time (registers)
                        float g0[8], u0[8], g1[8], u1[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const bool in = c + j0 + j < N;
                            const float *gr = a.gu + ((long long)it.z + c + j0 + j) * a.ld_gu;
                            g0[j] = (in && ok) ? gr[f] : 0.f;
                            u0[j] = (in && ok) ? gr[F + f] : 0.f;
                            g1[j] = (in && ok1) ? gr[f + 128] : 0.f;
                            u1[j] = (in && ok1) ? gr[F + f + 128] : 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (c + j0 + j >= N) continue;
                            __nv_bfloat16 *dr = a.dgu + ((long long)it.z + c + j0 + j) * a.ld_dgu;
                            float dg, du;
                            if (ok) {
                                dglu(__uint_as_float(r0[j0 + j]), g0[j], u0[j], a.beta1, a.beta2, dg, du);
                                dr[f] = __float2bfloat16_rn(dg);
                                dr[F + f] = __float2bfloat16_rn(du);
                            }
                            if (TWO && ok1) {
                                dglu(__uint_as_float(r1[j0 + j]), g1[j], u1[j], a.beta1, a.beta2, dg, du);
                                dr[f + 128] = __float2bfloat16_rn(dg);
                                dr[F + f + 128] = __float2bfloat16_rn(du);
                            }
                        }
                    }
                } else {
                    uint32_t r0[16], r1[16];
                    TMEM_LD16(tb + c, r0);
                    if (TWO) TMEM_LD16(tb + SUB1 + c, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c + j >= N) continue;
                        const long long row = (long long)it.z + c + j;
                        const float v0 = __uint_as_float(r0[j]), v1 = TWO ? __uint_as_float(r1[j]) : 0.f;
                        if (EPI == EPI_BF16) {
                            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) + row * a.out_ld + f;
                            if (ok) orow[0] = __float2bfloat16_rn(v0);
                            if (ok1) orow[128] = __float2bfloat16_rn(v1);
                        } else if (EPI == EPI_F32T) {
                            float *orow = static_cast<float *>(a.out) + row * a.out_ld + f;
                            if (ok) orow[0] = v0;
                            if (ok1) orow[128] = v1;
                        } else if (EPI == EPI_GU32) {      // gate at f, up at F + f
                            float *orow = static_cast<float *>(a.out) + row * a.out_ld + f;
                            if (ok) {
                                orow[0] = v0;
                                orow[a.out_cols] = v1;
                            }
                        }
                    }
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            if (++buf == NBUF) { buf = 0; tph ^= 1; }
        }
    } else if (warp >= Cfg::GATHER_WARP0) {
        // ------------------------------------------------ token-row gather (cp.async, kept in L2)
        const uint64_t pol = policy_evict_last();
        const int gt = threadIdx.x - Cfg::GATHER_WARP0 * 32;   // 0..127
        const int ch = gt & 7;                         // 16-byte chunk of the 128-byte row
        const int rsub = gt >> 3;                      // rows rsub, rsub + 16, ...
        int stage = 0, qs = 0;
        uint32_t phase = 0, qp = 0;
        for (;;) {
            int4 it;
            if (!pop(qs, qp, it, true)) {
                cp_async_wait_all();
                goto done;
            }
            if (it.w < 0) break;
            const int N = it.w, Np = (N + 15) & ~15;
            constexpr int RJ = Cfg::PASS / 16;
            const __nv_bfloat16 *src[RJ];
#pragma unroll
            for (int j = 0; j < RJ; ++j) {
                const int r = rsub + 16 * j;
                long long row = 0;
                if (r < N) row = a.b_index ? a.b_index[it.z + r] : (long long)(it.z + r);
                src[j] = a.b_src + row * a.b_ld + ch * 8;
            }
            for (int kb = 0; kb < a.kblocks; ++kb) {
                if (!mbar_wait(&b_empty[stage], phase ^ 1, abort_flag)) {
                    cp_async_wait_all();
                    goto done;
                }
                const uint32_t sb = su32(sB + stage * Cfg::B_BYTES);
                const bool kok = kb * 64 + ch * 8 < a.b_K;
#pragma unroll
                for (int j = 0; j < RJ; ++j) {
                    const int r = rsub + 16 * j;
                    if (r < Np) {
                        const uint32_t dst = sb + r * 128 + ((ch ^ (r & 7)) << 4);
                        cp_async16_hint(dst, src[j] + kb * 64, (r < N && kok) ? 16u : 0u, pol);
                    }
                }
                cp_async_arrive_noinc(&b_full[stage]);
                if (++stage == BST) { stage = 0; phase ^= 1; }
            }
        }
        cp_async_wait_all();
    }
done:
    if (STAGED) bulk_wait_all();   // output stores read shared memory until they complete
    __syncthreads();
    if (abort_flag->abort) {   // every role has stopped: let copies and MMAs in flight finish
        if (warp == 0 && lane == 0) {
            drain_ring(a_full, AST, p_stage, p_phase, p_wrapped);
        }
        if (warp == 1 && lane == 0) {
            umma_commit(mma_drain);
            mbar_wait_drain(mma_drain, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && abort_flag->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// ---------------------------------------------------------------- grouped, MXFP4 x MXFP8
// The routed experts of the MXFP4 layer on the block-scaled tensor cores (kind::mxf8f6f4):
// the same work items and queue as grouped_kernel, with K blocks of 128 (four K = 32 MMAs per
// sub-tile).  The MMA wants the E2M1 weights one byte per value: each 16-byte chunk of a
// 128-byte (K = 128) row holds 16 values in its first 8 bytes, in the 128-byte swizzle, which
// TMA writes from the packed rows itself (the 16U4_ALIGN16B type, whose completion counts the
// packed bytes).  Its boxes are 64 bytes wide, and TMA moves about 0.18 box rows per clock per
// SM (a probe: 64-byte rows stream at 4.2 TB/s whatever the ring depth, 128-byte rows at
// 6.8-7.0 TB/s), which bounds this weight stream; packed 128-byte rows expanded by a warp in
// shared memory, or 8-byte cp.async copies into the layout, both measured slower.  Four loader
// warps gather the pass's token rows from L2 (16-byte cp.async; E4M3 codes, 128 bytes per row
// and stage) into the same ring stage.  The same warps, one per TMEM lane quadrant, write each
// stage's E8M0 scales into
// tensor memory where the MMA reads them: a slot of 16 columns between the accumulators
// (SF_COL + 16 s) holds the weight rows' scales of sub-tile 0 (columns +0..3: lane quadrant q
// reads column +q), of sub-tile 1 (+4..7) and the tokens' scales (+8..13: token n at lane
// n % 32 of every quadrant, column +8 + n / 32), four K = 32 steps to a 32-bit column.  EPI_GLU
// writes h as MXFP8: a warp's 32 lanes are 32 consecutive features of one token, one block, so
// the block maximum is a warp reduction.
template <int EPI, int PASS_>
struct MxCfg {
    static constexpr int NSUB = 2;
    static constexpr int PASS = PASS_;                 // tokens per pass (<= 192: scale columns)
    static constexpr int KB = 128;                     // K per stage
    static constexpr int A_BYTES = NSUB * 128 * KB;    // one byte per weight value (half padding)
    static constexpr int B_BYTES = PASS * KB;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    // the weights' bytes in flight are 16 KB of HBM a stage: as many stages as fit
    static constexpr int STAGES = (224 * 1024) / STAGE < 8 ? (224 * 1024) / STAGE : 8;
    static constexpr int SUB1_COL = 256;
    // scale slots of the stages: SF_COL + 16 s, between the two accumulators
    static constexpr int SF_COL = PASS <= 64 ? 64 : PASS;
    static constexpr int EPI_WARPS = 8;
    static constexpr int LOAD_WARP0 = 2 + EPI_WARPS;
    static constexpr int THREADS = (LOAD_WARP0 + 4) * 32;  // items + weights, MMA, epilogue, loaders
    // after the ring: the item queue, the mbarriers (queue, weights, token rows, scales, stage
    // free, accumulator, drain), the TMEM address and the wait state
    static constexpr int TAIL = 16 * G_TQ + 8 * (2 * G_TQ + 4 * STAGES + 3) + 8 + 16;
    static constexpr int SMEM = STAGES * STAGE + 1024 + TAIL;
    static_assert(STAGES >= 3 && SMEM <= 232448, "shared memory");
    static_assert(PASS <= SF_COL && SF_COL + 16 * STAGES <= SUB1_COL && SUB1_COL + PASS <= 512 && SF_COL % 16 == 0,
                  "TMEM columns");
};

template <int EPI, int PASS>
__global__ void __launch_bounds__(MxCfg<EPI, PASS>::THREADS, 1) grouped_mx_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                                 const GroupedArgs a) {
    using Cfg = MxCfg<EPI, PASS>;
    constexpr int ST = Cfg::STAGES, SUB1 = Cfg::SUB1_COL;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int4 *q_items = reinterpret_cast<int4 *>(smem + ST * Cfg::STAGE);
    uint64_t *q_full = reinterpret_cast<uint64_t *>(q_items + G_TQ);
    uint64_t *q_empty = q_full + G_TQ;
    uint64_t *a_full = q_empty + G_TQ;      // a stage's weights have landed
    uint64_t *full = a_full + ST;           // its token rows have landed
    uint64_t *sf_full = full + ST;          // its scales are in tensor memory
    uint64_t *empty = sf_full + ST;         // the MMAs that read it are done
    uint64_t *tfull = empty + ST;
    uint64_t *tempty = tfull + 1;
    uint64_t *mma_drain = tempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_drain + 1);
    volatile WaitCtl *abort_flag = reinterpret_cast<volatile WaitCtl *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int p_stage = 0;                  // the weight producer's ring position, kept for the drain
    uint32_t p_phase = 0;
    bool p_wrapped = false;
    if (threadIdx.x == 0) {
        mbar_init(mma_drain, 1);
        for (int s = 0; s < G_TQ; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1 + Cfg::EPI_WARPS + 4);   // MMA thread, epilogue, loader warps
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&full[s], G_GATHER_THREADS);
            mbar_init(&sf_full[s], 4);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, Cfg::EPI_WARPS);
        wait_ctl_init(abort_flag, a.wait_limit_ns);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = *tmem_slot;

    auto pop = [&](int &qs, uint32_t &qp, int4 &it, bool warp_wide) -> bool {
        if (!mbar_wait(&q_full[qs], qp, abort_flag)) return false;
        it = q_items[qs];
        if (warp_wide) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qs]);
        } else {
            mbar_arrive(&q_empty[qs]);
        }
        if (++qs == G_TQ) { qs = 0; qp ^= 1; }
        return true;
    };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ item fetch + weights by TMA
        const uint64_t pol_first = policy_evict_first();
        const int n_items = *a.n_items;
        int &s = p_stage;
        uint32_t &ph = p_phase;
        int qs = 0;
        uint32_t qp = 0;
        for (;;) {
            const int idx = atomicAdd(a.counter, 1);
            const int4 it = idx < n_items ? a.items[idx] : make_int4(0, 0, 0, -1);
            if (!mbar_wait(&q_empty[qs], qp ^ 1, abort_flag)) goto done;
            q_items[qs] = it;
            mbar_arrive(&q_full[qs]);
            if (++qs == G_TQ) { qs = 0; qp ^= 1; }
            if (it.w < 0) break;
            const bool multi = (it.y >> 16) != 0;
            const int row0 = it.x * a.a_rows_pe + (it.y & 0xffff) * a.a_fb_stride;
            for (int kb = 0; kb < a.kblocks; ++kb) {
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) goto done;
                mbar_expect_tx(&a_full[s], Cfg::A_BYTES / 2);
                const uint32_t sa = su32(smem + s * Cfg::STAGE);
                if (multi) {       // other passes of this tile run alongside: normal L2 policy
                    tma_load_2d(sa, &wmap, &a_full[s], kb * Cfg::KB, row0);
                    tma_load_2d(sa + 128 * Cfg::KB, &wmap, &a_full[s], kb * Cfg::KB, row0 + a.a_sub1);
                } else {           // streamed once
                    tma_load_2d_hint(sa, &wmap, &a_full[s], kb * Cfg::KB, row0, pol_first);
                    tma_load_2d_hint(sa + 128 * Cfg::KB, &wmap, &a_full[s], kb * Cfg::KB, row0 + a.a_sub1,
                                     pol_first);
                }
                if (++s == ST) { s = 0; ph ^= 1; p_wrapped = true; }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int s = 0, qs = 0;
        uint32_t ph = 0, tph = 0, qp = 0;
        for (;;) {
            int4 it;
            if (!pop(qs, qp, it, false)) goto done;
            if (it.w < 0) break;
            const int Np = (it.w + 15) & ~15;
            if (!mbar_wait(tempty, tph ^ 1, abort_flag)) goto done;
            tc_after();
            const uint32_t d = tmem_base;
            for (int kb = 0; kb < a.kblocks; ++kb) {
                if (!mbar_wait(&a_full[s], ph, abort_flag)) goto done;
                if (!mbar_wait(&full[s], ph, abort_flag)) goto done;
                if (!mbar_wait(&sf_full[s], ph, abort_flag)) goto done;
                fence_proxy_async();
                tc_after();
                const uint32_t sa = su32(smem + s * Cfg::STAGE);
                const uint32_t sb = sa + Cfg::A_BYTES;
                const uint32_t sf = tmem_base + Cfg::SF_COL + 16 * s;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    const uint32_t idesc = idesc_mx(128, Np, kk);
                    const uint64_t bd = sdesc(sb + kk * 32);
                    umma_mx(d, sdesc(sa + kk * 32), bd, idesc, sf, sf + 8, acc);
                    umma_mx(d + SUB1, sdesc(sa + 128 * Cfg::KB + kk * 32), bd, idesc, sf + 4, sf + 8, acc);
                }
                umma_commit(&empty[s]);
                if (++s == ST) { s = 0; ph ^= 1; }
            }
            umma_commit(tfull);
            tph ^= 1;
        }
    } else if (warp >= 2 && warp < Cfg::LOAD_WARP0) {
        // ------------------------------------------------ epilogue: warp w reads TMEM lane
        // quadrant w % 4; the two warps of a quadrant take alternate 16-column chunks
        constexpr int WPQ = Cfg::EPI_WARPS / 4;
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int lf = q * 32 + lane;                 // feature inside a 128-row sub-tile
        const float ib1 = 1.0f / a.beta1, ib2 = 1.0f / a.beta2;
        int qs = 0;
        uint32_t tph = 0, qp = 0;
        for (;;) {
            int4 it;
            if (!pop(qs, qp, it, true)) goto done;
            if (it.w < 0) break;
            const int fb = it.y & 0xffff, N = it.w, Np = (N + 15) & ~15;
            if (!mbar_wait(tfull, tph, abort_flag)) goto done;
            tc_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
            for (int c = half * 16; c < Np; c += 16 * WPQ) {
                uint32_t r0[16], r1[16];
                TMEM_LD16(tb + c, r0);
                TMEM_LD16(tb + SUB1 + c, r1);
                tmem_wait_ld();
                if (EPI == EPI_GLU) {
                    // sub-tiles = gate and up rows of feature f; h -> MXFP8 over the warp's 32
                    // features (one block), token by token
                    const int f = fb * 128 + lf;
                    uint8_t *codes = static_cast<uint8_t *>(a.out) + f;
                    uint32_t my_scale = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float hv = situ_glu_fast(__uint_as_float(r0[j]), __uint_as_float(r1[j]), ib1, a.beta1,
                                                       ib2, a.beta2);
                        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
                        const int e = mx8_exp(__uint_as_float(amax));
                        const uint32_t code = e4m3x2(hv * mx8_inv_scale(e), 0.f) & 0xFFu;
                        if (c + j < N) codes[((long long)it.z + c + j) * a.out_ld] = (uint8_t)code;
                        if (lane == j) my_scale = (uint32_t)(e + 127);
                    }
                    if (lane < 16 && c + lane < N)
                        a.out_scales[((long long)it.z + c + lane) * a.out_scale_ld + (f >> 5)] = (uint8_t)my_scale;
                } else {
                    // expert down: features fb * 256 + lf and fb * 256 + 128 + lf, y_e in bf16
                    const int f = fb * 256 + lf;
                    const bool ok = f < a.out_cols, ok1 = f + 128 < a.out_cols;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c + j >= N) continue;
                        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) + ((long long)it.z + c + j) * a.out_ld + f;
                        if (ok) orow[0] = __float2bfloat16_rn(__uint_as_float(r0[j]));
                        if (ok1) orow[128] = __float2bfloat16_rn(__uint_as_float(r1[j]));
                    }
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
            tph ^= 1;
        }
    } else if (warp >= Cfg::LOAD_WARP0) {
        // ------------------------------------------------ loaders: per stage, the pass's token
        // rows (16-byte copies from L2) and the scales
        const uint64_t pol_last = policy_evict_last();
        const int lt = threadIdx.x - Cfg::LOAD_WARP0 * 32;    // 0..127
        const int ch = lt & 7;                         // 16-byte chunk of a token row
        const int rsub = lt >> 3;                      // token rows rsub, rsub + 16, ...
        const int q = warp & 3;
        const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint8_t *bsrc = reinterpret_cast<const uint8_t *>(a.b_src);
        const uint32_t *bw = reinterpret_cast<const uint32_t *>(a.b_scales);
        constexpr int RJ = Cfg::PASS / 16;
        constexpr int NJ = Cfg::PASS / 32;
        constexpr int PF = 2;                          // scale words loaded PF stages ahead
        int s = 0, qs = 0;
        uint32_t ph = 0, qp = 0;
        for (;;) {
            int4 it;
            if (!pop(qs, qp, it, true)) {
                cp_async_wait_all();
                goto done;
            }
            if (it.w < 0) break;
            const int fb = it.y & 0xffff, N = it.w, Np = (N + 15) & ~15;
            const long long wrow0 = (long long)it.x * a.a_rows_pe + fb * a.a_fb_stride;
            const uint8_t *src[RJ];
#pragma unroll
            for (int j = 0; j < RJ; ++j) {
                const int r = rsub + 16 * j;
                long long row = 0;
                if (r < N) row = a.b_index ? a.b_index[it.z + r] : (long long)(it.z + r);
                src[j] = bsrc + row * a.b_ld + ch * 16;
            }
            const long long srow0 = wrow0 + q * 32 + lane;
            const long long srow1 = srow0 + a.a_sub1;
            const uint32_t *sa0 = srow0 < a.a_rows_total
                                      ? reinterpret_cast<const uint32_t *>(a.a_scales + srow0 * a.a_scale_ld) : nullptr;
            const uint32_t *sa1 = srow1 < a.a_rows_total
                                      ? reinterpret_cast<const uint32_t *>(a.a_scales + srow1 * a.a_scale_ld) : nullptr;
            int sbr[NJ];                               // token 32 j + lane's scale words at bw + sbr[j]
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int n = 32 * j + lane;
                sbr[j] = -1;
                if (n < N) sbr[j] = (a.b_index ? a.b_index[it.z + n] : it.z + n) * (a.b_scale_ld >> 2);
            }
            // a ring of PF register slots (static indices: the loop is unrolled by PF) hides the
            // L2 latency of the gathered scale loads
            uint32_t qa0[PF], qa1[PF], qb[PF][NJ];
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const bool in = i < a.kblocks;
                qa0[i] = (in && sa0) ? __ldg(sa0 + i) : 0u;
                qa1[i] = (in && sa1) ? __ldg(sa1 + i) : 0u;
#pragma unroll
                for (int j = 0; j < NJ; ++j) qb[i][j] = (in && sbr[j] >= 0) ? __ldg(bw + sbr[j] + i) : 0u;
            }
            for (int kb0 = 0; kb0 < a.kblocks; kb0 += PF) {
#pragma unroll
                for (int u = 0; u < PF; ++u) {
                    const int kb = kb0 + u;
                    if (kb < a.kblocks) {
                        if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                            cp_async_wait_all();
                            goto done;
                        }
                        const uint32_t sb = su32(smem + s * Cfg::STAGE) + Cfg::A_BYTES;
#pragma unroll
                        for (int j = 0; j < RJ; ++j) {
                            const int r = rsub + 16 * j;
                            if (r < Np) {
                                const uint32_t dst = sb + r * 128 + ((ch ^ (r & 7)) << 4);
                                cp_async16_hint(dst, src[j] + kb * Cfg::KB, r < N ? 16u : 0u, pol_last);
                            }
                        }
                        cp_async_arrive_noinc(&full[s]);
                        const uint32_t w0 = qa0[u], w1 = qa1[u];
                        uint32_t wb[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
                        for (int j = 0; j < NJ; ++j) wb[j] = qb[u][j];
                        const int kn = kb + PF;
                        const bool in = kn < a.kblocks;
                        qa0[u] = (in && sa0) ? __ldg(sa0 + kn) : 0u;
                        qa1[u] = (in && sa1) ? __ldg(sa1 + kn) : 0u;
#pragma unroll
                        for (int j = 0; j < NJ; ++j) qb[u][j] = (in && sbr[j] >= 0) ? __ldg(bw + sbr[j] + kn) : 0u;
                        tc_after();
                        const uint32_t col = Cfg::SF_COL + 16 * s;
                        tmem_st1(tq + col + q, w0);
                        tmem_st1(tq + col + 4 + q, w1);
                        tmem_st8(tq + col + 8, wb);
                        tmem_wait_st();
                        tc_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sf_full[s]);
                        if (++s == ST) { s = 0; ph ^= 1; }
                    }
                }
            }
        }
        cp_async_wait_all();
    }
done:
    __syncthreads();
    if (abort_flag->abort) {   // every role has stopped: let copies and MMAs in flight finish (the
                               // loaders waited for their own copies)
        if (warp == 0 && lane == 0) drain_ring(a_full, ST, p_stage, p_phase, p_wrapped);
        if (warp == 1 && lane == 0) {
            umma_commit(mma_drain);
            mbar_wait_drain(mma_drain, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && abort_flag->abort && a.status) atomicExch(&a.status[ST_TIMEOUT], 1);
}

// ---------------------------------------------------------------- router weight split
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid): each difference is exact in
// fp32 and the last one has at most 8 significant bits, so hi + mid + lo == w.
__global__ void split_router_kernel(const float *__restrict__ w, __nv_bfloat16 *__restrict__ out,
                                    long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const float v = w[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        out[i] = hi;
        out[n + i] = mid;
        out[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

// ---------------------------------------------------------------- host side
// 2-D bf16 tensor map: rows x cols (cols innermost), row pitch in elements, box 64 x box_rows,
// 128-byte swizzle, out-of-range elements read as zero.
int make_map(CUtensorMap *m, const void *base, long long rows, long long cols, long long pitch,
             int box_rows) {
    return tmap_encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, pitch, 64, box_rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename K>
int set_smem(K kern, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "smem attribute: %s", cudaGetErrorString(e));
    return SLMOE_OK;
}

template <int BN, int EPI, int PACC, int MAJ = 0>
int launch_dense(const TmaPack &maps, DenseArgs a, cudaStream_t st) {
    using Cfg = DenseCfg<BN, EPI, PACC>;
    a.tiles_n = (a.N + Cfg::BN_OUT - 1) / Cfg::BN_OUT;
    a.tiles = ((a.M + Cfg::BM_TILE - 1) / Cfg::BM_TILE) * a.tiles_n;
    if (a.tiles == 0) return SLMOE_OK;
    auto kern = dense_kernel<BN, EPI, PACC, MAJ>;
    int rc = set_smem(kern, Cfg::SMEM);
    if (rc) return rc;
    const int sms = sm_count();
    const int grid = a.tiles < sms ? a.tiles : sms;
    kern<<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(maps, a);
    return check_launch("dense_kernel");
}

// Weight-tile width of a dense GEMM: 256 rows, except for a batch of one row tile (decode),
// where the GEMM is bound by its weight reads and 64-row tiles spread them over four times as
// many SMs.  (Larger batches keep the wide tiles even when they do not fill the SMs: with
// 4096 tokens the narrow tiles were 40 % slower.)
int dense_bn(long long M, long long n_out, bool glu) {
    const long long wide_out = glu ? 128 : 256;
    const long long tiles = ((M + 255) / 256) * ((n_out + wide_out - 1) / wide_out);
    return (M <= 256 && tiles < sm_count()) ? 64 : 256;
}

template <int EPI>
int launch_dense_bn(int bn, const TmaPack &maps, const DenseArgs &a, cudaStream_t st) {
    return bn == 64 ? launch_dense<64, EPI, 1>(maps, a, st) : launch_dense<256, EPI, 1>(maps, a, st);
}

template <int EPI, int PASS>
int launch_grouped_mx(const CUtensorMap &wmap, const GroupedArgs &a, cudaStream_t st) {
    using Cfg = MxCfg<EPI, PASS>;
    auto kern = grouped_mx_kernel<EPI, PASS>;
    int rc = set_smem(kern, Cfg::SMEM);
    if (rc) return rc;
    kern<<<sm_count(), Cfg::THREADS, Cfg::SMEM, st>>>(wmap, a);
    return check_launch("grouped_mx_kernel");
}

// omap: the output's tensor map (DBUF: bf16 [rows, out_cols], boxes of 128 features x 16 rows)
template <int EPI, bool DBUF, bool AMN = false>
int launch_grouped(const CUtensorMap &wmap, const GroupedArgs &a, cudaStream_t st, const CUtensorMap *omap = nullptr) {
    using Cfg = GCfg<DBUF>;
    auto kern = grouped_kernel<EPI, DBUF, AMN>;
    int rc = set_smem(kern, Cfg::SMEM);
    if (rc) return rc;
    CUtensorMap none;
    memset(&none, 0, sizeof(none));
    if (DBUF && EPI == EPI_BF16 && !omap)
        return fail(SLMOE_EINVAL, "grouped_kernel: the staged output needs its tensor map");
    kern<<<sm_count(), Cfg::THREADS, Cfg::SMEM, st>>>(wmap, omap ? *omap : none, a);
    return check_launch("grouped_kernel");
}

}  // namespace

// Split-K finish of the router: scores = sigmoid(sum of the splits' logit sums, in split
// order, + mu) -- the router epilogue's formula.
__global__ void __launch_bounds__(256) router_splitk_reduce_kernel(const float *__restrict__ P, int S, int M,
                                                                  int E, const float *__restrict__ mu,
                                                                  float *__restrict__ scores) {
    const long long total = (long long)M * E;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(idx % E);
        float acc = 0.f;
        for (int ks = 0; ks < S; ++ks) acc += P[(long long)ks * total + idx];
        const float v = acc + (mu ? mu[e] : 0.f);
        scores[idx] = 1.0f / (1.0f + expf(-v));
    }
}

int tc_router_scores(const slmoe_config *c, const void *x, const float *W_r, const float *mu,
                     __nv_bfloat16 *wsplit, float *scores, int32_t *status, int *counter, float *partial,
                     cudaStream_t st) {
    const long long n = (long long)c->E * c->d;
    split_router_kernel<<<(int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, st>>>(W_r, wsplit, n);
    int rc = check_launch("split_router");
    if (rc) return rc;
    TmaPack maps;
    memset(&maps, 0, sizeof(maps));
    DenseArgs a = {};
    a.M = c->T;
    a.N = c->E;
    a.nseg = 3;
    for (int s = 0; s < 3; ++s) {
        if ((rc = make_map(&maps.a[s], x, c->T, c->d, c->d, 128))) return rc;
        if ((rc = make_map(&maps.b[s], wsplit + (size_t)s * n, c->E, c->d, c->d, RT_BN))) return rc;
        a.kblocks[s] = (c->d + 63) / 64;
    }
    a.C = scores;
    a.ldc = c->E;
    a.mu = mu;
    a.status = status;
    a.counter = counter;
    a.tiles_n = (a.N + RT_BN - 1) / RT_BN;
    a.tiles_mn = ((a.M + 127) / 128) * a.tiles_n;
    a.tiles = a.tiles_mn;
    if (a.tiles == 0) return SLMOE_OK;
    const int sms = sm_count();
    // a batch of at most ROUTER_SPLITK_MAX_M tokens has too few tiles to fill the SMs: split
    // the 3 x d / 64 K blocks over up to ROUTER_SPLITK_MAX CTAs per tile (at least two
    // drain chunks each), fp32 logit sums in the workspace, finished by the reduce kernel
    for (int s = 1; s < a.nseg; ++s)
        if (a.kblocks[s] != a.kblocks[0]) return fail(SLMOE_EINVAL, "router pieces differ in K");
    int S = 1;
    if (partial && a.M <= ROUTER_SPLITK_MAX_M && a.tiles_mn < sms) {
        const int ktot = 3 * a.kblocks[0];
        S = (sms + a.tiles_mn - 1) / a.tiles_mn;
        if (S > ROUTER_SPLITK_MAX) S = ROUTER_SPLITK_MAX;
        if (S > ktot / (2 * RT_DRAIN)) S = ktot / (2 * RT_DRAIN);
    }
    if (S >= 2) {
        a.ksplit = S;
        a.partial = partial;
        a.ldp = a.N;
        a.tiles = a.tiles_mn * S;
        if ((rc = set_smem(router_kernel<true>, RT_SMEM))) return rc;
        router_kernel<true><<<a.tiles < sms ? a.tiles : sms, RT_THREADS, RT_SMEM, st>>>(maps, a);
        if ((rc = check_launch("router_kernel"))) return rc;
        const long long total = (long long)a.M * a.N;
        const long long blocks = (total + 255) / 256 < 4LL * sms ? (total + 255) / 256 : 4LL * sms;
        router_splitk_reduce_kernel<<<(int)blocks, 256, 0, st>>>(partial, S, a.M, a.N, mu, scores);
        return check_launch("router_splitk_reduce");
    }
    if ((rc = set_smem(router_kernel<false>, RT_SMEM))) return rc;
    router_kernel<false><<<a.tiles < sms ? a.tiles : sms, RT_THREADS, RT_SMEM, st>>>(maps, a);
    return check_launch("router_kernel");
}

int tc_forward_front(const slmoe_config *c, const void *x, const slmoe_weights *w, const TcForward &f,
                     cudaStream_t st) {
    const int T = c->T, d = c->d, dl = c->d_latent;
    const int ns = c->n_shared, Is = c->I_shared;
    int rc;
    using bf = __nv_bfloat16;
    {   // latent down-projection: x_lat = x W_in^T
        TmaPack maps;
        memset(&maps, 0, sizeof(maps));
        const int bn = dense_bn(T, dl, false);
        if ((rc = make_map(&maps.a[0], x, T, d, d, 128))) return rc;
        if ((rc = make_map(&maps.b[0], w->W_in, dl, d, d, bn))) return rc;
        DenseArgs a = {};
        a.M = T; a.N = dl; a.nseg = 1; a.kblocks[0] = (d + 63) / 64;
        a.C = f.x_lat; a.ldc = dl; a.status = f.status; a.counter = f.counters + 1;
        if (c->dtype == SLMOE_MXFP4) {   // MXFP8 codes [T, dl], then their scales [T, dl / 32]
            a.scales = static_cast<uint8_t *>(f.x_lat) + (size_t)T * dl;
            a.ld_scales = dl / 32;
            rc = launch_dense_bn<EPI_MX8>(bn, maps, a, st);
        } else {
            if ((rc = tmap_encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, f.x_lat, T, dl, dl, 64, 32,
                                     CU_TENSOR_MAP_SWIZZLE_128B)))
                return rc;
            rc = launch_dense_bn<EPI_BF16>(bn, maps, a, st);
        }
        if (rc) return rc;
    }
    stage_event(3, st);
    const int bn_s = dense_bn(T, Is, true);
    for (int s = 0; s < ns; ++s) {   // shared experts, gate|up + SiTU-GLU on full d
        TmaPack maps;
        memset(&maps, 0, sizeof(maps));
        if ((rc = make_map(&maps.a[0], x, T, d, d, 128))) return rc;
        // the weight tile is bn_s / 2 gate rows and bn_s / 2 up rows, loaded as two boxes
        if ((rc = make_map(&maps.b[0], static_cast<const bf *>(w->W13_s) + (size_t)s * 2 * Is * d, 2 * Is, d, d,
                           bn_s / 2)))
            return rc;
        DenseArgs a = {};
        a.M = T; a.N = Is; a.nseg = 1; a.kblocks[0] = (d + 63) / 64; a.glu_up_row = Is;
        a.C = static_cast<bf *>(f.h_s) + (size_t)s * Is; a.ldc = (long long)ns * Is;
        a.beta1 = c->beta1; a.beta2 = c->beta2; a.status = f.status; a.counter = f.counters + 2 + s;
        if ((rc = launch_dense_bn<EPI_GLU>(bn_s, maps, a, st))) return rc;
    }
    stage_event(7, st);
    return SLMOE_OK;
}

int tc_worklists(const slmoe_config *c, const TcForward &f, cudaStream_t st) {
    const int E = c->E, I = c->I, dl = c->d_latent;
    const long long Tk = (long long)c->T * c->k;
    const int nfb1 = (I + 127) / 128, nfb2 = (dl + down_block(c) - 1) / down_block(c);
    const int pass = grouped_pass(c);
    const long long Tk_items = (Tk + pass - 1) / pass;
    worklist_kernel<<<1, 1024, 0, st>>>(f.counts, f.offsets, E, nfb1, pass, f.items1, nfb2, pass, f.items2,
                                        f.counters + 8, (int)(nfb1 * (E + Tk_items)), (int)(nfb2 * (E + Tk_items)));
    return check_launch("worklist");
}

// The routed experts of the MXFP4 layer: gate|up + SiTU-GLU (h as MXFP8) and down on the
// block-scaled tensor cores, K blocks of 128.  Packed weights [rows, K / 2] bytes through TMA
// (16U4_ALIGN16B: K a multiple of 128, the base 32-byte aligned); x_lat and h are MXFP8 codes
// [rows, K] followed by their scales [rows, K / 32] in their workspace regions.
static int mx_routed_experts(const slmoe_config *c, const slmoe_weights *w, const TcForward &f,
                             cudaStream_t st) {
    const int T = c->T, dl = c->d_latent, E = c->E, I = c->I;
    const long long Tk = (long long)T * c->k;
    uint8_t *xq = static_cast<uint8_t *>(f.x_lat), *hq = static_cast<uint8_t *>(f.h);
    int rc;
    {   // gate|up + SiTU-GLU: h[perm row] = GLU(W13[e] x_lat[token]), MXFP8 along I
        CUtensorMap wm;
        if ((rc = tmap_encode_fp4(&wm, w->W13, (long long)E * 2 * I, dl))) return rc;
        GroupedArgs a = {};
        a.kblocks = dl / 128;
        a.a_rows_pe = 2 * I; a.a_sub1 = I; a.a_fb_stride = 128;
        a.items = f.items1; a.n_items = f.counters + 8; a.counter = f.counters + 6;
        a.b_index = f.perm;
        a.b_src = reinterpret_cast<const __nv_bfloat16 *>(xq); a.b_ld = dl; a.b_K = dl;
        a.out = hq; a.out_ld = I; a.out_cols = I;
        a.beta1 = c->beta1; a.beta2 = c->beta2; a.status = f.status;
        a.a_scales = w->W13_scale; a.a_scale_ld = dl / 32; a.a_rows_total = (long long)E * 2 * I;
        a.b_scales = xq + (size_t)T * dl; a.b_scale_ld = dl / 32;
        a.out_scales = hq + (size_t)Tk * I; a.out_scale_ld = I / 32;
        rc = grouped_pass(c) == MX_SHORT_PASS ? launch_grouped_mx<EPI_GLU, MX_SHORT_PASS>(wm, a, st)
                                              : launch_grouped_mx<EPI_GLU, MX_LONG_PASS>(wm, a, st);
        if (rc) return rc;
    }
    stage_event(4, st);
    {   // down: y_e[row] = W2[e] h[row] (bf16)
        CUtensorMap wm;
        if ((rc = tmap_encode_fp4(&wm, w->W2, (long long)E * dl, I))) return rc;
        GroupedArgs a = {};
        a.kblocks = I / 128;
        a.a_rows_pe = dl; a.a_sub1 = 128; a.a_fb_stride = 256;
        a.items = f.items2; a.n_items = f.counters + 9; a.counter = f.counters + 7;
        a.b_index = nullptr;
        a.b_src = reinterpret_cast<const __nv_bfloat16 *>(hq); a.b_ld = I; a.b_K = I;
        a.out = f.y_e; a.out_ld = dl; a.out_cols = dl;
        a.beta1 = c->beta1; a.beta2 = c->beta2; a.status = f.status;
        a.a_scales = w->W2_scale; a.a_scale_ld = I / 32; a.a_rows_total = (long long)E * dl;
        a.b_scales = hq + (size_t)Tk * I; a.b_scale_ld = I / 32;
        rc = grouped_pass(c) == MX_SHORT_PASS ? launch_grouped_mx<EPI_BF16, MX_SHORT_PASS>(wm, a, st)
                                              : launch_grouped_mx<EPI_BF16, MX_LONG_PASS>(wm, a, st);
        if (rc) return rc;
    }
    return SLMOE_OK;
}

int tc_forward_back(const slmoe_config *c, const slmoe_weights *w, const TcForward &f, void *y,
                    cudaStream_t st) {
    const int T = c->T, d = c->d, dl = c->d_latent, E = c->E, k = c->k, I = c->I;
    const int ns = c->n_shared, Is = c->I_shared;
    const long long Tk = (long long)T * k;
    int rc;
    using bf = __nv_bfloat16;

    (void)E;
    if (c->dtype == SLMOE_MXFP4) {
        if ((rc = mx_routed_experts(c, w, f, st))) return rc;
    } else {
        {   // routed experts, gate|up + SiTU-GLU: h[perm row] = GLU(W13[e] x_lat[token])
            CUtensorMap wm;
            if ((rc = make_map(&wm, w->W13, (long long)E * 2 * I, dl, dl, 128))) return rc;
            GroupedArgs a = {};
            a.kblocks = (dl + 63) / 64;
            a.a_rows_pe = 2 * I; a.a_sub1 = I; a.a_fb_stride = 128;
            a.items = f.items1; a.n_items = f.counters + 8; a.counter = f.counters + 6;
            a.b_index = f.perm;
            a.b_src = static_cast<const bf *>(f.x_lat); a.b_ld = dl; a.b_K = dl;
            a.out = f.h; a.out_ld = I; a.out_cols = I;
            a.beta1 = c->beta1; a.beta2 = c->beta2; a.status = f.status;
            if ((rc = launch_grouped<EPI_GLU, false>(wm, a, st))) return rc;
        }
        stage_event(4, st);
        {   // routed experts, down: y_e[row] = W2[e] h[row]
            CUtensorMap wm;
            if ((rc = make_map(&wm, w->W2, (long long)E * dl, I, I, 128))) return rc;
            GroupedArgs a = {};
            a.kblocks = (I + 63) / 64;
            a.a_rows_pe = dl; a.a_sub1 = 128; a.a_fb_stride = down_block(c);
            a.items = f.items2; a.n_items = f.counters + 9; a.counter = f.counters + 7;
            a.b_index = nullptr;
            a.b_src = static_cast<const bf *>(f.h); a.b_ld = I; a.b_K = I;
            a.out = f.y_e; a.out_ld = dl; a.out_cols = dl;
            a.beta1 = c->beta1; a.beta2 = c->beta2; a.status = f.status;
            if (down_split(c)) {
                CUtensorMap om;
                if ((rc = tmap_encode_2d(&om, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, f.y_e, Tk, dl, dl, 128 * DOWN_NSUB, 16,
                                         CU_TENSOR_MAP_SWIZZLE_NONE)))
                    return rc;
                if ((rc = launch_grouped<EPI_BF16, true>(wm, a, st, &om))) return rc;
            } else if ((rc = launch_grouped<EPI_BF16, false>(wm, a, st))) {
                return rc;
            }
        }
    }
    stage_event(5, st);
    (void)Tk;
    if ((rc = launch_combine_rmsnorm(DT_BF16, f.y_e, f.topk_w, f.slot_pos, w->gamma, T, dl, k, c->eps, f.z, st)))
        return rc;
    stage_event(6, st);
    {   // y = z W_out^T + sum_s h_s W2_s^T, K cut into 1 + n_shared segments
        TmaPack maps;
        memset(&maps, 0, sizeof(maps));
        DenseArgs a = {};
        a.M = T; a.N = d; a.nseg = 1 + ns;
        const int bn = dense_bn(T, d, false);
        if ((rc = make_map(&maps.a[0], f.z, T, dl, dl, 128))) return rc;
        if ((rc = make_map(&maps.b[0], w->W_out, d, dl, dl, bn))) return rc;
        a.kblocks[0] = (dl + 63) / 64;
        for (int s = 0; s < ns; ++s) {
            if ((rc = make_map(&maps.a[1 + s], static_cast<const bf *>(f.h_s) + (size_t)s * Is, T, Is,
                               (long long)ns * Is, 128)))
                return rc;
            if ((rc = make_map(&maps.b[1 + s], static_cast<const bf *>(w->W2_s) + (size_t)s * d * Is, d, Is, Is,
                               bn)))
                return rc;
            a.kblocks[1 + s] = (Is + 63) / 64;
        }
        a.C = y; a.ldc = d; a.status = f.status; a.counter = f.counters + 5;
        if ((rc = tmap_encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, T, d, d, 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B)))
            return rc;
        if ((rc = launch_dense_bn<EPI_F32>(bn, maps, a, st))) return rc;
    }
    stage_event(8, st);
    return SLMOE_OK;
}

// ---------------------------------------------------------------- backward contractions
namespace {
template <int EPI, int MAJ>
int launch_tc_bwd_dense(int bn, const TmaPack &maps, const DenseArgs &a, cudaStream_t st) {
    return bn == 64 ? launch_dense<64, EPI, 1, MAJ>(maps, a, st) : launch_dense<256, EPI, 1, MAJ>(maps, a, st);
}
template <int EPI>
int launch_tc_bwd_maj(int maj, int bn, const TmaPack &maps, const DenseArgs &a, cudaStream_t st) {
    switch (maj) {
    case 0: return launch_tc_bwd_dense<EPI, 0>(bn, maps, a, st);
    case A_MN: return launch_tc_bwd_dense<EPI, A_MN>(bn, maps, a, st);
    case B_MN: return launch_tc_bwd_dense<EPI, B_MN>(bn, maps, a, st);
    default: return launch_tc_bwd_dense<EPI, A_MN | B_MN>(bn, maps, a, st);
    }
}
}  // namespace

int tc_dense_gemm(int maj, int M, int N, int K, TcOperand A, TcOperand B, void *C, long long ldc, int accumulate,
                  const TcDglu *dg, int32_t *status, int *counter, cudaStream_t st) {
    if (M == 0 || N == 0) return SLMOE_OK;
    if (K == 0) return fail(SLMOE_EINVAL, "dense GEMM with K = 0");
    const int bn = dense_bn(M, N, false);
    TmaPack maps;
    memset(&maps, 0, sizeof(maps));
    int rc;
    if (maj & A_MN) rc = make_map(&maps.a[0], A.p, K, M, A.pitch, 64);
    else rc = make_map(&maps.a[0], A.p, M, K, A.pitch, 128);
    if (rc) return rc;
    if (maj & B_MN) rc = make_map(&maps.b[0], B.p, K, N, B.pitch, 64);
    else rc = make_map(&maps.b[0], B.p, N, K, B.pitch, bn);
    if (rc) return rc;
    DenseArgs a = {};
    a.M = M; a.N = N; a.nseg = 1; a.kblocks[0] = (K + 63) / 64;
    a.C = C; a.ldc = ldc; a.accumulate = accumulate; a.status = status; a.counter = counter;
    if (dg) {
        a.gu = dg->gu; a.ld_gu = dg->ld_gu; a.F = dg->F; a.dgu = dg->dgu; a.ld_dgu = dg->ld_dgu;
        a.dbeta1 = dg->beta1; a.dbeta2 = dg->beta2;
        return launch_tc_bwd_maj<EPI_DGLU>(maj, bn, maps, a, st);
    }
    if ((rc = tmap_encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, M, N, ldc, 32, 32,
                             CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    return launch_tc_bwd_maj<EPI_F32>(maj, bn, maps, a, st);
}

int tc_grouped_bwd(int kind, const slmoe_config *c, const void *W, const void *rows, const int32_t *row_index,
                   const int4 *items, const int *n_items, int *counter, void *out, const float *gu,
                   __nv_bfloat16 *dgu, int32_t *status, cudaStream_t st) {
    const int E = c->E, I = c->I, dl = c->d_latent;
    CUtensorMap wm;
    GroupedArgs a = {};
    a.items = items; a.n_items = n_items; a.counter = counter; a.status = status;
    a.beta1 = c->beta1; a.beta2 = c->beta2;
    a.b_index = row_index;
    a.b_src = static_cast<const __nv_bfloat16 *>(rows);
    a.out = out;
    int rc;
    if (kind == TC_BWD_GU32) {
        // pre-activations of the routed experts, as the forward gate|up: gu[row] = W13[e] x_lat
        if ((rc = make_map(&wm, W, (long long)E * 2 * I, dl, dl, 128))) return rc;
        a.kblocks = (dl + 63) / 64;
        a.a_rows_pe = 2 * I; a.a_sub1 = I; a.a_fb_stride = 128;
        a.b_ld = dl; a.b_K = dl;
        a.out_ld = 2 * I; a.out_cols = I;
        return launch_grouped<EPI_GU32, false>(wm, a, st);
    }
    if (kind == TC_BWD_DGLU) {
        // dh = W2[e]^T dy_e (W2[e] stored [d_l, I]: MN-major), then [dg | du]
        if ((rc = make_map(&wm, W, (long long)E * dl, I, I, 64))) return rc;
        a.kblocks = (dl + 63) / 64;
        a.a_rows_pe = dl; a.a_sub1 = 0; a.a_fb_stride = 128;   // one 128-feature sub-tile, two sets
        a.b_ld = dl; a.b_K = dl;
        a.out_cols = I; a.gu = gu; a.ld_gu = 2 * I; a.dgu = dgu; a.ld_dgu = 2 * I;
        return launch_grouped<EPI_DGLU_T, true, true>(wm, a, st);
    }
    // TC_BWD_DXE: the x_lat gradient of each expert row, W13[e]^T [dg | du] (W13[e] stored [2I, d_l])
    if ((rc = make_map(&wm, W, (long long)E * 2 * I, dl, dl, 64))) return rc;
    a.kblocks = (2 * I + 63) / 64;
    a.a_rows_pe = 2 * I; a.a_sub1 = 128; a.a_fb_stride = 256;
    a.b_ld = 2 * I; a.b_K = 2 * I;
    a.out_ld = dl; a.out_cols = dl;
    return launch_grouped<EPI_F32T, false, true>(wm, a, st);
}

int tc_worklist_single(const int32_t *counts, const int32_t *offsets, int E, int nfb, int4 *items, int *n_items,
                       int max_items, cudaStream_t st) {
    worklist_kernel<<<1, 1024, 0, st>>>(counts, offsets, E, nfb, GCfg<false>::PASS, items, 0, GCfg<false>::PASS, items,
                                        n_items, max_items, 0);
    return check_launch("worklist");
}

// One tile of the dense kernel whose producer issues no copies: the MMA thread's first wait
// runs out after wait_limit_ns, every role leaves its loop, there is nothing in flight to
// drain, TMEM is freed and status[2] is set.  No operand is read (the tensor maps are never
// used) and nothing but status is written (M = 0: no output row exists).
int tc_wait_abort_check(int32_t *status, unsigned long long wait_limit_ns, cudaStream_t st) {
    using Cfg = DenseCfg<64, EPI_BF16, 1>;
    TmaPack maps;
    memset(&maps, 0, sizeof(maps));
    DenseArgs a = {};
    a.M = 0;
    a.N = 64;
    a.nseg = 1;
    a.kblocks[0] = 1;
    a.tiles_n = 1;
    a.tiles = 1;
    a.status = status;
    a.wait_limit_ns = wait_limit_ns;
    a.stall_producer = 1;
    auto kern = dense_kernel<64, EPI_BF16, 1>;
    int rc = set_smem(kern, Cfg::SMEM);
    if (rc) return rc;
    kern<<<1, Cfg::THREADS, Cfg::SMEM, st>>>(maps, a);
    return check_launch("dense_kernel (wait abort check)");
}

}  // namespace slmoe
